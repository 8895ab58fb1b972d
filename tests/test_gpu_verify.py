"""GPU parity of the causal verify attention (vc_verify_attn) against the fp64
oracle.  bf16 with d = 128 runs the TMA + tcgen05 kernel; fp32 runs the
CUDA-core kernel.  Tolerance: max |gpu - oracle| <= 2e-2 * max |oracle|."""
import numpy as np
import pytest
import torch

import oracle
from lossless_draft_verify_gb300 import inputs
from helpers import assert_attn_close, f32, lib

pytestmark = pytest.mark.gpu


def _case(vc, B, Dq, Hq, Hkv, d, ctx, dtype, seed, pad=7):
    Ls = max(ctx) + Dq + pad
    q = inputs.normal_bf16((B, Dq, Hq, d), seed, device="cuda").to(dtype)
    k = inputs.normal_bf16((B, Hkv, Ls, d), seed + 1, device="cuda").to(dtype)
    v = inputs.normal_bf16((B, Hkv, Ls, d), seed + 2, device="cuda").to(dtype)
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    ws = vc.Workspace(vc.vc_verify_attn_workspace_bytes(dtype, B, Dq, Hq, Hkv, d, max(ctx)))
    out = torch.full_like(q, float("nan"))
    scale = inputs.default_scale(d)
    vc.vc_verify_attn(q, k, v, ctx_t, max(ctx), scale, out, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    return q, k, v, out, scale


@pytest.mark.parametrize("B,Dq,Hq,Hkv,ctx", [
    (2, 5, 8, 2, [300, 123]),        # grp 4, ragged contexts, several key tiles and splits
    (2, 32, 8, 2, [640, 1000]),      # one full 128-row tile
    (1, 33, 8, 2, [700]),            # 132 rows: the 4 rows past the tile go to the tail warp
    (2, 34, 8, 2, [640, 1000]),      # 136 rows: 8 tail rows (the most the tail warp takes)
    (2, 33, 8, 2, [0, 513]),         # tail rows with an empty and a ragged context
    (1, 17, 8, 1, [300]),            # grp 8, 136 rows
    (1, 65, 4, 2, [200]),            # grp 2, 130 rows
    (1, 35, 8, 2, [260]),            # 140 rows: too many for the tail warp, two full tiles
    (2, 16, 8, 1, [257, 64]),        # grp 8
    (1, 40, 4, 4, [90]),             # grp 1
    (1, 7, 4, 2, [0]),               # empty context: the block attends to itself
])
def test_verify_tensor_core_matches_oracle(B, Dq, Hq, Hkv, ctx):
    vc = lib()
    q, k, v, out, scale = _case(vc, B, Dq, Hq, Hkv, 128, ctx, torch.bfloat16, seed=sum(ctx) + Dq)
    want = oracle.verify_attn(f32(q), f32(k), f32(v), ctx, scale)
    assert_attn_close(out, want, what=f"tc B{B} Dq{Dq} {Hq}/{Hkv} ctx{ctx}")


@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.float32), (64, torch.bfloat16)])
def test_verify_cuda_core_matches_oracle(d, dtype):
    vc = lib()
    ctx = [515, 200]
    q, k, v, out, scale = _case(vc, 2, 17, 4, 2, d, ctx, dtype, seed=5)
    want = oracle.verify_attn(f32(q), f32(k), f32(v), ctx, scale)
    err, ref = assert_attn_close(out, want, rel=1e-4 if dtype == torch.float32 else 2e-2, what="simt")


def test_verify_full_size_sampled():
    """16 sequences x 32 drafted queries x 32/8 heads over a 32768-token bf16
    cache, the launch configuration the benchmark times; sampled kv units
    against the oracle."""
    vc = lib()
    B, Dq, Hq, Hkv, d, L = 16, 32, 32, 8, 128, 32768
    q, k, v, out, scale = _case(vc, B, Dq, Hq, Hkv, d, [L] * B, torch.bfloat16, seed=3, pad=0)
    units = [0, 37, 127]                       # b * Hkv + kvh
    bs = sorted({u // Hkv for u in units})
    qs, ks, vs = f32(q[bs]), f32(k[bs]), f32(v[bs])
    sub_units = [bs.index(u // Hkv) * Hkv + u % Hkv for u in units]
    want = oracle.verify_attn(qs, ks, vs, [L] * len(bs), scale, units=sub_units)
    got = out[bs]
    for u in sub_units:
        b, kh = divmod(u, Hkv)
        heads = slice(kh * 4, kh * 4 + 4)
        assert_attn_close(got[b, :, heads], want[b, :, heads], what=f"unit {u}")


def test_verify_full_size_dq33_sampled():
    """The acceptance semantics' verify block (D = 32 drafts + 1) at full
    size: 132 rows per kv unit, the tail rows done inside the first tile's
    CTA; sampled kv units against the oracle."""
    vc = lib()
    B, Dq, Hq, Hkv, d, L = 16, 33, 32, 8, 128, 32768
    q, k, v, out, scale = _case(vc, B, Dq, Hq, Hkv, d, [L] * B, torch.bfloat16, seed=4, pad=0)
    units = [5, 64, 126]
    bs = sorted({u // Hkv for u in units})
    qs, ks, vs = f32(q[bs]), f32(k[bs]), f32(v[bs])
    sub_units = [bs.index(u // Hkv) * Hkv + u % Hkv for u in units]
    want = oracle.verify_attn(qs, ks, vs, [L] * len(bs), scale, units=sub_units)
    got = out[bs]
    for u in sub_units:
        b, kh = divmod(u, Hkv)
        heads = slice(kh * 4, kh * 4 + 4)
        assert_attn_close(got[b, :, heads], want[b, :, heads], what=f"unit {u}")
        assert_attn_close(got[b, 32:, heads], want[b, 32:, heads], what=f"unit {u} tail row")
