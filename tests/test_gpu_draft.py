"""GPU parity of the draft decode attention (vc_draft_attn) against the fp64
oracle on the oracle's own quantized cache (bit-identical to the GPU's, see
test_gpu_quantize), and over dense (compacted or full) caches.
Tolerance: max |gpu - oracle| <= 2e-2 * max |oracle| per output tensor."""
import numpy as np
import pytest
import torch

import oracle
from lossless_draft_verify_gb300 import inputs
from helpers import assert_attn_close, f32, lib

pytestmark = pytest.mark.gpu


def _run_kivi(vc, B, Hq, Hkv, L, d, bits, R, dtype=torch.bfloat16, seed=0, extra_groups=0, rotate=False):
    k, v = inputs.kv_with_outliers(B, Hkv, L, d, seed=seed, device="cuda", dtype=dtype)
    q = inputs.normal_bf16((B, Hq, d), seed + 100, device="cuda").to(dtype)
    G = 32
    maxg = max(1, (L - R) // G + extra_groups)
    cache = vc.QCache(B, Hkv, d, bits, maxg, R + G + 8, R, res_dtype=dtype, rotate=rotate)
    vc.vc_quantize_kv(k, v, cache)
    view = cache.view()
    ws = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    scale = inputs.default_scale(d)
    vc.vc_draft_attn(q, view, scale, out, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    return k, v, q, out, scale


@pytest.mark.parametrize("B,Hq,Hkv,L,d,bits,R,dtype", [
    (2, 8, 2, 1000, 128, 2, 128, torch.bfloat16),    # many groups, ragged residual
    (3, 8, 2, 777, 128, 4, 128, torch.bfloat16),
    (2, 4, 2, 517, 64, 4, 0, torch.float32),         # tiny-decoder shape (fp32, grp 2)
    (1, 4, 4, 300, 128, 2, 16, torch.bfloat16),      # grp 1
    (2, 8, 2, 100, 128, 2, 128, torch.bfloat16),     # residual only (no group)
    (1, 8, 2, 32, 64, 2, 0, torch.bfloat16),         # exactly one group, empty residual
    (2, 8, 2, 3000, 128, 2, 1024, torch.bfloat16),   # long full-precision window: several ring splits
    (1, 4, 2, 2000, 64, 4, 600, torch.float32),      # fp32 ring over several splits
])
def test_draft_kivi_matches_oracle(B, Hq, Hkv, L, d, bits, R, dtype):
    vc = lib()
    k, v, q, out, scale = _run_kivi(vc, B, Hq, Hkv, L, d, bits, R, dtype, seed=L + bits)
    qc = oracle.kivi_quantize(f32(k), f32(v), bits, 32, R)
    want = oracle.kivi_decode_attn(f32(q), qc, scale)
    assert_attn_close(out, want, what=f"kivi {B}x{Hq}/{Hkv}x{L}x{d} b{bits}")


def test_draft_kivi_spare_capacity_and_ragged_lengths():
    """Record capacity beyond the used groups, and per-sequence lengths that
    differ (appended tokens), still attend exactly the cached tokens."""
    vc = lib()
    B, Hq, Hkv, d, bits, R, G = 3, 8, 2, 128, 2, 64, 32
    L0 = 400
    k, v = inputs.kv_with_outliers(B, Hkv, L0 + 80, d, seed=3, device="cuda")
    q = inputs.normal_bf16((B, Hq, d), 77, device="cuda")
    cache = vc.QCache(B, Hkv, d, bits, 40, R + G + 96, R)
    vc.vc_quantize_kv(k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(), cache)
    add = [0, 37, 80]
    kn = k[:, :, L0:].contiguous()
    vn = v[:, :, L0:].contiguous()
    vc.vc_qcache_append(cache, kn, vn, torch.tensor(add, dtype=torch.int32, device="cuda"), requantize=True)
    view = cache.view()
    ws = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    vc.vc_draft_attn(q, view, 0.09, out, ws)
    torch.cuda.synchronize()
    for b in range(B):
        L = L0 + add[b]
        qc = oracle.kivi_quantize(f32(k[b:b + 1, :, :L]), f32(v[b:b + 1, :, :L]), bits, G, R)
        want = oracle.kivi_decode_attn(f32(q[b:b + 1]), qc, 0.09)
        assert_attn_close(out[b:b + 1], want, what=f"seq {b}")


def test_draft_kivi_one_sequence_many_splits():
    """One 32768-token sequence with 8 kv heads: each unit is cut into the
    largest number of splits the merge takes."""
    vc = lib()
    k, v, q, out, scale = _run_kivi(vc, 1, 32, 8, 32768, 128, 2, 128, seed=11)
    qc = oracle.kivi_quantize(f32(k), f32(v), 2, 32, 128)
    want = oracle.kivi_decode_attn(f32(q), qc, scale)
    assert_attn_close(out, want, what="B1 32k")


@pytest.mark.parametrize("R", [64, 512])
def test_draft_kivi_mixed_lengths(R):
    """Sequences of very different lengths (with R = 64: quantized groups 1,
    91, 29, 2; with R = 512 two sequences are ring only), grown by appends so
    that the ring wraps around many times."""
    vc = lib()
    B, Hq, Hkv, d, bits, G = 4, 8, 2, 128, 2, 32
    L0, target = 100, [100, 3000, 1000, 131]
    k, v = inputs.kv_with_outliers(B, Hkv, max(target), d, seed=21, device="cuda")
    q = inputs.normal_bf16((B, Hq, d), 121, device="cuda")
    cache = vc.QCache(B, Hkv, d, bits, 100, R + G + 64, R)
    vc.vc_quantize_kv(k[:, :, :L0].contiguous(), v[:, :, :L0].contiguous(), cache)
    have = [L0] * B
    while any(h < t for h, t in zip(have, target)):
        n = [min(64, t - h) for h, t in zip(have, target)]
        kn = torch.zeros(B, Hkv, 64, d, dtype=k.dtype, device="cuda")
        vn = torch.zeros_like(kn)
        for b in range(B):
            kn[b, :, :n[b]] = k[b, :, have[b]:have[b] + n[b]]
            vn[b, :, :n[b]] = v[b, :, have[b]:have[b] + n[b]]
        vc.vc_qcache_append(cache, kn, vn, torch.tensor(n, dtype=torch.int32, device="cuda"), requantize=True)
        have = [h + m for h, m in zip(have, n)]
    view = cache.view()
    ws = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    vc.vc_draft_attn(q, view, 0.09, out, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    assert cache.n_groups.cpu().tolist() == [max(0, (t - R) // G) for t in target]
    for b in range(B):
        L = target[b]
        qc = oracle.kivi_quantize(f32(k[b:b + 1, :, :L]), f32(v[b:b + 1, :, :L]), bits, G, R)
        want = oracle.kivi_decode_attn(f32(q[b:b + 1]), qc, 0.09)
        assert_attn_close(out[b:b + 1], want, what=f"seq {b} (L={L})")


@pytest.mark.parametrize("B,Hq,Hkv,L,d,bits,R,dtype", [
    (2, 8, 2, 1000, 128, 2, 128, torch.bfloat16),
    (2, 4, 2, 517, 64, 4, 16, torch.float32),
    (2, 8, 2, 2000, 128, 2, 600, torch.bfloat16),     # ring over several splits
])
def test_draft_kivi_rotated_cache_matches_oracle(B, Hq, Hkv, L, d, bits, R, dtype):
    """Rotated keys (and queries rotated inside the kernel) against the
    oracle's rotated cache, read through its rotated queries."""
    vc = lib()
    k, v, q, out, scale = _run_kivi(vc, B, Hq, Hkv, L, d, bits, R, dtype, seed=L + 7, rotate=True)
    qc = oracle.kivi_quantize(f32(k), f32(v), bits, 32, R, rotate=True, rotate_bf16=dtype == torch.bfloat16)
    want = oracle.kivi_decode_attn(f32(q), qc, scale)
    assert_attn_close(out, want, what=f"rotated {B}x{Hq}/{Hkv}x{L}x{d} b{bits}")


@pytest.mark.parametrize("dtype,d,Hq", [(torch.bfloat16, 128, 8), (torch.bfloat16, 64, 4), (torch.bfloat16, 128, 2),
                                        (torch.float32, 64, 8)])
def test_draft_dense_matches_oracle(dtype, d, Hq):
    vc = lib()
    B, Hkv, Ls = 3, 2, 700
    k, v = inputs.kv_with_outliers(B, Hkv, Ls, d, seed=9, device="cuda", dtype=dtype, n_out=0)
    q = inputs.normal_bf16((B, Hq, d), 19, device="cuda").to(dtype)
    lens = torch.tensor([700, 333, 1], dtype=torch.int32, device="cuda")
    view = vc.dense_view(k, v, lens, 700)
    ws = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    vc.vc_draft_attn(q, view, 0.1, out, ws)
    torch.cuda.synchronize()
    want = oracle.dense_decode_attn(f32(q), f32(k), f32(v), lens.cpu().numpy(), 0.1)
    assert_attn_close(out, want, what="dense")


def test_draft_dense_compacted_workload_sampled():
    """Decode attention over a compacted cache of the token-dropping workload's
    shape ([4, 8, 33024, 128] bf16, 32/8 heads); sampled sequences against the
    oracle."""
    vc = lib()
    B, Hq, Hkv, L, d = 4, 32, 8, 33024, 128
    k, v = inputs.kv_with_outliers(B, Hkv, L, d, seed=12, device="cuda", n_out=0)
    q = inputs.normal_bf16((B, Hq, d), 13, device="cuda")
    lens = torch.tensor([L, L - 5, 17, L], dtype=torch.int32, device="cuda")
    view = vc.dense_view(k, v, lens, L)
    ws = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    scale = inputs.default_scale(d)
    vc.vc_draft_attn(q, view, scale, out, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    for b in (1, 2):
        want = oracle.dense_decode_attn(f32(q[b:b + 1]), f32(k[b:b + 1]), f32(v[b:b + 1]),
                                        lens[b:b + 1].cpu().numpy(), scale)
        assert_attn_close(out[b:b + 1], want, what=f"seq {b}")


def test_draft_full_size_sampled():
    """The 16-sequence, 32/8-head, 32768-token 2-bit workload in the launch
    configuration the benchmark times; outputs of sampled sequences against
    the oracle."""
    vc = lib()
    B, Hq, Hkv, L, d, R = 16, 32, 8, 32768, 128, 128
    k, v, q, out, scale = _run_kivi(vc, B, Hq, Hkv, L, d, 2, R, seed=1)
    for b in (0, 7, 15):
        qc = oracle.kivi_quantize(f32(k[b:b + 1]), f32(v[b:b + 1]), 2, 32, R)
        want = oracle.kivi_decode_attn(f32(q[b:b + 1]), qc, scale)
        assert_attn_close(out[b:b + 1], want, what=f"full-size seq {b}")
