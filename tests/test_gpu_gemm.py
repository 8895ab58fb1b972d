"""GPU parity of the decoder's GEMM (vc_gemm): y = x W (+ r) against the plain
definition in fp64 (numpy matmul of the exact inputs), and the property the
decoder's losslessness rests on: a row's result does not depend on how many
rows share the launch."""
import numpy as np
import pytest
import torch

from lossless_draft_verify_gb300 import inputs
from helpers import f32, lib

pytestmark = pytest.mark.gpu


def _run(vc, x, w, resid=None, decode_plan=False):
    M, K = x.shape
    N = w.shape[1]
    out = torch.full((M, N), float("nan"), dtype=x.dtype, device="cuda")
    ws = vc.Workspace(vc.vc_gemm_workspace_bytes(x.dtype, M, N, K))
    vc.vc_gemm(x, w, out, resid=resid, ws=ws, decode_plan=decode_plan)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("M,N,K,plan", [(8, 384, 512, False), (300, 256, 1024, False), (1, 128, 64, False),
                                        (129, 640, 4096, False), (8, 6144, 4096, True), (16, 4096, 14336, True),
                                        (3, 1024, 512, True), (40, 512, 1024, True)])
def test_gemm_bf16_matches_definition(M, N, K, plan):
    vc = lib()
    x = inputs.normal_bf16((M, K), 1 + M, device="cuda")
    w = inputs.normal_bf16((K, N), 2 + N, device="cuda", std=0.02)
    r = inputs.normal_bf16((M, N), 3, device="cuda")
    for resid in (None, r):
        got = f32(_run(vc, x, w, resid, decode_plan=plan)).astype(np.float64)
        want = f32(x).astype(np.float64) @ f32(w).astype(np.float64)
        if resid is not None:
            want = want + f32(resid)
        # fp32 accumulation of K products, one bf16 rounding of the result
        tol = 2.0 ** -8 * np.abs(want) + 1e-5 * np.sqrt(K) * np.abs(f32(x)).max() * np.abs(f32(w)).max() * 8
        assert np.isfinite(got).all()
        assert (np.abs(got - want) <= tol).all(), np.abs(got - want).max()


def test_gemm_bf16_in_place_residual():
    vc = lib()
    M, N, K = 40, 256, 512
    x = inputs.normal_bf16((M, K), 4, device="cuda")
    w = inputs.normal_bf16((K, N), 5, device="cuda", std=0.02)
    acc = inputs.normal_bf16((M, N), 6, device="cuda")
    want = _run(vc, x, w, acc.clone())
    ws = vc.Workspace(vc.vc_gemm_workspace_bytes(x.dtype, M, N, K))
    vc.vc_gemm(x, w, acc, resid=acc, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(acc, want)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gemm_rows_independent_of_batch(dtype):
    """Row r of a 300-row product equals, bit for bit, the same row computed
    alone and inside a 33-row block."""
    vc = lib()
    M, N, K = 300, 512, 1536
    x = inputs.normal_bf16((M, K), 7, device="cuda").to(dtype)
    w = inputs.normal_bf16((K, N), 8, device="cuda", std=0.02).to(dtype)
    full = _run(vc, x, w)
    for r in (0, 131, 299):
        one = _run(vc, x[r:r + 1].contiguous(), w)
        assert torch.equal(one[0], full[r])
    blk = _run(vc, x[100:133].contiguous(), w)
    assert torch.equal(blk, full[100:133])


def test_gemm_fp32_matches_definition():
    vc = lib()
    M, N, K = 70, 200, 260
    x = inputs.normal_bf16((M, K), 9, device="cuda").float() * 1.37
    w = inputs.normal_bf16((K, N), 10, device="cuda").float() * 0.05
    got = f32(_run(vc, x, w)).astype(np.float64)
    want = f32(x).astype(np.float64) @ f32(w).astype(np.float64)
    assert np.abs(got - want).max() <= 1e-5 * np.abs(want).max()
