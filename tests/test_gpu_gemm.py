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


@pytest.mark.parametrize("M,N,K", [(8, 6144, 4096), (8, 32000, 4096), (16, 4096, 14336), (3, 1024, 512)])
def test_gemm_of_normalised_rows_matches_definition(M, N, K):
    """vc_gemm_rms (the draft steps' q|k|v and head products): rmsnorm(x) W
    with the row scale 1 / sqrt(mean x^2 + eps) applied in the epilogue, within
    the fp32-accumulation bound of the fp64 definition; x un-normalised
    (rows of different scales)."""
    vc = lib()
    eps = 1e-5
    x = inputs.normal_bf16((M, K), 51 + M, device="cuda")
    x = (x.float() * torch.linspace(0.5, 8.0, M, device="cuda")[:, None]).to(torch.bfloat16)
    w = inputs.normal_bf16((K, N), 52 + N, device="cuda", std=0.02)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = vc.Workspace(vc.vc_gemm_workspace_bytes(x.dtype, M, N, K))
    vc.vc_gemm_rms(x, w, out, eps, ws=ws)
    torch.cuda.synchronize()
    xd = f32(x).astype(np.float64)
    h = xd / np.sqrt((xd * xd).mean(axis=1, keepdims=True) + eps)
    want = h @ f32(w).astype(np.float64)
    got = f32(out).astype(np.float64)
    tol = 2.0 ** -8 * np.abs(want) + 1e-5 * np.sqrt(K) * np.abs(h).max() * np.abs(f32(w)).max() * 8
    assert np.isfinite(got).all() and (np.abs(got - want) <= tol).all(), np.abs(got - want).max()


def test_swiglu_of_normalised_rows_matches_definition():
    """vc_gemm_rms with swiglu: act = silu(g) u of the normalised rows' gate and
    up products, within a few bf16 ulps of the fp64 definition."""
    vc = lib()
    M, F, K, eps = 8, 14336, 1024, 1e-5        # the draft steps' unsplit gate|up width
    x = (inputs.normal_bf16((M, K), 61, device="cuda").float() * 3.0).to(torch.bfloat16)
    w = inputs.normal_bf16((K, 2 * F), 62, device="cuda", std=0.05)
    act = torch.full((M, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc.vc_gemm_rms(x, w, act, eps, swiglu=True)
    torch.cuda.synchronize()
    xd = f32(x).astype(np.float64)
    h = xd / np.sqrt((xd * xd).mean(axis=1, keepdims=True) + eps)
    gu = (h @ f32(w).astype(np.float64)).reshape(M, F // 64, 2, 64)
    g, u = gu[:, :, 0, :].reshape(M, F), gu[:, :, 1, :].reshape(M, F)
    want = g / (1.0 + np.exp(-g)) * u
    got = f32(act).astype(np.float64)
    scale = np.maximum(np.abs(want), np.abs(g * u) * 0.0 + 1e-3)
    assert np.isfinite(got).all()
    assert (np.abs(got - want) <= 2.0 ** -6 * scale + 2e-3).all(), np.abs(got - want).max()


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


def _tile_argmax(out_f32: np.ndarray):
    """Per (row, 128-column tile): the largest value and the lowest column holding it."""
    M, N = out_f32.shape
    t = out_f32.reshape(M, N // 128, 128)
    return t.max(-1), (t.argmax(-1) + 128 * np.arange(N // 128)[None, :]).astype(np.int32)


@pytest.mark.parametrize("M,N,K,plan", [(8, 32000, 4096, True), (264, 32000, 4096, False), (33, 2048, 512, False),
                                        (5, 151936, 1024, True), (1, 128, 64, False), (130, 1024, 2048, False),
                                        (8, 4096, 4096, True)])
def test_gemm_argmax_epilogue_matches_stored_product(M, N, K, plan):
    """The argmax epilogue's tile maxima are those of the bf16 product vc_gemm
    stores with the same plan (one K split and split-K shapes), including ties
    planted by duplicating the winning column inside its tile, in a later
    tile and in an earlier tile (the lowest column must win)."""
    vc = lib()
    x = inputs.normal_bf16((M, K), 11 + M, device="cuda")
    w = inputs.normal_bf16((K, N), 12 + N, device="cuda", std=0.02)
    out = _run(vc, x, w, decode_plan=plan)
    a = int(f32(out)[0].argmax())
    for j in {a ^ 1, (a + 3 * 128) % N, (a - 2 * 128) % N}:
        w[:, j] = w[:, a]
    out = f32(_run(vc, x, w, decode_plan=plan))
    nt = N // 128
    tmax = torch.empty(M, nt, dtype=torch.float32, device="cuda")
    tidx = torch.empty(M, nt, dtype=torch.int32, device="cuda")
    ws = vc.Workspace(vc.vc_gemm_workspace_bytes(x.dtype, M, N, K))
    vc.vc_gemm_argmax(x, w, tmax, tidx, ws=ws, decode_plan=plan)
    torch.cuda.synchronize()
    want_v, want_i = _tile_argmax(out)
    np.testing.assert_array_equal(tmax.cpu().numpy(), want_v)
    np.testing.assert_array_equal(tidx.cpu().numpy(), want_i)
    # the planted tie: row 0's overall argmax is the lowest duplicate
    row0 = out[0]
    assert int(np.flatnonzero(row0 == row0.max())[0]) == min({a, a ^ 1, (a + 3 * 128) % N, (a - 2 * 128) % N})


@pytest.mark.parametrize("V", [2048, 151936])
def test_accept_from_tile_maxima_matches_oracle(V):
    """Greedy acceptance from the argmax epilogue's tile maxima equals the
    oracle's acceptance over the stored logits (and vc_accept's), for drafts
    that follow the greedy tokens for 0..D rows."""
    import oracle
    vc = lib()
    B, D, K = 5, 7, 512
    M = B * (D + 1)
    x = inputs.normal_bf16((M, K), 21, device="cuda")
    w = inputs.normal_bf16((K, V), 22, device="cuda", std=0.05)
    logits = _run(vc, x, w).view(B, D + 1, V)
    am = oracle.accept(f32(logits), np.zeros((B, D), np.int32))[2]
    keep = [0, 3, D, 1, 6]
    drafts = am[:, :D].copy()
    for b, k in enumerate(keep):
        if k < D:
            drafts[b, k] = (drafts[b, k] + 1) % V
    dr = torch.tensor(drafts, dtype=torch.int32, device="cuda")
    tmax = torch.empty(M, V // 128, dtype=torch.float32, device="cuda")
    tidx = torch.empty(M, V // 128, dtype=torch.int32, device="cuda")
    ws = vc.Workspace(vc.vc_gemm_workspace_bytes(x.dtype, M, V, K))
    vc.vc_gemm_argmax(x, w, tmax, tidx, ws=ws)
    n_acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    vc.vc_accept_tiles(tmax.view(B, D + 1, -1), tidx.view(B, D + 1, -1), dr, n_acc, nxt)
    n2, x2 = torch.full_like(n_acc, -1), torch.full_like(nxt, -1)
    wa = vc.Workspace(vc.vc_accept_workspace_bytes(B, D, V))
    vc.vc_accept(logits.contiguous(), dr, n2, x2, wa)
    torch.cuda.synchronize()
    want_n, want_x, _ = oracle.accept(f32(logits), drafts)
    assert n_acc.cpu().tolist() == list(want_n) == keep
    assert nxt.cpu().tolist() == list(want_x)
    assert n2.cpu().tolist() == list(want_n) and x2.cpu().tolist() == list(want_x)


@pytest.mark.parametrize("M,F,K,plan", [(8, 14336, 4096, True), (264, 14336, 4096, False), (8, 256, 256, False),
                                        (33, 1024, 512, False), (1, 64, 64, False)])
def test_gemm_swiglu_epilogue_matches_stored_product(M, F, K, plan):
    """The SwiGLU epilogue (gate and up columns interleaved per 64) equals
    silu(g) * u computed from the bf16 product vc_gemm stores with the same
    plan: gate column j is stored column 128 (j // 64) + j % 64, its up column
    64 further.  Within one bf16 ulp everywhere (exp is the host's here, the
    device's there) and equal for almost every element."""
    vc = lib()
    x = inputs.normal_bf16((M, K), 21 + M, device="cuda")
    w = inputs.normal_bf16((K, 2 * F), 22 + F, device="cuda", std=0.05)
    assert vc.vc_gemm_splits(torch.bfloat16, 2 * F, K, plan) == 1
    gu = f32(_run(vc, x, w, decode_plan=plan)).reshape(M, F // 64, 2, 64)
    g = gu[:, :, 0, :].reshape(M, F).astype(np.float32)
    u = gu[:, :, 1, :].reshape(M, F).astype(np.float32)
    want = (g / (np.float32(1) + np.exp(-g))) * u
    want_bf = f32(torch.from_numpy(want).to(torch.bfloat16))
    act = torch.full((M, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc.vc_gemm_swiglu(x, w, act, decode_plan=plan)
    torch.cuda.synchronize()
    got = f32(act)
    assert np.isfinite(got).all()
    ulp = np.maximum(np.abs(want_bf), 2.0 ** -126) * 2.0 ** -7
    assert (np.abs(got - want_bf) <= ulp).all(), np.abs(got - want_bf).max()
    assert (got == want_bf).mean() > 0.99


def test_gemm_swiglu_refuses_split_products():
    """A gate|up product the plan splits over K is refused (the decoder then
    stores the product and runs the separate SwiGLU pass)."""
    vc = lib()
    M, F, K = 40, 512, 1024
    assert vc.vc_gemm_splits(torch.bfloat16, 2 * F, K, True) > 1
    x = inputs.normal_bf16((M, K), 31, device="cuda")
    w = inputs.normal_bf16((K, 2 * F), 32, device="cuda", std=0.05)
    act = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vc.VcError) as e:
        vc.vc_gemm_swiglu(x, w, act, decode_plan=True)
    assert e.value.status == vc.VC_ERR_UNSUPPORTED
