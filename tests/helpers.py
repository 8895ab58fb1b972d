"""Shared helpers of the GPU parity tests: build/load the library once,
tensor conversions, the attention tolerance rule and the plain-logits
acceptance case."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def lib():
    need_gpu()
    from lossless_draft_verify_gb300 import build, vc
    build.build()
    vc.load()
    return vc


def f32(t: torch.Tensor) -> np.ndarray:
    """Exact fp32 image of a bf16/fp32 tensor, on the host."""
    return t.detach().float().cpu().numpy()


def assert_attn_close(got: torch.Tensor, want: np.ndarray, rel: float = 2e-2, what: str = ""):
    """Attention tolerance: max |gpu - oracle| <= rel * max |oracle| over the
    compared tensor (the relative max-abs rule for bf16 outputs)."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(g - want).max() if want.size else 0.0
    ref = np.abs(want).max() if want.size else 0.0
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert err <= rel * max(ref, 1e-30), f"{what}: max abs err {err:.3e} > {rel} * {ref:.3e}"
    return err, ref


def plain_accept_case(B, D, V, seed, device="cuda"):
    """Config-3 acceptance input as stated: bf16 logits ~ N(0,1) with no
    clamping or planted maximum (ties at the row maximum occur naturally),
    plus planted cross-split ties at the row maximum, and drafts equal to the
    oracle's row argmax up to a per-sequence divergence point k ~ U{0..D}.
    At k < D the draft is an index whose logit is strictly below the row
    maximum, so the divergence holds whatever the tie rule.  Returns
    (logits on device, drafts on device, k)."""
    import oracle
    from lossless_draft_verify_gb300 import inputs
    lg = inputs.normal_bf16((B, D + 1, V), seed, device=device)
    # the library scans a row of V >= 65536 in 4 slices of ceil(V / 4) rounded
    # up to 8 entries; ties are planted in different slices
    chunk = (V + 3) // 4
    chunk = (chunk + 7) // 8 * 8
    lo3 = 3 * chunk
    # row 0 of sequence 0: equal maxima in split 0 and split 3 -> the lower index
    lg[0, 0, 100] = 9.0
    lg[0, 0, lo3 + 17] = 9.0
    # row 1 of sequence 0: every other entry negative, the maximum is zero:
    # +0 in split 1 and -0 in split 3 -> the +0 (lower index)
    lg[0, 1] = -(lg[0, 1].float().abs() + 1.0).to(lg.dtype)
    lg[0, 1, chunk + 5] = 0.0
    lg[0, 1, lo3 + 9] = -0.0
    # row 0 of sequence 1: -0 in split 0, +0 in split 2 at the maximum
    lg[1, 0] = -(lg[1, 0].float().abs() + 1.0).to(lg.dtype)
    lg[1, 0, 3] = -0.0
    lg[1, 0, 2 * chunk + 1] = 0.0
    # row 2 of sequence 0: three-way tie across splits 1, 2, 3
    for j in (chunk + 40, 2 * chunk + 40, lo3 + 40):
        lg[0, 2, j] = 10.0
    host = f32(lg)
    _, _, am = oracle.accept(host, np.zeros((B, D), np.int32))
    g = np.random.default_rng(seed)
    k = g.integers(0, D + 1, size=B)
    k[0], k[1] = D, max(int(k[1]), 1)               # the planted rows are compared
    drafts = g.integers(0, V, size=(B, D)).astype(np.int32)
    for b in range(B):
        drafts[b, :k[b]] = am[b, :k[b]]
        if k[b] < D:
            row = host[b, k[b]]
            mx = row.max()
            j = int(g.integers(0, V))
            while row[j] == mx:
                j = (j + 1) % V
            drafts[b, k[b]] = j
    assert am[0, 0] == 100 and am[0, 1] == chunk + 5 and am[1, 0] == 3 and am[0, 2] == chunk + 40
    return lg, torch.from_numpy(drafts).to(device), k
