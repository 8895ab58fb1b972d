"""Shared helpers of the GPU parity tests: build/load the library once,
tensor conversions and the attention tolerance rule."""
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
