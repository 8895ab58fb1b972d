"""GPU parity of the packed full cache for the host link (vc_kv_pack /
vc_kv_unpack) against the oracle's row format: packed bytes equal the
oracle's byte for byte, unpacking restores every bit, rows that need more
than 7 escapes are counted and marked as the oracle marks them, and the
round's full-size cache packs and unpacks exactly."""
import numpy as np
import pytest
import torch

import oracle
from lossless_draft_verify_gb300 import inputs
from helpers import lib

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _pack(vc, x: torch.Tensor):
    d = x.shape[-1]
    p = torch.empty(*x.shape[:-1], vc.vc_kv_packed_row_bytes(d), dtype=torch.uint8, device="cuda")
    n_over = torch.zeros(1, dtype=torch.int32, device="cuda")
    vc.vc_kv_pack(x, p, n_over)
    return p, n_over


@pytest.mark.parametrize("rows,d,kind", [(1, 128, "normal"), (5, 64, "normal"), (3001, 128, "outlier"),
                                         (2047, 64, "wide"), (999, 128, "special"), (64, 128, "zeros")])
def test_pack_matches_oracle_and_round_trips(rows, d, kind):
    vc = lib()
    rng = np.random.default_rng(rows + d)
    if kind == "special":
        b = rng.integers(0, 1 << 16, (rows, d), dtype=np.uint16)          # NaN, inf, subnormals included
        b[: rows // 2, 4:] = 0x3F80 ^ rng.integers(0, 0x80, (rows // 2, d - 4), dtype=np.uint16)
        x = torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        x = torch.randn(rows, d, generator=torch.Generator().manual_seed(rows)).to(torch.bfloat16)
        if kind == "outlier":
            x[:, 3] *= 8
        elif kind == "wide":
            x *= torch.exp(torch.empty(rows, d).uniform_(-12, 12, generator=torch.Generator().manual_seed(1)))
            x = x.to(torch.bfloat16)
        elif kind == "zeros":
            x[::3] = 0
            x[1::3, ::5] = 0
        x = x.cuda()
    p, n_over = _pack(vc, x)
    want, over = oracle.kv_pack_rows(_bits(x))
    got = p.cpu().numpy()
    assert int(n_over.item()) == int(over.sum())
    np.testing.assert_array_equal(got[:, 1], want[:, 1])           # escape counts and marks
    ok = ~over
    np.testing.assert_array_equal(got[ok], want[ok])
    # unpack the rows that can be held: every bit back, from the GPU's bytes and from the oracle's
    keep = torch.from_numpy(np.flatnonzero(ok)).cuda()
    for src in (p[keep], torch.from_numpy(want[ok]).cuda()):
        y = torch.empty(len(keep), d, dtype=torch.bfloat16, device="cuda")
        vc.vc_kv_unpack(src.contiguous(), y)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(y), _bits(x)[ok])
    if kind in ("normal", "outlier"):
        assert not over.any()
    if kind == "zeros":
        # all-zero rows pack (base 0, no escape); rows with 26 zeros among
        # nonzero values need 26 escapes and are marked
        assert not over[0::3].any() and over[1::3].all() and not over[2::3].any()


def test_full_round_cache_round_trip():
    """The round's bf16 K cache [16, 8, 32801, 128] with its outlier channels:
    packed without a marked row, unpacked bit for bit; sampled rows against
    the oracle's bytes."""
    vc = lib()
    k, _ = inputs.kv_with_outliers(16, 8, 32801, 128, seed=1, device="cuda")
    p, n_over = _pack(vc, k)
    y = torch.empty_like(k)
    vc.vc_kv_unpack(p, y)
    torch.cuda.synchronize()
    assert int(n_over.item()) == 0
    assert torch.equal(y.view(torch.int16), k.view(torch.int16))
    idx = torch.from_numpy(np.random.default_rng(3).integers(0, k.numel() // 128, 4096)).cuda()
    rows = k.view(-1, 128)[idx]
    want, over = oracle.kv_pack_rows(_bits(rows))
    np.testing.assert_array_equal(p.view(-1, 208)[idx].cpu().numpy(), want)
    assert not over.any()


def test_writeback_packed_matches_oracle():
    """The packed write-back stores exactly the oracle's packing of the
    committed rows (i <= n_acc[b]) at ctx[b] + i, every layer, K and V, and
    leaves every other row of the host copy untouched."""
    vc = lib()
    nl, B, hkv, dq, d, Ls = 2, 3, 2, 9, 128, 40
    g = torch.Generator().manual_seed(11)
    kb = torch.randn(nl, B, hkv, dq, d, generator=g).to(torch.bfloat16).cuda()
    vb = torch.randn(nl, B, hkv, dq, d, generator=g).to(torch.bfloat16).cuda()
    n_acc = torch.tensor([0, 8, 3], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([5, 31, 20], dtype=torch.int32, device="cuda")      # sequence 1 runs past L_stride
    rb = vc.vc_kv_packed_row_bytes(d)
    kh = torch.full((nl, B, hkv, Ls, rb), 0xA5, dtype=torch.uint8).pin_memory()
    vh = torch.full((nl, B, hkv, Ls, rb), 0x5A, dtype=torch.uint8).pin_memory()
    n_over = torch.zeros(1, dtype=torch.int32, device="cuda")
    vc.vc_kv_writeback_packed(kb, vb, n_acc, ctx, kh, vh, n_over)
    torch.cuda.synchronize()
    assert int(n_over.item()) == 0
    want_k = np.full(kh.shape, 0xA5, np.uint8)
    want_v = np.full(vh.shape, 0x5A, np.uint8)
    kbits, vbits = _bits(kb), _bits(vb)
    for b in range(B):
        for i in range(int(n_acc[b]) + 1):
            pos = int(ctx[b]) + i
            if pos >= Ls:
                continue
            want_k[:, b, :, pos] = oracle.kv_pack_rows(kbits[:, b, :, i].reshape(-1, d))[0].reshape(nl, hkv, rb)
            want_v[:, b, :, pos] = oracle.kv_pack_rows(vbits[:, b, :, i].reshape(-1, d))[0].reshape(nl, hkv, rb)
    np.testing.assert_array_equal(kh.numpy(), want_k)
    np.testing.assert_array_equal(vh.numpy(), want_v)
