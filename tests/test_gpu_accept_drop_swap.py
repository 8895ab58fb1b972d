"""GPU parity of greedy acceptance (bit-exact n_acc / next_tok), token
dropping (bit-exact kept indices and gathered rows) and the pinned-memory
swap-in, all through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from lossless_draft_verify_gb300 import inputs
from helpers import f32, lib, plain_accept_case

pytestmark = pytest.mark.gpu


def _accept(vc, logits, drafts):
    B, D1, V = logits.shape
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    nx = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = vc.Workspace(vc.vc_accept_workspace_bytes(B, D1 - 1, V))
    vc.vc_accept(logits, drafts, n, nx, ws)
    torch.cuda.synchronize()
    return n.cpu().numpy(), nx.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_accept_ties_and_signed_zero(dtype):
    vc = lib()
    g = torch.Generator().manual_seed(4)
    B, D, V = 7, 9, 1000
    lg = torch.randint(-3, 3, (B, D + 1, V), generator=g).to(torch.float32)
    lg[0, 0] = -1.0
    lg[0, 0, [5, 9]] = 0.0
    lg[0, 0, 7] = -0.0                                     # -0 ties +0; lowest index wins
    drafts = torch.randint(0, V, (B, D), generator=g, dtype=torch.int32)
    _, _, am = oracle.accept(lg.numpy(), drafts.numpy())
    for b in range(B):
        drafts[b, :b] = torch.from_numpy(am[b, :b])         # prefixes of various lengths
    lg_d = lg.to(dtype).cuda()
    n, nx = _accept(vc, lg_d, drafts.cuda())
    wn, wnx, _ = oracle.accept(f32(lg_d), drafts.numpy())
    assert n.tolist() == wn.tolist() and nx.tolist() == wnx.tolist()


def test_accept_horizon_zero_and_odd_vocab():
    vc = lib()
    lg = inputs.normal_bf16((3, 1, 37), 1, device="cuda")    # V not a multiple of 8: scalar path
    n, nx = _accept(vc, lg, torch.zeros(3, 0, dtype=torch.int32, device="cuda"))
    wn, wnx, _ = oracle.accept(f32(lg), np.zeros((3, 0), np.int32))
    assert n.tolist() == [0, 0, 0] and nx.tolist() == wnx.tolist()


def test_accept_full_size():
    """Logits [16, 33, 151936] bf16 with planted divergence points: exact."""
    vc = lib()
    case = inputs.accept_case(16, 32, 151936, seed=0, device="cuda")
    n, nx = _accept(vc, case.logits, case.drafts)
    wn, wnx, _ = oracle.accept(f32(case.logits), case.drafts.cpu().numpy())
    assert n.tolist() == wn.tolist() == case.diverge.tolist()
    assert nx.tolist() == wnx.tolist()


def test_accept_full_size_plain_normal_with_cross_split_ties():
    """[16, 33, 151936] bf16 ~ N(0,1), drafts from the oracle's argmax: the
    natural ties of bf16 rows and the planted ties across splits (equal maxima,
    -0 against +0) must all resolve to the lowest index, bit for bit."""
    vc = lib()
    lg, drafts, k = plain_accept_case(16, 32, 151936, seed=3)
    host = f32(lg)
    top = host.max(axis=2, keepdims=True)
    assert ((host == top).sum(axis=2) > 1).sum() >= 8          # natural ties present
    n, nx = _accept(vc, lg, drafts)
    wn, wnx, _ = oracle.accept(host, drafts.cpu().numpy())
    assert n.tolist() == wn.tolist() == k.tolist()
    assert nx.tolist() == wnx.tolist()


def test_accept_two_splits_with_ties():
    """V = 40000 (two splits): integer-valued logits, so the row maximum is
    tied across both splits in most rows."""
    vc = lib()
    g = torch.Generator().manual_seed(9)
    B, D, V = 6, 12, 40000
    lg = torch.randint(-40, 8, (B, D + 1, V), generator=g).to(torch.bfloat16)
    _, _, am = oracle.accept(f32(lg), np.zeros((B, D), np.int32))
    drafts = torch.randint(0, V, (B, D), generator=g, dtype=torch.int32)
    for b in range(B):
        drafts[b, :2 * b + 1] = torch.from_numpy(am[b, :2 * b + 1])
    n, nx = _accept(vc, lg.cuda(), drafts.cuda())
    wn, wnx, _ = oracle.accept(f32(lg), drafts.numpy())
    assert n.tolist() == wn.tolist() and nx.tolist() == wnx.tolist()


# --------------------------------------------------------------- drop ----

def _drop(vc, scores, k, v, keep_top, keep_recent):
    B, H, L, d = k.shape
    n_keep = vc.vc_drop_kept_count(L, keep_top, keep_recent)
    kept = torch.full((B, H, max(n_keep, 1)), -1, dtype=torch.int32, device="cuda")
    ko = torch.empty(B, H, max(n_keep, 1), d, dtype=k.dtype, device="cuda")
    vo = torch.empty_like(ko)
    ws = vc.Workspace(vc.vc_drop_tokens_workspace_bytes(B, H, L))
    vc.vc_drop_tokens(scores, k, v, keep_top, keep_recent, kept, ko, vo, ws)
    torch.cuda.synchronize()
    return n_keep, kept[..., :n_keep], ko[..., :n_keep, :], vo[..., :n_keep, :]


@pytest.mark.parametrize("B,H,L,top,recent,ties", [
    (2, 3, 10000, 2500, 256, False),
    (1, 2, 9000, 1000, 100, True),      # heavy ties: resolved by position
    (2, 2, 12000, 4000, 64, "zeros"),   # -0 and +0 at the threshold: equal scores
    (1, 1, 300, 1000, 50, False),       # keep every candidate
    (1, 1, 300, 0, 50, False),          # recent window only
    (1, 1, 40, 10, 100, False),         # window covers the sequence
])
def test_drop_matches_oracle(B, H, L, top, recent, ties):
    vc = lib()
    d = 128
    if ties == "zeros":
        g = torch.Generator().manual_seed(6)
        scores = torch.randint(-1, 2, (B, H, L), generator=g).to(torch.float32)
        neg = torch.rand(B, H, L, generator=g) < 0.5
        scores = torch.where((scores == 0) & neg, torch.tensor(-0.0), scores).cuda()
    elif ties:
        g = torch.Generator().manual_seed(2)
        scores = torch.randint(0, 20, (B, H, L), generator=g).to(torch.float32).cuda()
    else:
        scores = inputs.zipf_scores(B, H, L, seed=L, device="cuda")
    k, v = inputs.kv_with_outliers(B, H, L, d, seed=4, device="cuda", n_out=0)
    n_keep, kept, ko, vo = _drop(vc, scores, k, v, top, recent)
    want = oracle.drop_select(scores.cpu().numpy(), top, recent)
    assert kept.shape[-1] == want.shape[-1] == n_keep
    assert np.array_equal(kept.cpu().numpy(), want)
    assert torch.equal(ko, torch.take_along_dim(k, kept.long()[..., None], dim=2))
    assert torch.equal(vo, torch.take_along_dim(v, kept.long()[..., None], dim=2))


def test_drop_full_size():
    """4 x 8 x 131072 Zipf(1.1) scores, keep 32768 + 256: exact."""
    vc = lib()
    B, H, L, d = 4, 8, 131072, 128
    scores = inputs.zipf_scores(B, H, L, seed=0, device="cuda")
    k, v = inputs.kv_with_outliers(B, H, L, d, seed=8, device="cuda", n_out=0)
    n_keep, kept, ko, vo = _drop(vc, scores, k, v, L // 4, 256)
    want = oracle.drop_select(scores.cpu().numpy(), L // 4, 256)
    assert np.array_equal(kept.cpu().numpy(), want)
    for b, h in ((0, 0), (3, 7)):
        idx = kept[b, h].long()
        assert torch.equal(ko[b, h], k[b, h, idx]) and torch.equal(vo[b, h], v[b, h, idx])


# --------------------------------------------------------------- swap ----

def test_swap_in_pinned_and_rejects_pageable():
    vc = lib()
    src = torch.arange(1 << 20, dtype=torch.int32).pin_memory()
    dst = torch.zeros(1 << 20, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    ev.record(side)
    vc.vc_swap_in(dst, src, stream=side, done_event=ev)
    torch.cuda.current_stream().wait_event(ev)
    assert torch.equal(dst.cpu(), src)
    pageable = torch.zeros(16, dtype=torch.int32)
    with pytest.raises(vc.VcError) as e:
        vc.vc_swap_in(dst, pageable, nbytes=64, stream=side)
    assert e.value.status == vc.VC_ERR_INVALID


@pytest.mark.parametrize("rows", [0, 1, 37, 100])
def test_swap_in_rows_copies_the_prefix_of_every_block(rows):
    """vc_swap_in_rows: the first `rows` rows of every [pitch_rows][row] block
    arrive exactly; the device rows past them keep their old contents."""
    vc = lib()
    blocks, pitch, width = 6, 100, 208
    src = torch.randint(0, 256, (2, 3, pitch, width), dtype=torch.uint8).pin_memory()
    dst = torch.full((2, 3, pitch, width), 7, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    vc.vc_swap_in_rows(dst, src, rows, stream=side, done_event=ev)
    torch.cuda.current_stream().wait_event(ev)
    got = dst.cpu().reshape(blocks, pitch, width)
    want = src.reshape(blocks, pitch, width)
    assert torch.equal(got[:, :rows], want[:, :rows])
    assert bool((got[:, rows:] == 7).all())
    with pytest.raises(vc.VcError) as e:       # a pageable source is refused
        vc.vc_swap_in_rows(dst, torch.zeros_like(src).contiguous(), max(rows, 1), stream=side)
    assert e.value.status == vc.VC_ERR_INVALID


def test_paced_swap_in_keeps_its_rate_and_data():
    """vc_swap_in_paced: the bytes arrive intact and no faster than the
    emulated source rate (256 MiB at 25 GB/s: at least ~10.7 ms)."""
    vc = lib()
    n = 64 << 20
    src = torch.arange(n, dtype=torch.int32).pin_memory()
    dst = torch.zeros(n, dtype=torch.int32, device="cuda")
    pace = torch.zeros(4, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(side)
    vc.vc_swap_in_paced(dst, src, 25.0, pace, chunk_bytes=16 << 20, stream=side)
    t1.record(side)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    assert torch.equal(dst.cpu(), src)
    expect_ms = (4 * n) / 25e9 * 1e3
    assert ms >= 0.9 * expect_ms * 3 / 4, ms          # the last chunk is not paced
    assert ms < 20 * expect_ms, ms
