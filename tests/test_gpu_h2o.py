"""GPU parity of the H2O score accumulation (vc_draft_attn_h2o, dense and KIVI
views): the attention mass every cached token receives, summed over the query heads of its kv head,
added to fp32 scores at its original position (H2O, source 3 on the podparley
page), against the oracle's softmax weights (fp64).  Tolerance: the weights
are normalised by the attention's own sum of bf16-rounded probabilities, so
each mass is within 1% of the oracle's (relative to the unit's largest)."""
import numpy as np
import pytest
import torch

import oracle
from lossless_draft_verify_gb300 import inputs
from helpers import assert_attn_close, f32, lib

pytestmark = pytest.mark.gpu


def _check_mass(got, want, what):
    for u in np.ndindex(want.shape[:2]):
        g, w = got[u], want[u]
        assert np.isfinite(g).all(), what
        assert np.abs(g - w).max() <= 1e-2 * max(w.max(), 1e-30) + 1e-7, (what, u, np.abs(g - w).max(), w.max())


@pytest.mark.parametrize("d,Hq", [(128, 8), (64, 4), (128, 2)])
def test_h2o_scores_match_oracle(d, Hq):
    vc = lib()
    B, Hkv, Ls = 3, 2, 700
    k, v = inputs.kv_with_outliers(B, Hkv, Ls, d, seed=21, device="cuda", n_out=0)
    q = inputs.normal_bf16((B, Hq, d), 22, device="cuda")
    lens = torch.tensor([700, 333, 1], dtype=torch.int32, device="cuda")
    view = vc.dense_view(k, v, lens, Ls)
    ws = vc.Workspace(vc.vc_draft_attn_h2o_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    scores = torch.zeros(B, Hkv, Ls, dtype=torch.float32, device="cuda")
    scale = inputs.default_scale(d)
    for _ in range(2):                       # two decode steps accumulate
        vc.vc_draft_attn_h2o(q, view, scale, out, scores, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    want_o = oracle.dense_decode_attn(f32(q), f32(k), f32(v), lens.cpu().numpy(), scale)
    assert_attn_close(out, want_o, what="attention output")
    mass = oracle.h2o_mass(f32(q), f32(k), lens.cpu().numpy(), scale)
    got = scores.cpu().numpy().astype(np.float64)
    _check_mass(got, 2 * mass, f"d{d} Hq{Hq}")
    for b, n in enumerate(lens.tolist()):
        assert (got[b, :, n:] == 0).all()
        assert np.allclose(got[b].sum(axis=-1), 2 * Hq // Hkv, rtol=1e-2)


def test_h2o_scores_through_kept_positions():
    """Drop to a compacted cache, attend over it with accumulation: the mass
    lands at the kept tokens' original positions and nowhere else."""
    vc = lib()
    B, H, L, d, Hq = 2, 2, 4096, 128, 8
    scores_in = inputs.zipf_scores(B, H, L, seed=3, device="cuda")
    k, v = inputs.kv_with_outliers(B, H, L, d, seed=23, device="cuda", n_out=0)
    keep_top, keep_recent = 1024, 64
    n_keep = vc.vc_drop_kept_count(L, keep_top, keep_recent)
    kept = torch.empty(B, H, n_keep, dtype=torch.int32, device="cuda")
    ko = torch.empty(B, H, n_keep, d, dtype=torch.bfloat16, device="cuda")
    vo = torch.empty_like(ko)
    wsd = vc.Workspace(vc.vc_drop_tokens_workspace_bytes(B, H, L))
    vc.vc_drop_tokens(scores_in, k, v, keep_top, keep_recent, kept, ko, vo, wsd)
    q = inputs.normal_bf16((B, Hq, d), 24, device="cuda")
    lens = torch.full((B,), n_keep, dtype=torch.int32, device="cuda")
    view = vc.dense_view(ko, vo, lens, n_keep)
    ws = vc.Workspace(vc.vc_draft_attn_h2o_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    acc = torch.zeros(B, H, L, dtype=torch.float32, device="cuda")
    scale = inputs.default_scale(d)
    vc.vc_draft_attn_h2o(q, view, scale, out, acc, ws, kept_idx=kept)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    mass = oracle.h2o_mass(f32(q), f32(ko), lens.cpu().numpy(), scale)
    got = acc.cpu().numpy().astype(np.float64)
    kp = kept.cpu().numpy()
    on_kept = np.take_along_axis(got, kp.astype(np.int64), axis=2)
    _check_mass(on_kept, mass, "kept positions")
    mask = np.ones_like(got, dtype=bool)
    np.put_along_axis(mask, kp.astype(np.int64), False, axis=2)
    assert (got[mask] == 0).all()


@pytest.mark.parametrize("B,Hq,Hkv,L,d,bits,R,dtype", [
    (2, 8, 2, 1000, 128, 2, 128, torch.bfloat16),    # several splits, ragged ring
    (1, 8, 2, 3000, 128, 4, 1024, torch.bfloat16),   # long ring over several ring splits
    (2, 4, 2, 517, 64, 4, 0, torch.float32),         # fp32 caches (tiny-decoder shape)
    (2, 8, 2, 100, 128, 2, 128, torch.bfloat16),     # ring only
])
def test_h2o_scores_on_kivi_cache(B, Hq, Hkv, L, d, bits, R, dtype):
    """vc_draft_attn_h2o over a KIVI cache: each token's mass over the
    dequantized cache x^ (and the full-precision ring) against the oracle's
    softmax weights; two calls accumulate."""
    vc = lib()
    G = 32
    k, v = inputs.kv_with_outliers(B, Hkv, L, d, seed=L + 5, device="cuda", dtype=dtype)
    q = inputs.normal_bf16((B, Hq, d), L + 6, device="cuda").to(dtype)
    maxg = max(1, (L - R) // G)
    cache = vc.QCache(B, Hkv, d, bits, maxg, R + G + 8, R, res_dtype=dtype)
    vc.vc_quantize_kv(k, v, cache)
    view = cache.view()
    cap = cache.max_groups * G + cache.res_cap
    ws = vc.Workspace(vc.vc_draft_attn_h2o_workspace_bytes(view, Hq))
    out = torch.empty_like(q)
    scores = torch.zeros(B, Hkv, cap, dtype=torch.float32, device="cuda")
    scale = inputs.default_scale(d)
    for _ in range(2):
        vc.vc_draft_attn_h2o(q, view, scale, out, scores, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    # the oracle's cache: x^ = code * s + z on the quantized prefix, the ring as stored
    qc = oracle.kivi_quantize(f32(k), f32(v), bits, G, R)
    kh, _ = oracle.kivi_dequant(qc)
    nq = kh.shape[2]
    keff = np.concatenate([kh, f32(k)[:, :, nq:]], axis=2)
    assert_attn_close(out, oracle.kivi_decode_attn(f32(q), qc, scale), what="attention output")
    mass = oracle.h2o_mass(f32(q), keff, np.full(B, L), scale)
    got = scores.cpu().numpy().astype(np.float64)
    _check_mass(got[:, :, :L], 2 * mass, f"kivi b{bits} L{L}")
    assert (got[:, :, L:] == 0).all()
    assert np.allclose(got.sum(axis=-1), 2 * Hq // Hkv, rtol=1e-2)


@pytest.mark.parametrize("B,Dq,Hq,Hkv,ctx", [
    (2, 33, 8, 2, 1500),       # the acceptance block (Dq = D + 1), tail rows of the verify kernel
    (3, 32, 8, 2, 700),        # one full 128-row tile
    (1, 5, 8, 8, 300),         # grp 1
    (2, 17, 16, 2, 2000),      # grp 8: 136 rows
])
def test_verify_h2o_scores_match_oracle(B, Dq, Hq, Hkv, ctx):
    """vc_verify_attn_h2o: the verify output is unchanged and every key gets
    the attention mass of the block's rows that see it (causal within the
    block), against the oracle's softmax weights summed over the queries."""
    vc = lib()
    d = 128
    q = inputs.normal_bf16((B, Dq, Hq, d), 31, device="cuda")
    k = inputs.normal_bf16((B, Hkv, ctx + Dq, d), 32, device="cuda")
    v = inputs.normal_bf16((B, Hkv, ctx + Dq, d), 33, device="cuda")
    lens = [ctx, max(ctx - 111, 0), ctx // 2][:B]
    ctx_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = inputs.default_scale(d)
    out = torch.empty_like(q)
    ws = vc.Workspace(vc.vc_verify_attn_h2o_workspace_bytes(B, Dq, Hq, Hkv, d, ctx))
    scores = torch.zeros(B, Hkv, ctx + Dq, dtype=torch.float32, device="cuda")
    vc.vc_verify_attn_h2o(q, k, v, ctx_len, ctx, scale, out, scores, ws)
    torch.cuda.synchronize()
    assert vc.vc_poll_status(ws) == 0
    want_o = oracle.verify_attn(f32(q), f32(k), f32(v), lens, scale)
    assert_attn_close(out, want_o, what="verify output")
    # mass: sum over the block's queries i of the decode mass over keys 0 .. ctx + i
    mass = np.zeros((B, Hkv, ctx + Dq))
    for i in range(Dq):
        mass += oracle.h2o_mass(f32(q[:, i]), f32(k), np.array(lens) + i + 1, scale)
    got = scores.cpu().numpy().astype(np.float64)
    _check_mass(got, mass, f"verify Dq{Dq} grp{Hq // Hkv}")
    for b, n in enumerate(lens):
        assert (got[b, :, n + Dq:] == 0).all()
        assert np.allclose(got[b].sum(axis=-1), Dq * Hq // Hkv, rtol=1e-2)
