"""Pins of the oracle's attention, acceptance and token-dropping functions:
library routines (scipy's softmax), closed forms (one key, equal keys),
brute force on tiny inputs, and invariants that any correct implementation
must satisfy."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from lossless_draft_verify_gb300 import inputs


def _ref_attn(q, K, V, scale):
    return softmax(K.astype(np.float64) @ q.astype(np.float64) * scale) @ V.astype(np.float64)


def test_dense_decode_matches_scipy_softmax():
    rng = np.random.default_rng(0)
    B, Hq, Hkv, L, d = 2, 4, 2, 37, 16
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    lens = np.array([37, 11], np.int32)
    out = oracle.dense_decode_attn(q, k, v, lens, 0.25)
    for b in range(B):
        for h in range(Hq):
            kh = h // 2
            want = _ref_attn(q[b, h], k[b, kh, :lens[b]], v[b, kh, :lens[b]], 0.25)
            np.testing.assert_allclose(out[b, h], want, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(1)
    d = 8
    q = rng.standard_normal((1, 2, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, 5, d)).astype(np.float32)
    k = rng.standard_normal((1, 1, 5, d)).astype(np.float32)
    # one key: output is that key's value
    out = oracle.dense_decode_attn(q, k, v, [1], 1.0)
    np.testing.assert_array_equal(out[0, 0], v[0, 0, 0].astype(np.float64))
    # equal keys: output is the mean of the values
    keq = np.repeat(k[:, :, :1], 5, axis=2)
    out = oracle.dense_decode_attn(q, keq, v, [5], 1.0)
    np.testing.assert_allclose(out[0, 1], v[0, 0].astype(np.float64).mean(0), rtol=1e-13)
    # empty cache: defined as zero
    out = oracle.dense_decode_attn(q, k, v, [0], 1.0)
    assert not out.any()


def test_gqa_mapping_consecutive_heads():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 8, 4)).astype(np.float32)
    k = rng.standard_normal((1, 2, 6, 4)).astype(np.float32)
    v = np.zeros((1, 2, 6, 4), np.float32)
    v[0, 1] = 1.0                                  # only kv head 1 carries value 1
    out = oracle.dense_decode_attn(q, k, v, [6], 0.5)
    assert np.allclose(out[0, :4], 0) and np.allclose(out[0, 4:], 1)


def test_verify_is_causal_and_equals_decode_rows():
    rng = np.random.default_rng(3)
    B, Dq, Hq, Hkv, d, ctx = 2, 5, 4, 2, 16, 9
    Ls = ctx + Dq + 3
    q = rng.standard_normal((B, Dq, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Ls, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Ls, d)).astype(np.float32)
    ctxs = np.array([ctx, ctx - 4], np.int32)
    out = oracle.verify_attn(q, k, v, ctxs, 0.3)
    for b in range(B):
        for i in range(Dq):
            row = oracle.dense_decode_attn(q[b:b + 1, i], k[b:b + 1], v[b:b + 1],
                                           [ctxs[b] + i + 1], 0.3)
            np.testing.assert_array_equal(out[b, i], row[0])
    # keys after a query's own position do not influence it
    k2, v2 = k.copy(), v.copy()
    k2[:, :, ctx + 2:] = 100.0
    v2[:, :, ctx + 2:] = -7.0
    out2 = oracle.verify_attn(q, k2, v2, ctxs, 0.3)
    np.testing.assert_array_equal(out2[0, :2], out[0, :2])


def test_kivi_decode_equals_dense_over_dequantized_cache():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, L, d = 1, 4, 2, 100, 64
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    qc = oracle.kivi_quantize(k, v, 2, 32, 20)
    kh, vh = oracle.kivi_dequant(qc)
    kfull = np.concatenate([kh, qc["kres"]], axis=2)
    vfull = np.concatenate([vh, qc["vres"]], axis=2)
    out = oracle.kivi_decode_attn(q, qc, 0.125)
    for h in range(Hq):
        want = _ref_attn(q[0, h], kfull[0, h // 2], vfull[0, h // 2], 0.125)
        np.testing.assert_allclose(out[0, h], want, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- accept --

def _brute_accept(lg, drafts):
    B, D1, V = lg.shape
    n_acc, nxt = [], []
    for b in range(B):
        am = []
        for i in range(D1):
            best = 0
            for j in range(1, V):
                if lg[b, i, j] > lg[b, i, best]:
                    best = j
            am.append(best)
        n = D1 - 1
        for i in range(D1 - 1):
            if am[i] != drafts[b][i]:
                n = i
                break
        n_acc.append(n)
        nxt.append(am[n])
    return n_acc, nxt


def test_accept_brute_force_with_ties():
    rng = np.random.default_rng(5)
    B, D, V = 6, 7, 13
    lg = rng.integers(-2, 3, (B, D + 1, V)).astype(np.float32)   # many ties
    lg[0, 0, 3] = -0.0
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    # make some prefixes match the lowest-index argmax
    for b in range(B):
        for i in range(b):
            if i < D:
                drafts[b, i] = int(np.argmax(lg[b, i]))
    n_acc, nxt, _ = oracle.accept(lg, drafts)
    want_n, want_next = _brute_accept(lg, drafts)
    assert n_acc.tolist() == want_n and nxt.tolist() == want_next


def test_accept_special_cases():
    lg = np.zeros((1, 4, 5), np.float32)
    lg[0, :, 2] = 1.0
    n, nx, _ = oracle.accept(lg, [[2, 2, 2]])
    assert (n[0], nx[0]) == (3, 2)                     # full horizon accepted
    n, nx, _ = oracle.accept(lg, [[1, 2, 2]])
    assert (n[0], nx[0]) == (0, 2)                     # first draft rejected
    tie = np.zeros((1, 1, 5), np.float32)
    tie[0, 0, [1, 3]] = 2.0
    n, nx, _ = oracle.accept(tie, np.zeros((1, 0), np.int32))
    assert nx[0] == 1                                  # lowest index on ties
    z = np.array([[[-0.0, 0.0, -1.0]]], np.float32)
    assert oracle.accept(z, np.zeros((1, 0), np.int32))[1][0] == 0   # -0 == +0
    with pytest.raises(ValueError):
        oracle.accept(np.array([[[0.0, np.nan]]], np.float32), np.zeros((1, 0), np.int32))


def test_accept_generator_plants_the_divergence():
    case = inputs.accept_case(8, 9, 101, seed=3, dtype=__import__("torch").float32)
    n, nx, am = oracle.accept(case.logits.numpy(), case.drafts.numpy())
    assert n.tolist() == case.diverge.tolist()
    assert np.array_equal(am, case.planted.numpy())
    assert nx.tolist() == [int(case.planted[b, n[b]]) for b in range(8)]


# ------------------------------------------------------------------ drop --

def test_drop_brute_force():
    rng = np.random.default_rng(6)
    B, H, L = 2, 3, 50
    s = rng.integers(0, 6, (B, H, L)).astype(np.float32)    # ties resolved by position
    kept = oracle.drop_select(s, 12, 5)
    for b in range(B):
        for h in range(H):
            order = sorted(range(L - 5), key=lambda i: (-s[b, h, i], i))[:12]
            want = sorted(order) + list(range(L - 5, L))
            assert kept[b, h].tolist() == want


def test_drop_invariants_zipf():
    s = inputs.zipf_scores(2, 2, 4096, seed=1).numpy()
    kept = oracle.drop_select(s, 1024, 256)
    assert kept.shape == (2, 2, 1280)
    for b in range(2):
        for h in range(2):
            kk = kept[b, h]
            assert np.all(np.diff(kk) > 0)
            assert np.array_equal(kk[-256:], np.arange(4096 - 256, 4096))
            cand = np.zeros(4096 - 256, bool)
            cand[kk[:-256]] = True
            assert s[b, h, :3840][cand].min() >= s[b, h, :3840][~cand].max()


def test_drop_degenerate_sizes():
    s = np.arange(10, dtype=np.float32)[None, None]
    assert oracle.drop_select(s, 4, 20).tolist() == [[list(range(10))]]   # window covers all
    assert oracle.drop_select(s, 0, 3).tolist() == [[[7, 8, 9]]]
    assert oracle.drop_select(s, 100, 0).tolist() == [[list(range(10))]]
    k = np.arange(10 * 2, dtype=np.float32).reshape(1, 1, 10, 2)
    g = oracle.drop_gather(k, oracle.drop_select(s, 2, 1))
    assert g[0, 0, :, 0].tolist() == [14.0, 16.0, 18.0]


# --------------------------------------------------------------------------
# H2O accumulated-score increment (podparley source 3)
# --------------------------------------------------------------------------

def test_h2o_mass_sums_to_heads_per_kv_head():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, L, d = 2, 8, 2, 50, 16
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    lens = [50, 7]
    m = oracle.h2o_mass(q, k, lens, 0.3)
    for b in range(B):
        for h in range(Hkv):
            assert abs(m[b, h].sum() - Hq // Hkv) < 1e-12
            assert (m[b, h, lens[b]:] == 0).all()
            assert (m[b, h, :lens[b]] > 0).all()


def test_h2o_mass_closed_forms():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 8)).astype(np.float32)
    k = rng.standard_normal((1, 1, 9, 8)).astype(np.float32)
    # one key: every head puts all its mass there
    assert np.allclose(oracle.h2o_mass(q, k, [1], 1.0)[0, 0, 0], 4.0)
    # equal keys: uniform
    k[:] = k[:, :, :1]
    m = oracle.h2o_mass(q, k, [9], 1.0)
    assert np.allclose(m[0, 0], 4.0 / 9)


def test_h2o_mass_equals_attention_weights_of_the_c_oracle():
    """With one q head per kv head and V = identity rows, decode attention
    returns the softmax weights themselves: the C oracle's attention and the
    numpy mass must agree."""
    rng = np.random.default_rng(6)
    B, H, n, d = 2, 3, 12, 16
    q = rng.standard_normal((B, H, d)).astype(np.float32)
    k = rng.standard_normal((B, H, n, d)).astype(np.float32)
    v = np.zeros((B, H, n, d), np.float32)
    for j in range(n):
        v[:, :, j, j] = 1.0
    lens = np.array([12, 5], np.int32)
    o = oracle.dense_decode_attn(q, k, v, lens, 0.25)
    m = oracle.h2o_mass(q, k, lens, 0.25)
    assert np.allclose(o[:, :, :n], m, atol=1e-12)
