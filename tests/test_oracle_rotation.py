"""Pins of the oracle's key rotation (RotateKV-style compressor variant):
the binary32 Walsh-Hadamard butterfly against the Sylvester Hadamard matrix
(a worked example, exact integer cases, the binary32 rounding bound), its
algebra (involution, preserved dot products), bfloat16 rounding against an
independent conversion, and the rotated KIVI cache."""
import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle


def test_fwht_worked_example():
    # H_4 (Sylvester) times (1, 2, 3, 4): (10, -2, -4, 0)
    np.testing.assert_array_equal(oracle.fwht_f32(np.array([1, 2, 3, 4], np.float32)),
                                  np.array([10, -2, -4, 0], np.float32))


@pytest.mark.parametrize("d", [2, 4, 8, 64, 128])
def test_fwht_exact_on_small_integers(d):
    rng = np.random.default_rng(d)
    x = rng.integers(-1000, 1000, size=(7, d)).astype(np.float32)
    want = x.astype(np.float64) @ hadamard(d).astype(np.float64)
    np.testing.assert_array_equal(oracle.fwht_f32(x).astype(np.float64), want)


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_binary32_rounding_bound(d):
    rng = np.random.default_rng(10 + d)
    x = (rng.standard_normal((200, d)) * np.exp(rng.uniform(-8, 8, (200, d)))).astype(np.float32)
    got = oracle.fwht_f32(x).astype(np.float64)
    want = x.astype(np.float64) @ hadamard(d).astype(np.float64)
    # log2(d) rounded stages, each error <= 2^-24 of a partial sum <= sum |x|
    bound = np.log2(d) * 2.0 ** -24 * np.abs(x).astype(np.float64).sum(-1, keepdims=True)
    assert (np.abs(got - want) <= bound).all()
    assert not np.array_equal(got, want)        # the binary32 network does round


def test_fwht_involution_and_dot_products():
    rng = np.random.default_rng(3)
    d = 128
    x = rng.standard_normal((50, d)).astype(np.float32)
    y = rng.standard_normal((50, d)).astype(np.float32)
    twice = oracle.fwht_f32(oracle.fwht_f32(x)).astype(np.float64)
    np.testing.assert_allclose(twice, d * x.astype(np.float64), rtol=0, atol=1e-3)
    sk, sq = oracle.rotation_scales(d)
    assert sk * sq * d == 1.0 and sk == 2.0 ** -4 and sq == 2.0 ** -3
    assert oracle.rotation_scales(64) == (2.0 ** -3, 2.0 ** -3)
    kr = oracle.rotate_keys(x, bf16=False).astype(np.float64)
    qr = oracle.rotate_queries(y).astype(np.float64)
    want = (x.astype(np.float64) * y.astype(np.float64)).sum(-1)
    np.testing.assert_allclose((kr * qr).sum(-1), want, rtol=0, atol=1e-4)


def test_bf16_round_ties_and_against_torch():
    # 1 + 2^-8 is halfway between bf16 1 and 1 + 2^-7: ties to even (1);
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: to 1 + 2^-6
    vals = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -20], np.float32)
    np.testing.assert_array_equal(oracle.bf16_round(vals),
                                  np.array([1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7], np.float32))
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.bf16_round(x), want)


def test_rotated_kivi_cache():
    """The rotated cache holds rotated keys (ring rows bit for bit), obeys the
    quantizer's error bound on them, leaves values untouched, and reads back
    the dot products through rotated queries: with all keys equal, attention
    is the mean of the values exactly as without rotation."""
    rng = np.random.default_rng(5)
    B, H, L, d, R = 1, 2, 200, 128, 16
    k = oracle.bf16_round(rng.standard_normal((B, H, L, d)).astype(np.float32))
    v = oracle.bf16_round(rng.standard_normal((B, H, L, d)).astype(np.float32))
    qc = oracle.kivi_quantize(k, v, 4, 32, R, rotate=True)
    plain = oracle.kivi_quantize(k, v, 4, 32, R)
    kr = oracle.rotate_keys(k)
    nq = qc["nq"]
    np.testing.assert_array_equal(qc["kres"], kr[:, :, nq:])
    np.testing.assert_array_equal(qc["vcode"], plain["vcode"])
    kh, _ = oracle.kivi_dequant(qc)
    s = np.repeat(oracle.f16_value_fast(qc["kscale"]), 32, axis=2)
    assert (np.abs(kh - kr[:, :, :nq].astype(np.float64)) <= s / 2 * (1 + 2.0 ** -20)).all()
    # equal keys: every group is constant, the softmax is uniform
    k1 = np.broadcast_to(k[:, :, :1], k.shape).copy()
    qc1 = oracle.kivi_quantize(k1, v, 2, 32, R, rotate=True)
    q = rng.standard_normal((B, 4, d)).astype(np.float32)
    out = oracle.kivi_decode_attn(q, qc1, 0.1)
    _, vh = oracle.kivi_dequant(qc1)
    vall = np.concatenate([vh, qc1["vres"].astype(np.float64)], axis=2)
    want = np.repeat(vall.mean(axis=2), 2, axis=1)
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)
