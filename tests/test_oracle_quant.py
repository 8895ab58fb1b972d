"""Pins of the oracle's number formats and KIVI-style quantizer against things
other than itself: the IEEE 754 definitions (hand-derived golden values),
numpy's binary16 conversion, exact rational arithmetic, and the
half-step error bound that the quantization rule guarantees."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_f16_golden_directed_rounding():
    for x, rn, rd, ru in _golden_rows("f16_rounding.txt"):
        xf = float(np.float32(float(x)))
        assert oracle.f32_to_f16(xf, oracle.RN) == int(rn, 16), x
        assert oracle.f32_to_f16(xf, oracle.RD) == int(rd, 16), x
        assert oracle.f32_to_f16(xf, oracle.RU) == int(ru, 16), x


def test_f16_nearest_matches_numpy():
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10,
        (rng.standard_normal(2000) * 1e-5).astype(np.float32),      # subnormal range
        rng.uniform(-70000, 70000, 1000).astype(np.float32),        # overflow range
    ])
    for x in xs:
        want = np.float32(x).astype(np.float16).view(np.uint16)
        assert oracle.f32_to_f16(float(x), oracle.RN) == int(want), x


def test_f16_directed_bracket_and_adjacency():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 4,
                         (rng.standard_normal(1000) * 3e-6).astype(np.float32)])
    for x in xs:
        lo = np.uint16(oracle.f32_to_f16(float(x), oracle.RD)).view(np.float16)
        hi = np.uint16(oracle.f32_to_f16(float(x), oracle.RU)).view(np.float16)
        assert float(lo) <= float(x) <= float(hi)
        if float(lo) == float(x):
            assert float(hi) == float(x)
        else:
            assert np.nextafter(lo, np.float16(np.inf)) == hi


def test_f16_exact_values_are_fixed_points():
    allv = np.arange(0, 0x7C00, 7, dtype=np.uint16)
    for b in allv:
        v = float(np.uint16(b).view(np.float16))
        for m in (oracle.RN, oracle.RD, oracle.RU):
            assert oracle.f32_to_f16(v, m) == int(b)


def test_f16_value_decoding():
    for b in (0x0000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x3C23, 0x7BFF, 0xC000, 0x8001):
        assert oracle.f16_value([b])[0] == float(np.uint16(b).view(np.float16))


def test_quantize_worked_example():
    rows = {r[0]: r[1:] for r in _golden_rows("kivi_group_2bit.txt")}
    x = (np.arange(32) / 10).astype(np.float32)
    codes, s, z = oracle.quantize_group(x, int(rows["bits"][0]))
    assert s == int(rows["scale_bits"][0], 16)
    assert z == int(rows["zero_bits"][0], 16)
    assert codes.tolist() == [int(c) for c in rows["codes"]]


def _check_group(x, bits):
    codes, sb, zb = oracle.quantize_group(x, bits)
    s = float(np.uint16(sb).view(np.float16))
    z = float(np.uint16(zb).view(np.float16))
    qmax = (1 << bits) - 1
    assert z <= x.min()
    assert z + qmax * s >= x.max()
    assert codes.max() <= qmax
    xh = codes.astype(np.float64) * s + z
    assert np.all(np.abs(xh - x.astype(np.float64)) <= s / 2 * (1 + 2.0 ** -20) + 0.0)
    # nearest-grid-point check in exact rational arithmetic; where the fp32
    # quotient sits within 1e-5 of a half-integer, either neighbour is allowed
    if s > 0:
        for xi, ci in zip(x, codes):
            q = (Fraction(float(xi)) - Fraction(z)) / Fraction(s)
            fl = q.numerator // q.denominator
            frac = q - fl
            if abs(frac - Fraction(1, 2)) < Fraction(1, 100000):
                assert ci in (max(fl, 0), min(fl + 1, qmax))
            else:
                want = fl + (1 if frac > Fraction(1, 2) else 0)
                assert ci == min(max(want, 0), qmax)
    return codes, s, z


@pytest.mark.parametrize("bits", [2, 4])
def test_quantize_bound_random_and_outliers(bits):
    rng = np.random.default_rng(3 + bits)
    for trial in range(200):
        x = rng.standard_normal(32).astype(np.float32)
        if trial % 3 == 0:
            x[rng.integers(32)] *= 8          # outlier channel value
        if trial % 5 == 0:
            x = (x * 1e-3).astype(np.float32)  # tight group
        if trial % 7 == 0:
            x = (x - 5).astype(np.float32)     # all negative
        # bf16 images, as the cache stores bf16
        x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
        _check_group(x, bits)


def test_quantize_grid_aligned_group_is_exact():
    # values on the grid z0 + k*s0 with fp16 z0, s0 and both ends present:
    # the rule must return s = s0, z = z0 and codes k exactly
    z0, s0 = -1.0, 0.5
    k = np.array([0, 3, 1, 2] * 8)
    x = (z0 + k * s0).astype(np.float32)
    codes, s, z = _check_group(x, 2)
    assert (s, z) == (s0, z0)
    assert np.array_equal(codes, k)


def test_quantize_exact_ties_round_to_even():
    # grid z = 0, s = 1 (both ends present) and values exactly halfway between
    # codes: the quotient is exact in fp32, and the rule rounds half to even
    # (a rule that rounds halves up would give 1, 2, 3 here)
    x = np.array([0.0, 3.0, 0.5, 1.5, 2.5] + [1.0] * 27, np.float32)
    codes, s, z = _check_group(x, 2)
    assert (s, z) == (1.0, 0.0)
    assert codes[:5].tolist() == [0, 3, 0, 2, 2]
    # 4-bit: grid 0..15 with s = 1; halves 6.5 and 7.5 go to 6 and 8
    x = np.array([0.0, 15.0, 6.5, 7.5] + [3.0] * 28, np.float32)
    codes, s, z = _check_group(x, 4)
    assert (s, z) == (1.0, 0.0)
    assert codes[:4].tolist() == [0, 15, 6, 8]


def test_quantize_constant_groups():
    codes, s, z = _check_group(np.full(32, 0.75, np.float32), 2)   # fp16-exact
    assert s == 0.0 and z == 0.75 and not codes.any()
    x = np.full(32, np.float32(0.1))                                  # not fp16-exact
    codes, s, z = _check_group(x, 4)
    assert s > 0 and z < 0.1


def test_kivi_layout_and_residual_rule():
    rng = np.random.default_rng(5)
    B, H, L, d, G, R = 2, 3, 200, 64, 32, 40
    k = rng.standard_normal((B, H, L, d)).astype(np.float32)
    v = rng.standard_normal((B, H, L, d)).astype(np.float32)
    qc = oracle.kivi_quantize(k, v, 2, G, R)
    nq = ((L - R) // G) * G
    assert qc["nq"] == nq == 160
    assert qc["kres"].shape == (B, H, L - nq, d)
    assert qc["kscale"].shape == (B, H, nq // G, d)
    assert qc["vscale"].shape == (B, H, nq, d // G)
    # K is grouped over tokens per channel, V over channels per token
    g, c = 2, 17
    codes, s, z = oracle.quantize_group(k[1, 2, g * G:(g + 1) * G, c].copy(), 2)
    assert np.array_equal(qc["kcode"][1, 2, g * G:(g + 1) * G, c], codes)
    assert (qc["kscale"][1, 2, g, c], qc["kzero"][1, 2, g, c]) == (s, z)
    t, gc = 77, 1
    codes, s, z = oracle.quantize_group(v[0, 1, t, gc * G:(gc + 1) * G].copy(), 2)
    assert np.array_equal(qc["vcode"][0, 1, t, gc * G:(gc + 1) * G], codes)
    assert (qc["vscale"][0, 1, t, gc], qc["vzero"][0, 1, t, gc]) == (s, z)
    kh, vh = oracle.kivi_dequant(qc)
    assert np.all(np.abs(kh - k[:, :, :nq]) <= np.repeat(oracle.f16_value_fast(qc["kscale"]), G, 2) / 2 * (1 + 2 ** -20))


def test_incremental_equals_one_shot():
    rng = np.random.default_rng(6)
    k = rng.standard_normal((1, 2, 128, 64)).astype(np.float32)
    v = rng.standard_normal((1, 2, 128, 64)).astype(np.float32)
    full = oracle.kivi_quantize(k, v, 4, 32, 0)
    for g in range(4):
        part = oracle.kivi_quantize(k[:, :, g * 32:(g + 1) * 32].copy(),
                                    v[:, :, g * 32:(g + 1) * 32].copy(), 4, 32, 0)
        assert np.array_equal(part["kcode"], full["kcode"][:, :, g * 32:(g + 1) * 32])
        assert np.array_equal(part["kscale"][:, :, 0], full["kscale"][:, :, g])
        assert np.array_equal(part["vcode"], full["vcode"][:, :, g * 32:(g + 1) * 32])
