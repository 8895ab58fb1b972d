"""Pins of the oracle's lossless packing of bf16 K/V rows for the host link
(the format in oracle/__init__.py): a hand-worked row, exact round trips on
ordinary, wide-range and special-value rows, the escape count against the
values' magnitudes, and an exhaustive check of the code/escape rule on
two-value rows against a plain scalar restatement."""
import itertools

import numpy as np
import pytest

import oracle


def bits_of(x) -> np.ndarray:
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_worked_row():
    # 1.0, -2.0, 0.5, 2^-20, 0.0, 3.0, -0.0, 1.5 (all exact in bf16)
    b = np.array([[0x3F80, 0xC000, 0x3F00, 0x3580, 0x0000, 0x4040, 0x8000, 0x3FC0]], np.uint16)
    # largest exponent field 128 (2.0, 3.0) -> base 114; 2^-20 (field 107) and
    # the two zeros (field 0) are escaped
    want = [114, 3, 3, 107, 4, 0, 6, 0, 0, 0, 0, 0, 0, 0, 0, 0,
            0xED, 0xFC, 0xEF, 0xDF,                          # codes 13 14 12 15 15 14 15 13
            0x00, 0x80, 0x00, 0x00, 0x00, 0x40, 0x80, 0x40]  # sign | mantissa
    p, over = oracle.kv_pack_rows(b)
    assert p.tolist() == [want] and not over.any()
    np.testing.assert_array_equal(oracle.kv_unpack_rows(p, 8), b)


@pytest.mark.parametrize("kind", ["normal", "wide", "zeros", "outlier"])
def test_round_trip_exact(kind):
    rng = np.random.default_rng(7)
    rows, d = 3000, 128
    x = rng.standard_normal((rows, d)).astype(np.float32)
    if kind == "wide":
        x *= np.exp(rng.uniform(-12, 12, (rows, d))).astype(np.float32)
    elif kind == "zeros":
        x[rng.random((rows, d)) < 0.02] = 0.0
        x[::7] = 0.0
    elif kind == "outlier":
        x[:, 5] *= 8.0
    b = bits_of(oracle.bf16_round(x))
    p, over = oracle.kv_pack_rows(b)
    assert p.shape == (rows, 208)
    ok = ~over
    np.testing.assert_array_equal(oracle.kv_unpack_rows(p[ok], d), b[ok])
    assert (p[over, 1] == 255).all()
    if kind in ("normal", "outlier"):
        assert not over.any()
    if kind == "wide":
        assert over.any()           # a range of 2^35 needs more than 7 escapes somewhere


def test_special_values_round_trip_or_marked():
    rng = np.random.default_rng(8)
    b = rng.integers(0, 1 << 16, (4000, 64), dtype=np.uint16)      # every bit pattern, NaN and inf included
    b[:2000, 8:] = bits_of(oracle.bf16_round(rng.standard_normal((2000, 56))))
    b[2000:2500] = 0x7F80                                            # rows of +inf
    p, over = oracle.kv_pack_rows(b)
    np.testing.assert_array_equal(oracle.kv_unpack_rows(p[~over], 64), b[~over])
    assert not over[2000:2500].any()


def test_escape_count_from_magnitudes():
    """For rows of finite nonzero values, a value is escaped exactly when it
    is below 2^-14 times the binade of the row's largest magnitude."""
    rng = np.random.default_rng(9)
    x = oracle.bf16_round(rng.standard_normal((5000, 128)) * np.exp(rng.uniform(-3, 3, (5000, 1))))
    x[x == 0] = 1.0
    p, over = oracle.kv_pack_rows(bits_of(x))
    top = np.floor(np.log2(np.abs(x).max(axis=1)))          # the binade of the largest magnitude
    want = (np.abs(x) < np.exp2(top - 14)[:, None]).sum(axis=1)
    np.testing.assert_array_equal(np.where(over, -1, p[:, 1].astype(int)), np.where(want > 7, -1, want))
    assert np.all(p[:, 0] == top + 127 - 14)


def test_two_value_rows_exhaustive():
    """Every pair of exponent fields (with sign and mantissa patterns) against
    a scalar restatement of the rule: base = max - 14 floored at 0, code =
    field - base if that is in 0..14, else escaped with the field."""
    fields = [0, 1, 2, 13, 14, 15, 16, 100, 113, 114, 120, 127, 128, 200, 254, 255]
    for e0, e1 in itertools.product(fields, fields):
        b = np.array([[(e0 << 7) | 0x35, 0x8000 | (e1 << 7) | 0x4A]], np.uint16)
        p, over = oracle.kv_pack_rows(b)
        base = max(e0, e1) - 14 if max(e0, e1) >= 14 else 0
        codes = [e - base if 0 <= e - base <= 14 else 15 for e in (e0, e1)]
        escs = [(i, e) for i, e in enumerate((e0, e1)) if codes[i] == 15]
        row = [base, len(escs)] + [v for s in escs for v in s] + [0] * (14 - 2 * len(escs))
        row += [codes[0] | (codes[1] << 4), 0x35, 0x80 | 0x4A]
        assert p[0].tolist() == row and not over[0]
        np.testing.assert_array_equal(oracle.kv_unpack_rows(p, 2), b)
