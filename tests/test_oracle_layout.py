"""Pin of the oracle's packed-record reader against hand-derived probes of the
documented layout (tests/golden/record_layout.txt)."""
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "record_layout.txt")


def _rows():
    with open(GOLD) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_record_size():
    assert oracle.record_bytes(2, 128) == 3072
    assert oracle.record_bytes(4, 128) == 5120
    assert oracle.record_bytes(4, 64) == 2560


def test_single_bit_probes():
    for r in _rows():
        bits = int(r[1])
        rec = np.zeros(oracle.record_bytes(bits, 128), np.uint8)
        if r[0] == "code":
            byte, bit, sec, tok, ch = int(r[2]), int(r[3]), r[4], int(r[5]), int(r[6])
            rec[byte] = 1 << bit                     # code value 1
            out = oracle.unpack_records(rec, bits, 128)
            arr = out["kcode"] if sec == "K" else out["vcode"]
            other = out["vcode"] if sec == "K" else out["kcode"]
            assert arr[tok, ch] == 1, r
            assert arr.sum() == 1 and other.sum() == 0, r
        else:
            byte, name, row, col = int(r[2]), r[3], int(r[4]), int(r[5])
            rec[byte:byte + 2] = np.frombuffer(np.uint16(0x3C00).tobytes(), np.uint8)
            out = oracle.unpack_records(rec, bits, 128)
            assert out[name][row, col] == 0x3C00, r
            total = sum(int((out[n] != 0).sum()) for n in ("kscale", "kzero", "vscale", "vzero"))
            assert total == 1, r


def test_every_code_slot_maps_to_a_distinct_cell():
    # setting every code to its maximum in turn covers the (token, channel)
    # grid exactly once per section
    for bits in (2, 4):
        for d in (64, 128):
            rb = oracle.record_bytes(bits, d)
            ncode = 32 * d * bits // 8
            rec = np.zeros(rb, np.uint8)
            rec[:2 * ncode] = 0xFF
            out = oracle.unpack_records(rec, bits, d)
            assert np.all(out["kcode"] == (1 << bits) - 1)
            assert np.all(out["vcode"] == (1 << bits) - 1)
