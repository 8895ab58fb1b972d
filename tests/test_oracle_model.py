"""Pins of the oracle's decoding loop: the draft-and-verify output equals plain
full-KV greedy decoding (the pages' losslessness claim, paper page "What the
paper found" and abstract), and with the identity compressor every round
accepts the whole horizon."""
import numpy as np
import pytest

from lossless_draft_verify_gb300 import inputs
from oracle import model as om


def _tiny(prompt_len, seed=0):
    cfg = inputs.TinyConfig()
    m = om.TinyDecoder(inputs.tiny_weights(cfg, seed), cfg)
    return m, inputs.tiny_prompt(cfg, prompt_len, seed).tolist()


def test_draft_and_verify_equals_greedy_kivi4():
    m, prompt = _tiny(512)
    ref, margins = om.greedy_decode(m, prompt, 64)
    toks, acc = om.draft_and_verify(m, prompt, 64, 16, "kivi", bits=4, group=32, residual=0)
    assert toks == ref
    assert len(acc) >= 1 and all(0 <= a <= 16 for a in acc)


def test_draft_and_verify_equals_greedy_kivi2_short_prompt():
    m, prompt = _tiny(96, seed=1)
    ref, _ = om.greedy_decode(m, prompt, 40)
    toks, acc = om.draft_and_verify(m, prompt, 40, 8, "kivi", bits=2, group=32, residual=16)
    assert toks == ref


def test_identity_compressor_accepts_full_horizon():
    m, prompt = _tiny(128, seed=2)
    ref, _ = om.greedy_decode(m, prompt, 33)
    toks, acc = om.draft_and_verify(m, prompt, 33, 8, "identity")
    assert toks == ref
    assert acc == [8] * len(acc)


def test_a_wrong_verify_would_be_caught():
    # planted mistake, on the CPU, in a copy of the oracle: if the verify pass
    # used the compressed cache, the output would drift from greedy decoding
    m, prompt = _tiny(160, seed=3)
    ref, _ = om.greedy_decode(m, prompt, 48)
    dc = om.KiviDraftCache(m, 2, 32, 0)
    full = om.FullKV(m)
    lg, kv = om.forward_block(m, full, prompt, 0)
    for layer, (ks, vs) in enumerate(kv):
        for i in range(ks.shape[0]):
            dc.append(layer, ks[i], vs[i])
    dc.requantize()
    out = [om.argmax_lowest(lg[-1])]
    while len(out) < 48:               # lossy decoding: draft cache only
        out.append(om.argmax_lowest(om.draft_step(m, dc, out[-1], dc.length())))
    assert out != ref
