"""Pins of the oracle's tiny-decoder forward (oracle/model.py) against what the
Llama-style reading of the decoder fixes: rotate-half RoPE with theta 10000,
RMSNorm with eps inside the root, SwiGLU, grouped-query attention with query
head h reading kv head h // (Hq/Hkv), causal attention.  The pages run trained
LLMs and specify none of this (paper page, "What the paper found"); the reading
is the plainest one the rest of the pages support.

Each pin is chosen so that a plausible slip fails it: RoPE pairing or sign
(the worked 2-pair example), eps placement (the closed-form RMS), a gate/up swap
(the worked SwiGLU case), and any mistake in wiring the pieces together (a full
forward against a second, differently written implementation)."""
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

from lossless_draft_verify_gb300 import inputs
from oracle import model as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "decoder_pieces.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = np.array([float(v) for v in vals])
    return out


# ---------------------------------------------------------------- RoPE

def test_rope_worked_two_pair_example():
    g = _golden()
    x = g["rope_x"][None, :]                      # one head, head_dim 4
    got = om._rope(x, int(g["rope_pos"][0]), 10000.0)[0]
    np.testing.assert_allclose(got, g["rope_out"], rtol=0, atol=1e-15)


def test_rope_at_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((4, 64))
    assert np.array_equal(om._rope(x, 0, 10000.0), x)


def test_rope_rotates_each_pair_by_its_angle():
    hd, pos, theta = 64, 37, 10000.0
    x = np.random.default_rng(1).standard_normal((3, hd))
    y = om._rope(x, pos, theta)
    half = hd // 2
    for i in range(half):
        a = complex(x[0, i], x[0, i + half])
        b = complex(y[0, i], y[0, i + half])
        # norm of the pair kept, angle advanced by pos * theta^(-2i/hd)
        assert abs(abs(b) - abs(a)) < 1e-12
        want = pos * theta ** (-2.0 * i / hd)
        turn = math.remainder(np.angle(b / a) - want, 2 * math.pi)
        assert abs(turn) < 1e-9, (i, turn)


def test_rope_scores_depend_only_on_relative_position():
    hd = 64
    r = np.random.default_rng(2)
    q, k = r.standard_normal((1, hd)), r.standard_normal((1, hd))
    ref = float((om._rope(q, 20, 1e4) * om._rope(k, 13, 1e4)).sum())
    for m, n in [(7, 0), (107, 100), (1007, 1000)]:
        s = float((om._rope(q, m, 1e4) * om._rope(k, n, 1e4)).sum())
        assert abs(s - ref) < 1e-9 * max(1.0, abs(ref))


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_worked_example_pins_eps_inside_the_root():
    g = _golden()
    got = om._rmsnorm(g["rms_x"], float(g["rms_eps"][0]))
    np.testing.assert_allclose(got, g["rms_out"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_rmsnorm_output_rms_closed_form(eps):
    x = np.random.default_rng(3).standard_normal(256) * 0.3
    ms = float(np.mean(x * x))
    y = om._rmsnorm(x, eps)
    assert abs(float(np.mean(y * y)) - ms / (ms + eps)) < 1e-13
    # direction kept
    assert abs(float(np.dot(x, y)) / (np.linalg.norm(x) * np.linalg.norm(y)) - 1) < 1e-13


# ---------------------------------------------------------------- SwiGLU

class _Cfg:
    def __init__(self, **kw):
        self.__dict__.update(kw)


def test_swiglu_worked_two_wide_case():
    g = _golden()
    cfg = _Cfg(n_layers=1, d_model=2, n_heads=1, n_kv_heads=1, head_dim=2, d_ff=2,
               vocab=2, rope_theta=1e4, norm_eps=0.0)
    eye = np.eye(2)
    w = {"embed": eye, "lm_head": eye,
         "layers": [{"wq": eye, "wk": eye, "wv": eye, "wo": np.zeros((2, 2)),
                     "wg": eye, "wu": np.diag([2.0, 3.0]), "wd": eye}]}
    m = om.TinyDecoder(w, cfg)
    got = m.post_attn(0, g["swiglu_h"], np.zeros((1, 2)))
    np.testing.assert_allclose(got, g["swiglu_out"], rtol=0, atol=1e-15)


# ---------------------------------------------------------------- whole forward

def _second_forward(weights, cfg, tokens):
    """The same decoder written a second way: float64 torch matmuls over the
    whole sequence, RoPE as a complex rotation, attention through an explicit
    causal mask and scipy's softmax, GQA by repeating kv heads.  Returns the
    logits of every position."""
    f = {k: torch.as_tensor(np.asarray(v), dtype=torch.float64)
         for k, v in (("embed", weights["embed"]), ("lm_head", weights["lm_head"]))}
    T, hd, Hq, Hkv = len(tokens), cfg.head_dim, cfg.n_heads, cfg.n_kv_heads
    half = hd // 2
    freqs = cfg.rope_theta ** (-np.arange(half) * 2.0 / hd)
    rot = np.exp(1j * np.outer(np.arange(T), freqs))          # [T, half]

    def rope(x):                                               # x [T, H, hd]
        z = (x[..., :half] + 1j * x[..., half:]) * rot[:, None, :]
        return np.concatenate([z.real, z.imag], axis=-1)

    def norm(x):
        return x / np.sqrt((x ** 2).sum(-1, keepdims=True) / x.shape[-1] + cfg.norm_eps)

    h = f["embed"][torch.as_tensor(tokens)].numpy()
    mask = np.triu(np.full((T, T), -np.inf), 1)
    for lw in weights["layers"]:
        W = {k: np.asarray(v, dtype=np.float64) for k, v in lw.items()}
        x = norm(h)
        q = rope((x @ W["wq"]).reshape(T, Hq, hd))
        k = rope((x @ W["wk"]).reshape(T, Hkv, hd))
        v = (x @ W["wv"]).reshape(T, Hkv, hd)
        k = np.repeat(k, Hq // Hkv, axis=1)
        v = np.repeat(v, Hq // Hkv, axis=1)
        s = np.einsum("thd,uhd->htu", q, k) / math.sqrt(hd) + mask[None]
        o = np.einsum("htu,uhd->thd", softmax(s, axis=-1), v).reshape(T, Hq * hd)
        h = h + o @ W["wo"]
        x = norm(h)
        gte, up = x @ W["wg"], x @ W["wu"]
        h = h + (gte * expit(gte) * up) @ W["wd"]
    return norm(h) @ f["lm_head"].numpy()


def test_forward_block_matches_a_second_implementation():
    cfg = inputs.TinyConfig()
    wt = inputs.tiny_weights(cfg, seed=5)
    w64 = {"embed": wt["embed"].double().numpy(), "lm_head": wt["lm_head"].double().numpy(),
           "layers": [{k: v.double().numpy() for k, v in lw.items()} for lw in wt["layers"]]}
    toks = inputs.tiny_prompt(cfg, 11, seed=5).tolist()
    want = _second_forward(w64, cfg, toks)

    m = om.TinyDecoder(wt, cfg)
    cache = om.FullKV(m)
    lg0, _ = om.forward_block(m, cache, toks[:8], 0)          # prompt
    lg1, _ = om.forward_block(m, cache, toks[8:], 8)          # a later block
    got = np.concatenate([lg0, lg1])
    scale = np.abs(want).max()
    assert np.abs(got - want).max() <= 1e-12 * scale
    # the logits are not degenerate: rows differ and the argmax varies
    assert len({int(np.argmax(r)) for r in want}) > 3
