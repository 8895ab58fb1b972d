"""fp64 oracle of the tiny decoder, plain greedy decoding, and the VeriCache
draft-and-verify loop.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows the paper page ("What the paper found", abstract): the target model
drafts with a lossy copy of its KV state, one causal pass over the exact state
checks the drafted block, and the emitted tokens equal plain greedy decoding.
The acceptance rule is the greedy rule of speculative decoding (source 2 on
the podparley page): keep the longest drafted prefix that matches the verify
argmax, then emit the verify argmax at the first mismatch.

The model itself is not specified by the pages (they run a trained LLM); the
tiny decoder is the plainest Llama-style reading: pre-RMSNorm (weight 1),
rotate-half RoPE on q and k before caching, grouped-query attention with q-head
h reading kv-head h // (Hq/Hkv), SwiGLU MLP, final RMSNorm, untied LM head.

Determinism: every row is computed by the same element-wise numpy code, with
no BLAS call, so the verify pass over a block and step-by-step decoding perform
bit-identical arithmetic on each row.  That makes the losslessness property
exact in this oracle, not merely up to rounding.
"""
from __future__ import annotations

import numpy as np

from . import kivi_quantize, f16_value_fast


def _vecmat(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Row vector x [n] times w [n, m], accumulated row by row in order."""
    return (x[:, None] * w).sum(axis=0)


def _rmsnorm(x: np.ndarray, eps: float) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x) + eps)


def _rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """x [H, hd]; rotate-half RoPE: pair (i, i + hd/2) rotated by pos*theta^(-2i/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / hd)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One query [hd] against K, V [n, hd]: softmax(q K^T scale) V, fp64."""
    s = (K * q[None, :]).sum(axis=1) * scale
    m = s.max()
    p = np.exp(s - m)
    return (p[:, None] * V).sum(axis=0) / p.sum()


class TinyDecoder:
    """fp64 forward of the tiny decoder; weights come from the shared seeded
    generator as fp32 tensors and are widened exactly to fp64."""

    def __init__(self, weights: dict, cfg):
        def f(t):
            return np.asarray(t.detach().cpu().numpy() if hasattr(t, "detach") else t,
                              dtype=np.float64)
        self.cfg = cfg
        self.embed = f(weights["embed"])
        self.layers = [{k: f(v) for k, v in lw.items()} for lw in weights["layers"]]
        self.lm_head = f(weights["lm_head"])
        self.scale = 1.0 / np.sqrt(cfg.head_dim)

    # -- per-row pieces -----------------------------------------------------
    def qkv(self, layer: int, h: np.ndarray, pos: int):
        c, lw = self.cfg, self.layers[layer]
        x = _rmsnorm(h, c.norm_eps)
        q = _vecmat(x, lw["wq"]).reshape(c.n_heads, c.head_dim)
        k = _vecmat(x, lw["wk"]).reshape(c.n_kv_heads, c.head_dim)
        v = _vecmat(x, lw["wv"]).reshape(c.n_kv_heads, c.head_dim)
        return _rope(q, pos, c.rope_theta), _rope(k, pos, c.rope_theta), v

    def post_attn(self, layer: int, h: np.ndarray, o: np.ndarray) -> np.ndarray:
        c, lw = self.cfg, self.layers[layer]
        h = h + _vecmat(o.reshape(-1), lw["wo"])
        x = _rmsnorm(h, c.norm_eps)
        g = _vecmat(x, lw["wg"])
        u = _vecmat(x, lw["wu"])
        return h + _vecmat((g / (1.0 + np.exp(-g))) * u, lw["wd"])

    def logits(self, h: np.ndarray) -> np.ndarray:
        return _vecmat(_rmsnorm(h, self.cfg.norm_eps), self.lm_head)

    def attend_heads(self, q, Ks, Vs):
        """q [Hq, hd]; Ks/Vs: per kv head arrays [n, hd]."""
        grp = self.cfg.n_heads // self.cfg.n_kv_heads
        return np.stack([_attend(q[h], Ks[h // grp], Vs[h // grp], self.scale)
                         for h in range(self.cfg.n_heads)])


def argmax_lowest(x: np.ndarray) -> int:
    """argmax with the lowest index on ties (numpy's argmax returns the first
    occurrence of the maximum)."""
    return int(np.argmax(x))


class FullKV:
    """Full-precision KV cache: per layer, per kv head, a growing [n, hd] array."""

    def __init__(self, model: TinyDecoder):
        c = model.cfg
        self.K = [[np.zeros((0, c.head_dim)) for _ in range(c.n_kv_heads)] for _ in range(c.n_layers)]
        self.V = [[np.zeros((0, c.head_dim)) for _ in range(c.n_kv_heads)] for _ in range(c.n_layers)]

    def length(self) -> int:
        return self.K[0][0].shape[0]

    def append(self, layer, k, v):
        for h in range(k.shape[0]):
            self.K[layer][h] = np.concatenate([self.K[layer][h], k[h][None]], axis=0)
            self.V[layer][h] = np.concatenate([self.V[layer][h], v[h][None]], axis=0)

    def truncate(self, n):
        for layer in range(len(self.K)):
            for h in range(len(self.K[layer])):
                self.K[layer][h] = self.K[layer][h][:n]
                self.V[layer][h] = self.V[layer][h][:n]


def forward_block(model: TinyDecoder, cache: FullKV, tokens, pos0: int):
    """Run tokens at positions pos0.. against the full cache (causal), append
    their K/V, return (logits [n, V], per-layer K/V of the block)."""
    c = model.cfg
    hs = [model.embed[t].copy() for t in tokens]
    new_kv = []
    for layer in range(c.n_layers):
        qs, ks, vs = [], [], []
        for i, h in enumerate(hs):
            q, k, v = model.qkv(layer, h, pos0 + i)
            qs.append(q)
            ks.append(k)
            vs.append(v)
        for i in range(len(hs)):
            cache.append(layer, ks[i], vs[i])
        new_kv.append((np.stack(ks), np.stack(vs)))
        n_before = cache.K[layer][0].shape[0] - len(hs)
        outs = []
        for i in range(len(hs)):
            n = n_before + i + 1                    # causal: keys 0 .. pos0 + i
            Ks = [cache.K[layer][h][:n] for h in range(c.n_kv_heads)]
            Vs = [cache.V[layer][h][:n] for h in range(c.n_kv_heads)]
            outs.append(model.attend_heads(qs[i], Ks, Vs))
        hs = [model.post_attn(layer, hs[i], outs[i]) for i in range(len(hs))]
    return np.stack([model.logits(h) for h in hs]), new_kv


def greedy_decode(model: TinyDecoder, prompt, n_new: int):
    """Plain full-KV greedy decoding: the losslessness reference."""
    cache = FullKV(model)
    lg, _ = forward_block(model, cache, list(prompt), 0)
    out = [argmax_lowest(lg[-1])]
    margins = [_margin(lg[-1])]
    while len(out) < n_new:
        pos = cache.length()
        lg, _ = forward_block(model, cache, [out[-1]], pos)
        out.append(argmax_lowest(lg[-1]))
        margins.append(_margin(lg[-1]))
    return out, margins


def _margin(row: np.ndarray) -> float:
    """Gap between the largest and the second-largest logit."""
    top2 = np.sort(row)[-2:]
    return float(top2[1] - top2[0])


class KiviDraftCache:
    """The compressed (draft) cache: per layer and kv head, KIVI-quantized
    groups of G tokens (dequantized to fp64 by x^ = code*s + z) followed by a
    full-precision residual of fp32-rounded K/V.  Groups are aligned to
    position 0, so quantizing incrementally equals quantizing in one shot."""

    def __init__(self, model: TinyDecoder, bits: int, group: int, residual: int):
        c = model.cfg
        self.c, self.bits, self.G, self.R = c, bits, group, residual
        self.qK = [[np.zeros((0, c.head_dim)) for _ in range(c.n_kv_heads)] for _ in range(c.n_layers)]
        self.qV = [[np.zeros((0, c.head_dim)) for _ in range(c.n_kv_heads)] for _ in range(c.n_layers)]
        self.rK = [[np.zeros((0, c.head_dim), np.float32) for _ in range(c.n_kv_heads)] for _ in range(c.n_layers)]
        self.rV = [[np.zeros((0, c.head_dim), np.float32) for _ in range(c.n_kv_heads)] for _ in range(c.n_layers)]

    def length(self):
        return self.qK[0][0].shape[0] + self.rK[0][0].shape[0]

    def append(self, layer, k, v):
        for h in range(k.shape[0]):
            self.rK[layer][h] = np.concatenate([self.rK[layer][h], k[h][None].astype(np.float32)])
            self.rV[layer][h] = np.concatenate([self.rV[layer][h], v[h][None].astype(np.float32)])

    def truncate(self, n):
        """Roll back to n tokens (never below the quantized prefix)."""
        for layer in range(self.c.n_layers):
            for h in range(self.c.n_kv_heads):
                nq = self.qK[layer][h].shape[0]
                assert n >= nq
                self.rK[layer][h] = self.rK[layer][h][:n - nq]
                self.rV[layer][h] = self.rV[layer][h][:n - nq]

    def requantize(self):
        """Quantize every full group that has left the residual window."""
        for layer in range(self.c.n_layers):
            for h in range(self.c.n_kv_heads):
                while self.rK[layer][h].shape[0] - self.G >= self.R:
                    gk = self.rK[layer][h][:self.G]
                    gv = self.rV[layer][h][:self.G]
                    qc = kivi_quantize(gk[None, None], gv[None, None], self.bits, self.G, 0)
                    G, d = self.G, self.c.head_dim
                    ks = f16_value_fast(qc["kscale"][0, 0])           # [1, d]
                    kz = f16_value_fast(qc["kzero"][0, 0])
                    vs = f16_value_fast(qc["vscale"][0, 0])           # [G, d/G]
                    vz = f16_value_fast(qc["vzero"][0, 0])
                    kh = qc["kcode"][0, 0].astype(np.float64) * ks + kz
                    vh = (qc["vcode"][0, 0].astype(np.float64) * np.repeat(vs, G, axis=1)
                          + np.repeat(vz, G, axis=1))
                    assert kh.shape == (G, d)
                    self.qK[layer][h] = np.concatenate([self.qK[layer][h], kh])
                    self.qV[layer][h] = np.concatenate([self.qV[layer][h], vh])
                    self.rK[layer][h] = self.rK[layer][h][self.G:]
                    self.rV[layer][h] = self.rV[layer][h][self.G:]

    def keys(self, layer, h):
        return np.concatenate([self.qK[layer][h], self.rK[layer][h].astype(np.float64)])

    def values(self, layer, h):
        return np.concatenate([self.qV[layer][h], self.rV[layer][h].astype(np.float64)])


class IdentityDraftCache:
    """The identity compressor: the draft cache is the full-precision cache."""

    def __init__(self, model: TinyDecoder):
        self.full = FullKV(model)
        self.c = model.cfg

    def length(self):
        return self.full.length()

    def append(self, layer, k, v):
        self.full.append(layer, k, v)

    def truncate(self, n):
        self.full.truncate(n)

    def requantize(self):
        pass

    def keys(self, layer, h):
        return self.full.K[layer][h]

    def values(self, layer, h):
        return self.full.V[layer][h]


def draft_step(model: TinyDecoder, dcache, token: int, pos: int) -> np.ndarray:
    """One draft step on the compressed cache: append the token's K/V, attend
    over every cached token, return logits."""
    c = model.cfg
    h = model.embed[token].copy()
    for layer in range(c.n_layers):
        q, k, v = model.qkv(layer, h, pos)
        dcache.append(layer, k, v)
        Ks = [dcache.keys(layer, i) for i in range(c.n_kv_heads)]
        Vs = [dcache.values(layer, i) for i in range(c.n_kv_heads)]
        h = model.post_attn(layer, h, model.attend_heads(q, Ks, Vs))
    return model.logits(h)


def draft_and_verify(model: TinyDecoder, prompt, n_new: int, horizon: int,
                     compressor: str = "kivi", bits: int = 4, group: int = 32,
                     residual: int = 0):
    """VeriCache decoding.  Returns (tokens, accepted lengths per round).

    Round: the pending token x sits at position P (its K/V not yet cached).
    Draft D tokens on the compressed cache (inputs x, d1..d_{D-1}); verify
    [x, d1..dD] at positions P..P+D on the full cache; n = longest prefix with
    argmax(row i) == d_{i+1}; emit d1..dn and argmax(row n); keep the verify
    pass's K/V of the n+1 committed inputs in both caches (the draft cache is
    rolled back to P first and re-quantized)."""
    full = FullKV(model)
    lg, new_kv = forward_block(model, full, list(prompt), 0)
    if compressor == "kivi":
        dc = KiviDraftCache(model, bits, group, residual)
    elif compressor == "identity":
        dc = IdentityDraftCache(model)
    else:
        raise ValueError(compressor)
    for layer, (ks, vs) in enumerate(new_kv):
        for i in range(ks.shape[0]):
            dc.append(layer, ks[i], vs[i])
    dc.requantize()
    out = [argmax_lowest(lg[-1])]
    accepted = []
    while len(out) < n_new:
        P = full.length()
        x = out[-1]
        drafts, tok = [], x
        for j in range(horizon):
            dl = draft_step(model, dc, tok, P + j)
            tok = argmax_lowest(dl)
            drafts.append(tok)
        vl, vkv = forward_block(model, full, [x] + drafts, P)
        n = horizon
        for i in range(horizon):
            if argmax_lowest(vl[i]) != drafts[i]:
                n = i
                break
        nxt = argmax_lowest(vl[n])
        accepted.append(n)
        full.truncate(P + n + 1)
        dc.truncate(P)
        for layer, (ks, vs) in enumerate(vkv):
            for i in range(n + 1):
                dc.append(layer, ks[i], vs[i])
        dc.requantize()
        out.extend(drafts[:n] + [nxt])
    return out[:n_new], accepted
