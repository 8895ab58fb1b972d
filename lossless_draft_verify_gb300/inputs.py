"""Seeded synthetic input generators shared by the tests, the smoke check and
the benchmark.

This module holds none of the method's arithmetic: it only draws random
tensors with the shapes and value distributions of the workloads and rounds
them to their storage type.  Both the CUDA path and the CPU oracle consume the
tensors it returns.  Generation uses torch's seeded generators so that the
large workloads can be drawn directly in device memory; small cases are drawn
on the CPU.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """bf16 tensor ~ N(0, std^2), drawn in fp32 and rounded to nearest bf16."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def normal_f32(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x * std if std != 1.0 else x


# --------------------------------------------------------------------------
# draft-attention workload: bf16 K/V ~ N(0,1) with fixed outlier K channels
# --------------------------------------------------------------------------

def outlier_channels(Hkv: int, d: int, n_out: int, seed: int) -> torch.Tensor:
    """[Hkv, n_out] distinct channel indices per KV head (fixed over tokens
    and sequences)."""
    g = _gen(seed, "cpu")
    return torch.stack([torch.randperm(d, generator=g)[:n_out] for _ in range(Hkv)])


def kv_with_outliers(B, Hkv, L, d, seed, device="cpu", n_out=4, out_scale=8.0,
                     dtype=torch.bfloat16):
    """K, V [B,Hkv,L,d] ~ N(0,1); n_out channels of K per head scaled by
    out_scale before rounding to the storage type."""
    g = _gen(seed, device)
    k = torch.randn(B, Hkv, L, d, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(B, Hkv, L, d, generator=g, device=device, dtype=torch.float32)
    if n_out:
        ch = outlier_channels(Hkv, d, n_out, seed + 7919).to(device)
        for h in range(Hkv):
            k[:, h, :, ch[h]] *= out_scale
    return k.to(dtype), v.to(dtype)


# --------------------------------------------------------------------------
# greedy-acceptance workload: logits ~ N(0,1) with a planted unique row
# maximum, drafts that follow it up to a random divergence point
# --------------------------------------------------------------------------

@dataclass
class AcceptCase:
    logits: torch.Tensor          # [B, D+1, V]
    drafts: torch.Tensor          # [B, D] int32
    diverge: torch.Tensor         # [B] int32: index of the first mismatching draft (D: none)
    planted: torch.Tensor         # [B, D+1] int32: position of the planted maximum


def accept_case(B, D, V, seed, device="cpu", dtype=torch.bfloat16, clamp=6.0, peak=8.0,
                diverge=None) -> AcceptCase:
    """Row values ~ N(0,1) clamped to [-clamp, clamp]; one planted entry per
    row set to `peak` (> clamp), so the row maximum is unique by construction.
    Drafts copy the planted positions up to a per-sequence divergence point
    k ~ U{0..D}; draft k (if k < D) is a different position, later drafts are
    uniform.  The expected accepted length is therefore k without any argmax
    being taken here."""
    g = _gen(seed, device)
    lg = torch.randn(B, D + 1, V, generator=g, device=device, dtype=torch.float32)
    lg.clamp_(-clamp, clamp)
    gc = _gen(seed + 1, "cpu")
    planted = torch.randint(0, V, (B, D + 1), generator=gc, dtype=torch.int64)
    if diverge is None:
        kdiv = torch.randint(0, D + 1, (B,), generator=gc, dtype=torch.int64)
    else:
        kdiv = torch.as_tensor(diverge, dtype=torch.int64).reshape(B)
    drafts = torch.randint(0, V, (B, max(D, 1)), generator=gc, dtype=torch.int64)[:, :D].clone()
    for b in range(B):
        k = int(kdiv[b])
        drafts[b, :k] = planted[b, :k]
        if k < D:
            off = int(torch.randint(1, V, (1,), generator=gc))
            drafts[b, k] = (planted[b, k] + off) % V
    lg.scatter_(2, planted.to(device).unsqueeze(-1), peak)
    return AcceptCase(lg.to(dtype), drafts.to(torch.int32).to(device), kdiv.to(torch.int32),
                      planted.to(torch.int32))


# --------------------------------------------------------------------------
# token-dropping workload: Zipf(1.1) accumulated scores over a random
# permutation of positions
# --------------------------------------------------------------------------

def zipf_scores(B, H, L, seed, a=1.1, device="cpu") -> torch.Tensor:
    """scores[b,h,pos] = (rank+1)^-a with rank a seeded random permutation of
    positions per (b,h); all values distinct in fp32 for L <= 2^17."""
    g = _gen(seed, "cpu")
    ranks = torch.stack([torch.randperm(L, generator=g) for _ in range(B * H)]).reshape(B, H, L)
    s = (ranks.to(torch.float64) + 1.0).pow(-a).to(torch.float32)
    return s.to(device)


# --------------------------------------------------------------------------
# tiny random-init decoder (the 2-layer fp32 model of the end-to-end check)
# --------------------------------------------------------------------------

@dataclass
class TinyConfig:
    n_layers: int = 2
    d_model: int = 256
    n_heads: int = 4
    n_kv_heads: int = 2
    head_dim: int = 64
    d_ff: int = 512
    vocab: int = 512
    init_std: float = 0.02
    head_scale: float = 20.0
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6


def tiny_weights(cfg: TinyConfig, seed: int = 0) -> dict:
    """fp32 weights ~ N(0, 0.02^2), LM head scaled by 20; matrices are stored
    [in, out] so that a row vector times the matrix gives the projection."""
    g = _gen(seed, "cpu")

    def w(i, o, s=1.0):
        return (torch.randn(i, o, generator=g, dtype=torch.float32) * (cfg.init_std * s))

    D, F = cfg.d_model, cfg.d_ff
    qd, kvd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    out = {"embed": w(cfg.vocab, D), "layers": []}
    for _ in range(cfg.n_layers):
        out["layers"].append({"wq": w(D, qd), "wk": w(D, kvd), "wv": w(D, kvd),
                              "wo": w(qd, D), "wg": w(D, F), "wu": w(D, F), "wd": w(F, D)})
    out["lm_head"] = w(D, cfg.vocab, cfg.head_scale)
    return out


def tiny_prompt(cfg: TinyConfig, length: int = 512, seed: int = 0) -> torch.Tensor:
    g = _gen(seed, "cpu")
    return torch.randint(0, cfg.vocab, (length,), generator=g, dtype=torch.int64)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


# --------------------------------------------------------------------------
# 8-layer GQA decoder of the end-to-end workload (7B-class widths)
# --------------------------------------------------------------------------

@dataclass
class DecoderConfig:
    n_layers: int = 8
    d_model: int = 4096
    n_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    d_ff: int = 14336
    vocab: int = 32000
    init_std: float = 0.02
    head_scale: float = 20.0
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6


def decoder_weights_packed(cfg, seed: int = 0, device="cuda", dtype=torch.bfloat16) -> dict:
    """Weights ~ N(0, 0.02^2) (LM head x20) drawn on `device` directly in the
    layout the decoder takes: embed [vocab][d], lm_head [d][vocab] and per
    layer wqkv [d][(Hq+2Hkv) hd] (q|k|v), wo [Hq hd][d], wgu [d][2 ff]
    (gate and up columns interleaved per 64, the decoder's layout; every
    column is an independent draw, so the layout only names which columns are
    gate and which are up), wd [ff][d]."""
    g = _gen(seed, device)

    def w(i, o, s=1.0):
        x = torch.randn(i, o, generator=g, device=device, dtype=torch.float32)
        return x.mul_(cfg.init_std * s).to(dtype)

    D, F = cfg.d_model, cfg.d_ff
    qd, kvd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    out = {"embed": w(cfg.vocab, D), "wqkv": [], "wo": [], "wgu": [], "wd": []}
    for _ in range(cfg.n_layers):
        out["wqkv"].append(w(D, qd + 2 * kvd))
        out["wo"].append(w(qd, D))
        out["wgu"].append(w(D, 2 * F))
        out["wd"].append(w(F, D))
    out["lm_head"] = w(D, cfg.vocab, cfg.head_scale)
    return out


def random_prompts(B: int, length: int, vocab: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Uniform random token ids [B][length] (int32)."""
    g = _gen(seed, "cpu")
    return torch.randint(0, vocab, (B, length), generator=g, dtype=torch.int32).to(device)
