"""End-to-end decoding on the GPU through the C ABI (vc_decoder_*).

1. The tiny fp32 decoder (2 layers, d_model 256, 4/2 heads, head_dim 64,
   vocab 512; 512-token prompt, seed 0): plain greedy decoding and KIVI 4-bit
   draft-and-verify (horizon 16) on the GPU emit the oracle's greedy tokens,
   except at positions whose oracle top-2 logit margin is below 1e-3 (none
   occur at this seed); accepted lengths per round equal the oracle's.
2. A small bf16 decoder on the tensor-core path: a forward over a block of
   rows gives bit for bit the logits of one-row forwards (row independence),
   and draft-and-verify (2-bit, with the full cache swapped in from pinned
   host memory every round) emits exactly the GPU's own greedy tokens.
"""
import dataclasses

import numpy as np
import pytest
import torch

from lossless_draft_verify_gb300 import inputs
from helpers import lib

pytestmark = pytest.mark.gpu


def _tiny_case():
    from oracle import model as om
    cfg = inputs.TinyConfig()
    w = inputs.tiny_weights(cfg, 0)
    prompt = inputs.tiny_prompt(cfg, 512, 0)
    return cfg, w, prompt, om


def _status_ok(vc, ws):
    torch.cuda.synchronize()
    word = int(ws.buf[:4].view(torch.int32).item())
    assert vc.vc_poll_status(ws) == 0, f"status word {word:#x}"
    return True


def _first_exempt_mismatch(got, want, margins):
    for t, (a, b) in enumerate(zip(got, want)):
        if a != b:
            assert margins[t] < 1e-3, f"token {t}: gpu {a} != oracle {b} at margin {margins[t]:.3e}"
            return t
    return None


def test_tiny_decoder_greedy_matches_oracle():
    vc = lib()
    from lossless_draft_verify_gb300 import decode
    cfg, w, prompt, om = _tiny_case()
    ref, margins = om.greedy_decode(om.TinyDecoder(w, cfg), prompt.tolist(), 64)
    dec = vc.Decoder(cfg, w, dtype=torch.float32)
    run = decode.VeriCacheRunner(dec, 1, 512 + 64, 16, bits=4, residual=0)
    run.prefill(prompt.view(1, -1).to("cuda", torch.int32))
    got = run.greedy(64)[0]
    _first_exempt_mismatch(got, ref, margins)
    assert _status_ok(vc, run.ws)


def test_tiny_decoder_draft_and_verify_matches_oracle():
    vc = lib()
    from lossless_draft_verify_gb300 import decode
    cfg, w, prompt, om = _tiny_case()
    model = om.TinyDecoder(w, cfg)
    ref, margins = om.greedy_decode(model, prompt.tolist(), 64)
    ref_dv, ref_acc = om.draft_and_verify(model, prompt.tolist(), 64, 16, "kivi", bits=4, group=32, residual=0)
    assert ref_dv == ref
    dec = vc.Decoder(cfg, w, dtype=torch.float32)
    run = decode.VeriCacheRunner(dec, 1, 512 + 64 + 32, 16, bits=4, residual=0, host_cache=True)
    run.prefill(prompt.view(1, -1).to("cuda", torch.int32))
    toks, acc = run.generate(64)
    t = _first_exempt_mismatch(toks[0], ref, margins)
    if t is None:
        assert acc[0] == ref_acc, (acc[0], ref_acc)
    assert _status_ok(vc, run.ws)


@dataclasses.dataclass
class SmallCfg:
    n_layers: int = 2
    d_model: int = 512
    n_heads: int = 8
    n_kv_heads: int = 2
    head_dim: int = 128
    d_ff: int = 1024
    vocab: int = 2048
    init_std: float = 0.02
    head_scale: float = 20.0
    rope_theta: float = 10000.0
    norm_eps: float = 1e-6


def _small_decoder(vc, seed=0):
    cfg = SmallCfg()
    w = inputs.tiny_weights(cfg, seed)
    return cfg, vc.Decoder(cfg, w, dtype=torch.bfloat16)


def test_bf16_block_forward_equals_row_by_row():
    vc = lib()
    cfg, dec = _small_decoder(vc)
    B, P, n = 2, 300, 9
    g = torch.Generator().manual_seed(3)
    toks = torch.randint(0, cfg.vocab, (B, P + n), generator=g, dtype=torch.int32).cuda()
    Ls = P + n + 8
    shape = (cfg.n_layers, B, cfg.n_kv_heads, Ls, cfg.head_dim)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vcache = torch.zeros_like(kc)
    ws = vc.Workspace(dec.workspace_bytes(B, P, Ls - P))
    ctx0 = torch.zeros(B, dtype=torch.int32, device="cuda")
    last = torch.zeros(B, cfg.vocab, dtype=torch.bfloat16, device="cuda")
    vc.vc_decoder_forward(dec, None, toks, P + n, B, P, ctx0, 0, kc, vcache, last, ws, last_only=True)
    # the block of n rows at positions P..P+n-1
    ctxP = torch.full((B,), P, dtype=torch.int32, device="cuda")
    blk = torch.zeros(B, n, cfg.vocab, dtype=torch.bfloat16, device="cuda")
    kc2, vc2 = kc.clone(), vcache.clone()
    vc.vc_decoder_forward(dec, None, toks[:, P:], P + n, B, n, ctxP, P, kc2, vc2, blk, ws)
    # the same rows one at a time
    rows = []
    for i in range(n):
        c = torch.full((B,), P + i, dtype=torch.int32, device="cuda")
        one = torch.zeros(B, cfg.vocab, dtype=torch.bfloat16, device="cuda")
        vc.vc_decoder_forward(dec, None, toks[:, P + i:], P + n, B, 1, c, P + i, kc, vcache, one, ws,
                              last_only=True)
        rows.append(one)
    torch.cuda.synchronize()
    assert _status_ok(vc, ws)
    for i in range(n):
        assert torch.equal(blk[:, i], rows[i]), f"row {i}"
    assert torch.equal(kc[:, :, :, :P + n], kc2[:, :, :, :P + n])
    assert torch.isfinite(blk.float()).all()


@pytest.mark.parametrize("host_cache", [True, False])
def test_bf16_draft_and_verify_equals_greedy(host_cache):
    vc = lib()
    from lossless_draft_verify_gb300 import decode
    cfg, dec = _small_decoder(vc, seed=1)
    B, P, n_new, D = 3, 700, 48, 8
    g = torch.Generator().manual_seed(4)
    prompt = torch.randint(0, cfg.vocab, (B, P), generator=g, dtype=torch.int32).cuda()
    ref_run = decode.VeriCacheRunner(dec, B, P + n_new + 2 * D, D, bits=2, residual=128, prefill_chunk=256)
    ref_run.prefill(prompt)
    ref = ref_run.greedy(n_new)
    run = decode.VeriCacheRunner(dec, B, P + n_new + 2 * D, D, bits=2, residual=128, host_cache=host_cache,
                                 prefill_chunk=256)
    run.prefill(prompt)
    toks, acc = run.generate(n_new)
    assert toks == ref
    assert _status_ok(vc, run.ws) and _status_ok(vc, ref_run.ws)
    assert all(0 <= a <= D for seq in acc for a in seq)
