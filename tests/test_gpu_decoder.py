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


@pytest.mark.parametrize("host_cache,fused_head,rotate,graph,pack", [(True, True, False, False, False),
                                                                  (False, True, False, False, False),
                                                                  (False, False, False, False, False),
                                                                  (False, True, True, False, False),
                                                                  (True, True, False, True, False),
                                                                  (True, True, False, True, True)])
def test_bf16_draft_and_verify_equals_greedy(host_cache, fused_head, rotate, graph, pack):
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
                                 prefill_chunk=256, fused_head=fused_head, rotate=rotate, use_graph=graph,
                                 pack_host=pack)
    run.prefill(prompt)
    toks, acc = run.generate(n_new)
    assert run.pack_host == pack
    assert (run._graph is not None) == graph
    assert toks == ref
    assert _status_ok(vc, run.ws) and _status_ok(vc, ref_run.ws)
    assert all(0 <= a <= D for seq in acc for a in seq)


@pytest.mark.parametrize("pack,graph", [(True, True), (False, False)])
def test_staggered_groups_equal_greedy(pack, graph):
    """Two request groups ping-ponging (decode.StaggeredPair: one group's swap
    runs while the other drafts and verifies) emit exactly the greedy tokens of
    their own sequences, and a host copy that the swaps read stays consistent
    across the interleaving."""
    vc = lib()
    from lossless_draft_verify_gb300 import decode
    cfg, dec = _small_decoder(vc, seed=1)
    B, P, n_new, D = 4, 700, 40, 8
    g = torch.Generator().manual_seed(5)
    prompt = torch.randint(0, cfg.vocab, (B, P), generator=g, dtype=torch.int32).cuda()
    ref_run = decode.VeriCacheRunner(dec, B, P + n_new + 2 * D, D, bits=2, residual=128, prefill_chunk=256)
    ref_run.prefill(prompt)
    ref = ref_run.greedy(n_new)
    runs = [decode.VeriCacheRunner(dec, 2, P + n_new * (D + 1) + 2 * D, D, bits=2, residual=128, host_cache=True,
                                   prefill_chunk=256, pack_host=pack) for _ in range(2)]
    runs[0].prefill(prompt[:2].contiguous())
    runs[1].prefill(prompt[2:].contiguous())
    first = runs[0].x.cpu().tolist() + runs[1].x.cpu().tolist()
    pair = decode.StaggeredPair(*runs)
    cycles = n_new
    logs = [r.new_log(cycles) for r in runs]
    for i in range(cycles):
        if graph and i == 2:
            torch.cuda.synchronize()
            for r in runs:
                r.capture_draft_graph()
        pair.cycle(logs[0], logs[1], i)
    torch.cuda.synchronize()
    toks = [[first[b]] + t for b, t in enumerate(logs[0].tokens() + logs[1].tokens())]
    for b in range(B):
        assert toks[b][:n_new] == ref[b], b
    for r in runs:
        r.check_packed()
        assert _status_ok(vc, r.ws)


def test_bf16_fused_verify_equals_logits_and_scan():
    """vc_decoder_verify (LM head with the argmax epilogue, acceptance over the
    tile maxima) gives the n_acc / next that the oracle's acceptance finds on
    the logits vc_decoder_forward writes, with drafts that follow the greedy
    tokens for a random number of rows and then diverge."""
    import oracle
    vc = lib()
    cfg, dec = _small_decoder(vc, seed=2)
    B, P, D = 4, 200, 6
    g = torch.Generator().manual_seed(5)
    prompt = torch.randint(0, cfg.vocab, (B, P), generator=g, dtype=torch.int32).cuda()
    Ls = P + D + 8
    shape = (cfg.n_layers, B, cfg.n_kv_heads, Ls, cfg.head_dim)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vcache = torch.zeros_like(kc)
    ws = vc.Workspace(dec.workspace_bytes(B, P, Ls - P))
    ctx0 = torch.zeros(B, dtype=torch.int32, device="cuda")
    last = torch.zeros(B, cfg.vocab, dtype=torch.bfloat16, device="cuda")
    vc.vc_decoder_forward(dec, None, prompt, P, B, P, ctx0, 0, kc, vcache, last, ws, last_only=True)
    torch.cuda.synchronize()
    x = torch.tensor(oracle.accept(last.float().cpu().numpy()[:, None, :], np.zeros((B, 0), np.int32))[1],
                     dtype=torch.int32, device="cuda")
    ctxP = torch.full((B,), P, dtype=torch.int32, device="cuda")
    # greedy drafts for every row: one forward per row on a copy of the cache
    kg, vg = kc.clone(), vcache.clone()
    tok, greedy = x.clone(), []
    for i in range(D):
        c = torch.full((B,), P + i, dtype=torch.int32, device="cuda")
        one = torch.zeros(B, cfg.vocab, dtype=torch.bfloat16, device="cuda")
        vc.vc_decoder_forward(dec, tok, None, 0, B, 1, c, P + i, kg, vg, one, ws, last_only=True)
        torch.cuda.synchronize()
        tok = torch.tensor(oracle.accept(one.float().cpu().numpy()[:, None, :], np.zeros((B, 0), np.int32))[1],
                           dtype=torch.int32, device="cuda")
        greedy.append(tok)
    drafts = torch.stack(greedy, 1).contiguous()
    keep = [0, 2, D, 4]                          # rows of each sequence that follow the greedy tokens
    for b, k in enumerate(keep):
        if k < D:
            drafts[b, k] = (drafts[b, k] + 1) % cfg.vocab
    logits = torch.zeros(B, D + 1, cfg.vocab, dtype=torch.bfloat16, device="cuda")
    k1, v1 = kc.clone(), vcache.clone()
    vc.vc_decoder_forward(dec, x, drafts, D, B, D + 1, ctxP, P, k1, v1, logits, ws)
    n_acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    k2, v2 = kc.clone(), vcache.clone()
    vc.vc_decoder_verify(dec, x, drafts, D, B, ctxP, P, k2, v2, n_acc, nxt, ws)
    torch.cuda.synchronize()
    assert _status_ok(vc, ws)
    want_n, want_next, _ = oracle.accept(logits.float().cpu().numpy(), drafts.cpu().numpy())
    assert n_acc.cpu().tolist() == list(want_n) and nxt.cpu().tolist() == list(want_next)
    assert n_acc.cpu().tolist() == keep
    assert torch.equal(k1, k2) and torch.equal(v1, v2)


def _launch_order_probe(graph: bool) -> dict:
    """Four draft-and-verify rounds of the small bf16 decoder: every round's
    drafts, accepted lengths and next tokens."""
    vc = lib()
    from lossless_draft_verify_gb300 import decode
    cfg, dec = _small_decoder(vc, seed=1)
    B, P, D, rounds = 3, 700, 8, 4
    g = torch.Generator().manual_seed(6)
    prompt = torch.randint(0, cfg.vocab, (B, P), generator=g, dtype=torch.int32).cuda()
    run = decode.VeriCacheRunner(dec, B, P + rounds * (D + 1) + 2 * D, D, bits=2, residual=128,
                                 prefill_chunk=256, use_graph=graph)
    run.prefill(prompt)
    log = run.new_log(rounds)
    for r in range(rounds):
        run.round(log, r)
    assert _status_ok(vc, run.ws)
    return {"drafts": log.drafts.cpu().tolist(), "n_acc": log.n_acc.cpu().tolist(), "nxt": log.nxt.cpu().tolist()}


@pytest.mark.parametrize("graph", [False, True])
def test_programmatic_launch_changes_no_result(graph):
    """Programmatic dependent launch (the default) lets each kernel start
    while the previous one drains; it must not change any result.  The same
    rounds run in a child process with VC_PDL=0 (every launch fully
    serialized) give bit for bit the same drafts (the lossy draft steps),
    accepted lengths and next tokens."""
    import json
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import json, sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "from test_gpu_decoder import _launch_order_probe; "
            "print(json.dumps(_launch_order_probe(%r)))") % (here, os.path.dirname(here), graph)
    env = dict(os.environ, VC_PDL="0")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    serialized = json.loads(out.stdout.strip().splitlines()[-1])
    assert os.environ.get("VC_PDL", "1") != "0"
    assert _launch_order_probe(graph) == serialized


def test_config5_model_spot_check_against_oracle():
    """The 8-layer bf16 decoder of the end-to-end workload (d_model 4096,
    32/8 heads, SwiGLU 14336, vocab 32000) against the fp64 oracle on the same
    weights: a 32-token prompt, then 8 greedy tokens (full-KV decoding, the
    losslessness reference of the model workload).  The oracle runs row by
    row, so each (row, layer) streams about 1.7 GB of fp64 weights; 39 rows
    take about a minute and a half, where a 2048-token prompt would take over
    an hour.  The GPU computes in bf16 (weights exact, activations rounded
    between kernels), so the prompt's last-row logits must agree within 5% of
    their largest magnitude (rms error within 1%), and the tokens must agree
    while the oracle's top-2 margin exceeds six times the rms logit error (a
    margin is the difference of two logits, each off by about the rms error);
    at the first position where it does not, the two sequences may part and
    the comparison stops there."""
    from lossless_draft_verify_gb300 import decode
    from oracle import model as om
    vc = lib()
    cfg = inputs.DecoderConfig()
    P, n_new = 32, 8
    W = inputs.decoder_weights_packed(cfg, seed=0, device="cuda")
    dec = vc.Decoder.from_packed(cfg, W["embed"], W["lm_head"], W["wqkv"], W["wo"], W["wgu"], W["wd"])
    prompt = inputs.random_prompts(1, P, cfg.vocab, seed=5, device="cuda")
    run = decode.VeriCacheRunner(dec, 1, P + n_new + 64, 8, bits=2, residual=0, prefill_chunk=64)
    run.prefill(prompt)
    torch.cuda.synchronize()
    gpu_logits = run.last_logits.float().cpu().numpy()[0]
    gpu_tokens = run.greedy(n_new)[0]
    torch.cuda.synchronize()
    # the oracle's weights: the same bf16 values, widened exactly to fp64
    qd, kvd, F, D = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.d_ff, cfg.d_model
    layers = []
    for l in range(cfg.n_layers):
        wqkv = W["wqkv"][l].double().cpu()
        gu = W["wgu"][l].double().cpu().reshape(D, F // 64, 2, 64)      # gate and up interleaved per 64
        layers.append({"wq": wqkv[:, :qd].numpy(), "wk": wqkv[:, qd:qd + kvd].numpy(),
                       "wv": wqkv[:, qd + kvd:].numpy(), "wo": W["wo"][l].double().cpu().numpy(),
                       "wg": gu[:, :, 0].reshape(D, F).numpy(), "wu": gu[:, :, 1].reshape(D, F).numpy(),
                       "wd": W["wd"][l].double().cpu().numpy()})
    weights = {"embed": W["embed"].double().cpu().numpy(), "lm_head": W["lm_head"].double().cpu().numpy(),
               "layers": layers}
    del W, dec, run
    torch.cuda.empty_cache()
    model = om.TinyDecoder(weights, cfg)
    cache = om.FullKV(model)
    lg, _ = om.forward_block(model, cache, [int(t) for t in prompt[0].tolist()], 0)
    want_logits = lg[-1]
    err = np.abs(gpu_logits - want_logits).max()
    rms = float(np.sqrt(np.mean((gpu_logits - want_logits) ** 2)))
    top = np.abs(want_logits).max()
    assert err <= 5e-2 * top and rms <= 1e-2 * top, (err, rms, top)
    want_tokens = [om.argmax_lowest(want_logits)]
    margins = [om._margin(want_logits)]
    while len(want_tokens) < n_new:
        lg, _ = om.forward_block(model, cache, [want_tokens[-1]], cache.length())
        want_tokens.append(om.argmax_lowest(lg[-1]))
        margins.append(om._margin(lg[-1]))
    compared = 0
    for t in range(n_new):
        if margins[t] <= 6 * rms:
            break                                   # a near tie at bf16 precision: the sequences may part
        assert gpu_tokens[t] == want_tokens[t], (t, gpu_tokens[t], want_tokens[t], margins[t], rms)
        compared += 1
        if gpu_tokens[t] != want_tokens[t]:
            break
    print(f"config-5 spot check: logit error max {err:.3e} rms {rms:.3e} of max {top:.2f}; "
          f"tokens compared {compared} of {n_new}; oracle margins {[round(m, 3) for m in margins]}")
    assert compared >= 1
