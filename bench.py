"""Benchmark of the draft-and-verify hot path on GB300.

Default (--workload model): one step = one VeriCache round of an 8-layer GQA
decoder (d_model 4096, 32/8 heads, head dim 128, SwiGLU 14336, vocab 32000,
bf16 random-init weights) for 8 sequences with 32768-token prompts:
  side stream: swap the full KV cache of every layer in from pinned host memory
               (held as lossless packed rows, expanded on the GPU);
  main stream: 32 draft steps of the model on its 2-bit KIVI caches (one CUDA
               graph), then the verify forward of the 33-token block over the
               full cache, greedy acceptance, the commit of the accepted rows to
               the draft caches and their write-back to the host copy.
Metric: lossless tokens/s = emitted tokens (accepted drafts + one per
sequence) per round / round time.  The same line carries the full-KV baseline
(plain greedy decoding with the cache swapped in before every token), the
losslessness check against it with its near-tie count, the swap's measured
overlap with drafting, the draft-attention roofline inside the decoder, and the
per-kernel numbers of the one-layer kernel workloads at B16 (draft attention
over the 2-bit cache, verify attention, acceptance over [16, 33, 151936]).

--workload round: one layer's hot path at 32k for 16 sequences (swap, 32 draft
attention steps, verify attention, acceptance over planted logits, commit).
--kernel NAME: one kernel alone at its own workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun): independent replicas, one per GPU, weak scaling.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# workload: the draft-attention and verify configurations at 32k context
B, HQ, HKV, D_HEAD, CTX = 16, 32, 8, 128, 32768
HORIZON = 32                      # drafted tokens per round
DQ = HORIZON + 1                  # verify block: pending token + drafts
VOCAB = 151936
BITS, GROUP, RESIDUAL = 2, 32, 128
METRIC = "lossless tokens/s at 32k ctx; draft-attn HBM GB/s and verify-attn TC % of peak"
WORKLOAD = ("verify_round_32k: B16 x 32/8 heads x d128, 32768-token context, KIVI 2-bit g32 R128 "
            "draft cache, horizon 32 (verify block 33), bf16 full KV swapped in from pinned host, "
            "accept over [16,33,151936] bf16 logits")
WORKLOAD_PACKED = WORKLOAD.replace("bf16 full KV swapped in from pinned host",
                                   "bf16 full KV swapped in from pinned host (held losslessly packed, "
                                   "expanded on the GPU)")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# DRAM bytes (read + write) of one draft launch at the 32768-token context,
# from one ncu capture of the draft kernel, keyed by the code digest (SHA-256
# without comments or blank lines) of the sources it was built from: a changed
# kernel reports traffic null until it is captured again.
DRAFT_TRAFFIC = {
    "sources": ("lossless_draft_verify_gb300/csrc/draft_attn.cu", "lossless_draft_verify_gb300/csrc/vc_common.cuh"),
    "sha256": ("8c0c9ce64474c47871902141eb7d70c8a550ff7a5f5d442e2e8e938e2597b714",
               "0ef2dd4e95c52fb9f0c6061fe73f4251def32e1390a8a92b67daed799a6b2f12"),
    "bytes": 409.689088e6 + 3.538176e6,
    "algorithmic_bytes": 409731072,
}


def code_digest(path: str) -> str:
    """SHA-256 of a C++/CUDA source with its comments and blank lines removed,
    so that an edit to comments alone does not count as a changed kernel."""
    import hashlib
    import re
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    lines = [ln.rstrip() for ln in src.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def captured_traffic(table: dict, per_launch_bytes: float):
    """Captured DRAM traffic scaled to a launch of `per_launch_bytes`
    algorithmic bytes, or None when the kernel's code changed."""
    for rel, want in zip(table["sources"], table["sha256"]):
        if code_digest(os.path.join(ROOT, rel)) != want:
            return None
    return table["bytes"] * per_launch_bytes / table["algorithmic_bytes"]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j.get("hbm_gbs"), j.get("bf16_tflops"), j.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (clocks and throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
# the round
# --------------------------------------------------------------------------

class Round:
    """One step of the hot path for all B sequences.  With stagger = 2 the
    full-cache swap-in and the verify pass run per half batch (cross-resource
    staggering, paper page "What the paper found"): half A's verify starts as
    soon as half A has arrived, while half B is still on the link, and the
    next step's swap of a half only waits for this step's verify of that half,
    so the host link never idles between steps.  Drafting, acceptance and the
    commit stay whole-batch launches."""

    def __init__(self, dev, stagger: int = 2, horizon: int = HORIZON, link_gbps: float | None = None,
                 bits: int = BITS, residual: int = RESIDUAL, packed: bool = False):
        from lossless_draft_verify_gb300 import inputs, vc
        self.vc, self.dev = vc, dev
        self.bits, self.residual = bits, residual
        HORIZON = self.D = horizon
        DQ = self.DQ = horizon + 1
        g = torch.Generator(device=dev)
        self.scale = inputs.default_scale(D_HEAD)
        Ls = CTX + DQ
        # full cache (context + the verify block's own K/V), resident copy on
        # the host in pinned memory, swapped in every round
        self.kfull, self.vfull = inputs.kv_with_outliers(B, HKV, Ls, D_HEAD, seed=1, device=dev)
        self.kfull_host = torch.empty(self.kfull.shape, dtype=torch.bfloat16).pin_memory()
        self.vfull_host = torch.empty(self.vfull.shape, dtype=torch.bfloat16).pin_memory()
        self.kfull_host.copy_(self.kfull)
        self.vfull_host.copy_(self.vfull)
        # packed host copy (lossless, 16 + 3d/2 bytes a row): the link moves
        # it into a device staging buffer and vc_kv_unpack restores the bf16
        self.packed = packed
        if packed:
            assert not link_gbps, "paced swaps move the bf16 cache"
            rb = vc.vc_kv_packed_row_bytes(D_HEAD)
            self.kpack = torch.empty(B, HKV, Ls, rb, dtype=torch.uint8, device=dev)
            self.vpack = torch.empty_like(self.kpack)
            n_over = torch.zeros(1, dtype=torch.int32, device=dev)
            vc.vc_kv_pack(self.kfull, self.kpack, n_over)
            vc.vc_kv_pack(self.vfull, self.vpack, n_over)
            if int(n_over.item()):
                # some row needs more than 7 escapes: this cache travels as bf16
                packed = self.packed = False
                del self.kpack, self.vpack
        if packed:
            self.kpack_host = self.kpack.cpu().pin_memory()
            self.vpack_host = self.vpack.cpu().pin_memory()
            # expansion runs on a stream of its own, so the link's copies stay
            # back to back; a part's staging rows are rewritten only after its
            # verify, which follows its expansion
            self.unpack_stream = torch.cuda.Stream(device=dev)
            self.ev_copied = [torch.cuda.Event() for _ in range(stagger)]
            # the expansion runs after the draft steps (its HBM traffic would
            # slow them); the copies still overlap them
            self.ev_drafted = torch.cuda.Event()
        # compressed draft cache of the context
        maxg = (CTX + DQ) // GROUP + 1
        self.cache = vc.QCache(B, HKV, D_HEAD, bits, maxg, residual + GROUP + DQ + 32, residual)
        vc.vc_quantize_kv(self.kfull, self.vfull, self.cache, L=CTX)
        torch.cuda.synchronize()
        self.len0 = self.cache.seq_len.clone()
        self.ng0 = self.cache.n_groups.clone()
        self.round_len = self.len0.clone()
        self.view = self.cache.view()
        # per-draft-step inputs: queries and the new token's K/V
        self.q_draft = inputs.normal_bf16((HORIZON, B, HQ, D_HEAD), 5, device=dev)
        self.k_step = inputs.normal_bf16((HORIZON, B, HKV, 1, D_HEAD), 6, device=dev)
        self.v_step = inputs.normal_bf16((HORIZON, B, HKV, 1, D_HEAD), 7, device=dev)
        self.ones = torch.ones(B, dtype=torch.int32, device=dev)
        self.o_draft = torch.empty_like(self.q_draft)
        # verify block and acceptance inputs
        self.q_ver = inputs.normal_bf16((B, DQ, HQ, D_HEAD), 8, device=dev)
        self.o_ver = torch.empty_like(self.q_ver)
        self.ctx = torch.full((B,), CTX, dtype=torch.int32, device=dev)
        self.k_blk = self.kfull[:, :, CTX:CTX + DQ].contiguous()
        self.v_blk = self.vfull[:, :, CTX:CTX + DQ].contiguous()
        case = inputs.accept_case(B, HORIZON, VOCAB, seed=0, device=dev)
        self.logits, self.drafts, self.diverge = case.logits, case.drafts, case.diverge
        self.n_acc = torch.zeros(B, dtype=torch.int32, device=dev)
        self.next_tok = torch.zeros(B, dtype=torch.int32, device=dev)
        # workspaces
        self.ws_d = vc.Workspace(vc.vc_draft_attn_workspace_bytes(self.view, HQ), device=dev)
        assert B % stagger == 0
        self.stagger = stagger
        self.link_gbps = link_gbps
        self.pace_ws = torch.zeros(4, dtype=torch.int32, device=dev)
        bp = B // stagger
        self.parts = [(i * bp, (i + 1) * bp) for i in range(stagger)]
        self.ws_v = vc.Workspace(vc.vc_verify_attn_workspace_bytes(torch.bfloat16, bp, DQ, HQ, HKV, D_HEAD, CTX),
                                 device=dev)
        self.ws_a = vc.Workspace(vc.vc_accept_workspace_bytes(B, HORIZON, VOCAB), device=dev)
        self.side = torch.cuda.Stream(device=dev)
        main = torch.cuda.current_stream()
        self.ev_swap = [torch.cuda.Event() for _ in self.parts]
        self.ev_ver = [torch.cuda.Event() for _ in self.parts]
        self.ev_acc = torch.cuda.Event()
        self.ev_in = torch.cuda.Event()
        for e in self.ev_swap + self.ev_ver + [self.ev_acc, self.ev_in]:
            e.record(main)
        # per step: (append + draft) per draft step, verify + its combine per part, accept, commit
        self.launches_per_step = HORIZON * 2 + 2 * stagger + 1 + 1 + (2 * stagger if packed else 0)
        # host-side copies of the per-step inputs (end-to-end measurement)
        self.h_q_draft = self.q_draft.cpu().pin_memory()
        self.h_k_step = self.k_step.cpu().pin_memory()
        self.h_v_step = self.v_step.cpu().pin_memory()
        self.h_q_ver = self.q_ver.cpu().pin_memory()
        self.h_logits = self.logits.cpu().pin_memory()
        self.h_drafts = self.drafts.cpu().pin_memory()
        self.h_nacc = torch.empty(B, dtype=torch.int32).pin_memory()
        self.h_next = torch.empty(B, dtype=torch.int32).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in
                             (self.h_q_draft, self.h_k_step, self.h_v_step, self.h_q_ver, self.h_logits,
                              self.h_drafts))
        self.d2h_bytes = 2 * B * 4
        self.swap_bytes = 2 * (self.kpack.numel() if packed else self.kfull.numel() * 2)

    def step(self, ev=None, e2e=False):
        vc, main = self.vc, torch.cuda.current_stream()
        if e2e:
            # this round's inputs arrive from pinned host memory, on the link's
            # stream ahead of the swap (once the previous step has read them)
            self.side.wait_event(self.ev_acc)
            for dst, src in ((self.q_draft, self.h_q_draft), (self.k_step, self.h_k_step),
                             (self.v_step, self.h_v_step), (self.q_ver, self.h_q_ver),
                             (self.logits, self.h_logits), (self.drafts, self.h_drafts)):
                vc.vc_swap_in(dst, src, stream=self.side)      # pinned host -> device through the C ABI
            self.ev_in.record(self.side)
            main.wait_event(self.ev_in)
        # swap-in of the full cache on the side stream, overlapped with drafting;
        # part p may be overwritten once the previous step's verify of p is done
        for p, (b0, b1) in enumerate(self.parts):
            self.side.wait_event(self.ev_ver[p])
            if ev is not None and p == 0:
                ev["swap0"].record(self.side)
            if self.link_gbps:
                vc.vc_swap_in_paced(self.kfull[b0:b1], self.kfull_host[b0:b1], self.link_gbps, self.pace_ws,
                                    stream=self.side)
                vc.vc_swap_in_paced(self.vfull[b0:b1], self.vfull_host[b0:b1], self.link_gbps, self.pace_ws,
                                    stream=self.side, done_event=self.ev_swap[p])
            elif self.packed:
                vc.vc_swap_in(self.kpack[b0:b1], self.kpack_host[b0:b1], stream=self.side)
                vc.vc_swap_in(self.vpack[b0:b1], self.vpack_host[b0:b1], stream=self.side,
                              done_event=self.ev_copied[p])
            else:
                vc.vc_swap_in(self.kfull[b0:b1], self.kfull_host[b0:b1], stream=self.side)
                vc.vc_swap_in(self.vfull[b0:b1], self.vfull_host[b0:b1], stream=self.side, done_event=self.ev_swap[p])
        if ev is not None and (not self.packed or self.link_gbps):
            ev["swap1"].record(self.side)
        for j in range(self.D):
            vc.vc_qcache_append(self.cache, self.k_step[j], self.v_step[j], self.ones, requantize=False)
            if ev is not None:
                ev["d0"][j].record(main)
            vc.vc_draft_attn(self.q_draft[j], self.view, self.scale, self.o_draft[j], self.ws_d)
            if ev is not None:
                ev["d1"][j].record(main)
        if self.packed and not self.link_gbps:
            # expansion of each part once it has landed and the draft steps have run
            self.ev_drafted.record(main)
            self.unpack_stream.wait_event(self.ev_drafted)
            for p, (b0, b1) in enumerate(self.parts):
                self.unpack_stream.wait_event(self.ev_copied[p])
                vc.vc_kv_unpack(self.kpack[b0:b1], self.kfull[b0:b1], stream=self.unpack_stream)
                vc.vc_kv_unpack(self.vpack[b0:b1], self.vfull[b0:b1], stream=self.unpack_stream)
                self.ev_swap[p].record(self.unpack_stream)
            if ev is not None:
                ev["swap1"].record(self.unpack_stream)
        for p, (b0, b1) in enumerate(self.parts):
            main.wait_event(self.ev_swap[p])
            if ev is not None:
                ev["v0"][p].record(main)
            vc.vc_verify_attn(self.q_ver[b0:b1], self.kfull[b0:b1], self.vfull[b0:b1], self.ctx[b0:b1], CTX,
                              self.scale, self.o_ver[b0:b1], self.ws_v)
            if ev is not None:
                ev["v1"][p].record(main)
            self.ev_ver[p].record(main)
        vc.vc_accept(self.logits, self.drafts, self.n_acc, self.next_tok, self.ws_a)
        self.ev_acc.record(main)
        if ev is not None:
            ev["a1"].record(main)
        vc.vc_qcache_commit(self.cache, self.k_blk, self.v_blk, self.round_len, self.n_acc)
        if e2e:
            self.h_nacc.copy_(self.n_acc, non_blocking=True)
            self.h_next.copy_(self.next_tok, non_blocking=True)
        # bench plumbing: return the synthetic cache to the round-start state
        self.cache.seq_len.copy_(self.len0, non_blocking=True)
        self.cache.n_groups.copy_(self.ng0, non_blocking=True)

    def tokens_per_round(self) -> int:
        return int((self.n_acc.long() + 1).sum().item())

    # algorithmic bytes / flops of one launch
    def draft_bytes(self, j: int) -> int:
        rec = self.vc.vc_record_bytes(self.bits, D_HEAD)
        ng = (CTX - self.residual) // GROUP
        n_res = CTX + j + 1 - ng * GROUP
        per_unit = ng * rec + 2 * n_res * D_HEAD * 2
        return B * HKV * per_unit + 2 * B * HQ * D_HEAD * 2

    def verify_bytes(self) -> int:
        return 2 * B * HKV * (CTX + self.DQ) * D_HEAD * 2 + 2 * B * self.DQ * HQ * D_HEAD * 2

    def verify_flops(self) -> int:
        rows_keys = sum(CTX + i + 1 for i in range(self.DQ))
        return 4 * D_HEAD * B * HQ * rows_keys


def make_events(n_draft, n_parts=1):
    mk = lambda: torch.cuda.Event(enable_timing=True)
    return {"swap0": mk(), "swap1": mk(), "v0": [mk() for _ in range(n_parts)], "v1": [mk() for _ in range(n_parts)],
            "a1": mk(), "d0": [mk() for _ in range(n_draft)], "d1": [mk() for _ in range(n_draft)]}


# --------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same round
# --------------------------------------------------------------------------

def oracle_inputs(rnd, n_seq: int) -> dict:
    """Host fp32 images of the first n_seq sequences of the round's inputs
    (from the device tensors when a round exists, else regenerated by the same
    seeded generators)."""
    import oracle
    from lossless_draft_verify_gb300 import inputs
    oracle.build()
    if rnd is not None:
        f = lambda t: t.float().cpu().numpy()
        kf, vf = f(rnd.kfull[:n_seq]), f(rnd.vfull[:n_seq])
        qd, ks, vs = f(rnd.q_draft[:, :n_seq]), f(rnd.k_step[:, :n_seq]), f(rnd.v_step[:, :n_seq])
        qv, lg, dr = f(rnd.q_ver[:n_seq]), f(rnd.logits[:n_seq]), rnd.drafts[:n_seq].cpu().numpy()
    else:
        k, v = inputs.kv_with_outliers(n_seq, HKV, CTX + DQ, D_HEAD, seed=1)
        kf, vf = k.float().numpy(), v.float().numpy()
        qd = inputs.normal_bf16((HORIZON, n_seq, HQ, D_HEAD), 5).float().numpy()
        ks = inputs.normal_bf16((HORIZON, n_seq, HKV, 1, D_HEAD), 6).float().numpy()
        vs = inputs.normal_bf16((HORIZON, n_seq, HKV, 1, D_HEAD), 7).float().numpy()
        qv = inputs.normal_bf16((n_seq, DQ, HQ, D_HEAD), 8).float().numpy()
        case = inputs.accept_case(n_seq, HORIZON, VOCAB, seed=0)
        lg, dr = case.logits.float().numpy(), case.drafts.numpy()
    qc = oracle.kivi_quantize(kf[:, :, :CTX], vf[:, :, :CTX], BITS, GROUP, RESIDUAL)
    return dict(n_seq=n_seq, kf=kf, vf=vf, qd=qd, ks=ks, vs=vs, qv=qv, lg=lg, dr=dr, qc=qc)


def oracle_round(x: dict):
    """The oracle's draft attention (every draft step, on the growing cache),
    verify attention and acceptance for the sampled sequences.  Returns
    (seconds, sampled kv units, threads)."""
    import oracle
    qc = dict(x["qc"])
    t0 = time.perf_counter()
    for j in range(HORIZON):
        qc["kres"] = np.concatenate([qc["kres"], x["ks"][j]], axis=2)
        qc["vres"] = np.concatenate([qc["vres"], x["vs"][j]], axis=2)
        oracle.kivi_decode_attn(x["qd"][j], qc, 1.0 / math.sqrt(D_HEAD))
    oracle.verify_attn(x["qv"], x["kf"], x["vf"], [CTX] * x["n_seq"], 1.0 / math.sqrt(D_HEAD))
    oracle.accept(x["lg"], x["dr"])
    dt = time.perf_counter() - t0
    units = x["n_seq"] * HKV
    return dt, units, min(oracle.num_threads(), units)


def sample_seqs() -> int:
    return max(1, min(B, (os.cpu_count() or 8) // HKV))


def cpu_baseline_record(rnd, tokens_per_round):
    x = oracle_inputs(rnd, sample_seqs())
    dt, units, threads = oracle_round(x)
    # the round's work is uniform over the 128 kv units: scale the sampled time
    t_round = dt * (B * HKV) / units
    return {"value": tokens_per_round / t_round, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{x['n_seq']} of {B} sequences ({units} of {B * HKV} kv units) of one round: {HORIZON} draft "
                      f"attentions, the verify attention and acceptance, fp64; time scaled by {B * HKV}/{units}",
            "sample_seconds": round(dt, 3)}


# --------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload == "model":
        run_reference_model(args, world)
        return
    from lossless_draft_verify_gb300 import inputs
    n_seq = sample_seqs()
    case = inputs.accept_case(B, HORIZON, VOCAB, seed=0)
    tokens = int((case.diverge.long() + 1).sum())
    x = oracle_inputs(None, n_seq)
    times = []
    for i in range(args.warmup + args.steps):
        dt, units, threads = oracle_round(x)
        if i >= args.warmup:
            times.append(dt * (B * HKV) / units)
    t = sum(times) / len(times)
    val = tokens / t
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_PACKED, "parallelism": "cpu oracle (OpenMP over kv units)",
                       "global_batch": B, "seq_len": CTX},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n_seq} of {B} sequences per step, time scaled by {B * HKV}/{units}"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_model(args, world):
    """The oracle on the decoder workload: every step times the bounded sample
    of model_oracle_sample (one draft row and one verify row through one
    layer, one head row) and scales it to a round.  Tokens per round: B, one
    per sequence, the accepted-draft count this random-init model shows at 2
    bits on the GPU (0 per round); the timing does not depend on it."""
    from lossless_draft_verify_gb300 import inputs
    cfg = inputs.DecoderConfig()
    P = args.prompt
    sample = ModelOracleSample(cfg, P, args.bits)
    times = []
    for i in range(args.warmup + args.steps):
        s = sample.time_once()
        if i >= args.warmup:
            times.append(model_round_seconds(cfg, s))
    t = statistics.mean(times)
    val = M_B / t
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (random-init weights)",
            "config": {"workload": MODEL_WORKLOAD.format(ctx=P, bits=args.bits), "global_batch": M_B,
                       "seq_len": P, "parallelism": "cpu oracle, one core"},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": "per step: one draft row and one verify row through one decoder layer at "
                                       f"{P} tokens of context and one LM-head row (oracle/model.py, fp64), scaled "
                                       f"to a round of {M_B}x{M_HORIZON} draft and {M_B}x{M_HORIZON + 1} verify rows "
                                       f"through {cfg.n_layers} layers; {M_B} tokens per round"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# single-kernel mode: one hot-path kernel at its own workload, for rooflines
# and profiler captures (python bench.py --kernel draft|verify|accept|quantize|drop|dense_draft)
# --------------------------------------------------------------------------

def run_kernel(args, dev):
    from lossless_draft_verify_gb300 import inputs, vc
    hbm, tf_burst, _, peak_src = measured_peaks()
    name = args.kernel
    B = args.batch
    rec = {}
    flops = None
    if name in ("draft", "quantize"):
        ctx = args.ctx
        if ctx < RESIDUAL + GROUP or ctx % GROUP:
            raise SystemExit(f"--ctx must be a multiple of {GROUP} of at least {RESIDUAL + GROUP}")
        k, v = inputs.kv_with_outliers(B, HKV, ctx, D_HEAD, seed=1, device=dev)
        cache = vc.QCache(B, HKV, D_HEAD, BITS, (ctx - RESIDUAL) // GROUP, RESIDUAL + GROUP + 8, RESIDUAL)
        vc.vc_quantize_kv(k, v, cache)
        rb = vc.vc_record_bytes(BITS, D_HEAD)
        ng = (ctx - RESIDUAL) // GROUP
        if name == "quantize":
            fn = lambda: vc.vc_quantize_kv(k, v, cache)
            nbytes = 2 * k.numel() * 2 + B * HKV * ng * rb
            rec = {"workload": f"KIVI 2-bit g32 prefill of bf16 K/V [{B},8,{ctx},128], R=128"}
        else:
            del k, v
            q = inputs.normal_bf16((B, HQ, D_HEAD), 5, device=dev)
            out = torch.empty_like(q)
            view = cache.view()
            ws = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, HQ), device=dev)
            scale = inputs.default_scale(D_HEAD)
            fn = lambda: vc.vc_draft_attn(q, view, scale, out, ws)
            nbytes = B * HKV * (ng * rb + 2 * RESIDUAL * D_HEAD * 2) + 2 * q.numel() * 2
            rec = {"workload": f"draft attention, KIVI 2-bit cache [{B},8,{ctx},128] R=128, q [{B},32,128] bf16"}
    elif name == "verify":
        dq = args.dq
        q = inputs.normal_bf16((B, dq, HQ, D_HEAD), 8, device=dev)
        k = inputs.normal_bf16((B, HKV, CTX + dq, D_HEAD), 9, device=dev)
        v = inputs.normal_bf16((B, HKV, CTX + dq, D_HEAD), 10, device=dev)
        ctx = torch.full((B,), CTX, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = vc.Workspace(vc.vc_verify_attn_workspace_bytes(torch.bfloat16, B, dq, HQ, HKV, D_HEAD, CTX), device=dev)
        scale = inputs.default_scale(D_HEAD)
        fn = lambda: vc.vc_verify_attn(q, k, v, ctx, CTX, scale, out, ws)
        nbytes = 2 * k.numel() * 2 + 2 * q.numel() * 2
        flops = 4 * D_HEAD * B * HQ * sum(CTX + i + 1 for i in range(dq))
        rec = {"workload": f"verify attention, Dq={dq}, bf16 K/V [{B},8,{CTX + dq},128], 32/8 heads"}
    elif name == "verify_h2o":
        # verify attention plus the H2O mass pass (a second pass over K)
        dq = args.dq
        q = inputs.normal_bf16((B, dq, HQ, D_HEAD), 8, device=dev)
        k = inputs.normal_bf16((B, HKV, CTX + dq, D_HEAD), 9, device=dev)
        v = inputs.normal_bf16((B, HKV, CTX + dq, D_HEAD), 10, device=dev)
        ctx = torch.full((B,), CTX, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        scores = torch.zeros(B, HKV, CTX + dq, dtype=torch.float32, device=dev)
        ws = vc.Workspace(vc.vc_verify_attn_h2o_workspace_bytes(B, dq, HQ, HKV, D_HEAD, CTX), device=dev)
        scale = inputs.default_scale(D_HEAD)
        fn = lambda: vc.vc_verify_attn_h2o(q, k, v, ctx, CTX, scale, out, scores, ws)
        # verify's K and V, the mass pass's K again, the scores read and written
        nbytes = 3 * k.numel() * 2 + 2 * q.numel() * 2 + 2 * scores.numel() * 4
        flops = 2 * 4 * D_HEAD * B * HQ * sum(CTX + i + 1 for i in range(dq))
        rec = {"workload": f"verify attention with H2O accumulation, Dq={dq}, bf16 K/V [{B},8,{CTX + dq},128], "
                           "32/8 heads"}
    elif name == "accept":
        case = inputs.accept_case(B, HORIZON, VOCAB, seed=0, device=dev)
        n = torch.empty(B, dtype=torch.int32, device=dev)
        nx = torch.empty(B, dtype=torch.int32, device=dev)
        ws = vc.Workspace(vc.vc_accept_workspace_bytes(B, HORIZON, VOCAB), device=dev)
        fn = lambda: vc.vc_accept(case.logits, case.drafts, n, nx, ws)
        nbytes = case.logits.numel() * 2
        rec = {"workload": "greedy acceptance, logits [16,33,151936] bf16"}
    elif name in ("drop", "dense_draft", "dense_draft_h2o"):
        Bd, Hd, Ld = 4, 8, 131072
        scores = inputs.zipf_scores(Bd, Hd, Ld, seed=0, device=dev)
        k, v = inputs.kv_with_outliers(Bd, Hd, Ld, D_HEAD, seed=8, device=dev, n_out=0)
        n_keep = vc.vc_drop_kept_count(Ld, Ld // 4, 256)
        kept = torch.empty(Bd, Hd, n_keep, dtype=torch.int32, device=dev)
        ko = torch.empty(Bd, Hd, n_keep, D_HEAD, dtype=torch.bfloat16, device=dev)
        vo = torch.empty_like(ko)
        ws = vc.Workspace(vc.vc_drop_tokens_workspace_bytes(Bd, Hd, Ld), device=dev)
        drop = lambda: vc.vc_drop_tokens(scores, k, v, Ld // 4, 256, kept, ko, vo, ws)
        if name == "drop":
            fn = drop
            nbytes = scores.numel() * 4 + 2 * 2 * ko.numel() * 2 + kept.numel() * 4
            rec = {"workload": "token dropping 4x: scores [4,8,131072] Zipf(1.1), keep 32768 + 256, gather K/V"}
        else:
            drop()
            q = inputs.normal_bf16((Bd, 4 * Hd, D_HEAD), 5, device=dev)
            out = torch.empty_like(q)
            lens = torch.full((Bd,), n_keep, dtype=torch.int32, device=dev)
            view = vc.dense_view(ko, vo, lens, n_keep)
            ws2 = vc.Workspace(vc.vc_draft_attn_workspace_bytes(view, 4 * Hd), device=dev)
            scale = inputs.default_scale(D_HEAD)
            if name == "dense_draft":
                fn = lambda: vc.vc_draft_attn(q, view, scale, out, ws2)
                nbytes = 2 * ko.numel() * 2 + 2 * q.numel() * 2
                rec = {"workload": "decode attention over the compacted cache [4,8,33024,128] bf16, 32/8 heads"}
            else:
                acc = torch.zeros(Bd, Hd, Ld, dtype=torch.float32, device=dev)
                ws3 = vc.Workspace(vc.vc_draft_attn_h2o_workspace_bytes(view, 4 * Hd), device=dev)
                fn = lambda: vc.vc_draft_attn_h2o(q, view, scale, out, acc, ws3, kept_idx=kept)
                # attention bytes + per kept row: scores written and read (16 B each), the
                # index read (4 B) and the accumulated score read and written (8 B)
                nbytes = 2 * ko.numel() * 2 + 2 * q.numel() * 2 + kept.numel() * (16 + 16 + 4 + 8)
                rec = {"workload": "decode attention over the compacted cache [4,8,33024,128] bf16, 32/8 heads, "
                                   "with H2O score accumulation at the kept positions"}
    elif name == "gemm":
        # the decoder's gate|up projection in a draft step: M = 8 rows, K 4096, N 2 x 14336
        M, K, N = 8, 4096, 2 * 14336
        x = inputs.normal_bf16((M, K), 30, device=dev)
        w = inputs.normal_bf16((K, N), 31, device=dev, std=0.02)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        ws = vc.Workspace(vc.vc_gemm_workspace_bytes(torch.bfloat16, M, N, K), device=dev)
        fn = lambda: vc.vc_gemm(x, w, y, ws=ws, decode_plan=True)
        nbytes = K * N * 2 + M * K * 2 + M * N * 2
        flops = 2 * M * N * K
        rec = {"workload": "draft-step GEMM x[8,4096] W[4096,28672] bf16 (decode plan)"}
    elif name == "unpack":
        # expansion of the round's packed full K cache [16, 8, 32801, 128]
        k, _ = inputs.kv_with_outliers(B, HKV, CTX + DQ, D_HEAD, seed=1, device=dev)
        rbytes = vc.vc_kv_packed_row_bytes(D_HEAD)
        pk = torch.empty(*k.shape[:-1], rbytes, dtype=torch.uint8, device=dev)
        n_over = torch.zeros(1, dtype=torch.int32, device=dev)
        vc.vc_kv_pack(k, pk, n_over)
        assert int(n_over.item()) == 0
        out = torch.empty_like(k)
        fn = lambda: vc.vc_kv_unpack(pk, out)
        nbytes = pk.numel() + out.numel() * 2
        rec = {"workload": f"expansion of the packed full K cache [{B},8,{CTX + DQ},128] ({rbytes} of 256 bytes a row)"}
    elif name == "swap":
        # full-cache swap-in (host link): one copy, or the cache split in
        # chunks issued on as many side streams
        k = torch.empty(B, HKV, CTX + DQ, D_HEAD, dtype=torch.bfloat16, device=dev)
        v = torch.empty_like(k)
        kh = torch.empty(k.shape, dtype=torch.bfloat16).pin_memory()
        vh = torch.empty(k.shape, dtype=torch.bfloat16).pin_memory()
        nch = max(1, args.chunks)
        streams = [torch.cuda.Stream(device=dev) for _ in range(nch)]
        main = torch.cuda.current_stream()
        kc, vc_ = k.view(-1).chunk(nch), v.view(-1).chunk(nch)
        khc, vhc = kh.view(-1).chunk(nch), vh.view(-1).chunk(nch)

        def fn():
            for i, st in enumerate(streams):
                st.wait_stream(main)
                vc.vc_swap_in(kc[i], khc[i], stream=st)
                vc.vc_swap_in(vc_[i], vhc[i], stream=st)
            for st in streams:
                main.wait_stream(st)
        nbytes = 2 * k.numel() * 2
        rec = {"workload": f"full-KV swap-in, 2 x [16,8,{CTX + DQ},128] bf16 from pinned host, {nch} chunk(s)"}
    else:
        raise SystemExit(f"unknown kernel {name}")
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    # a working set that fits in L2 is flushed before every timed launch (a
    # 256 MB write, outside the events); larger ones stream from HBM anyway
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if nbytes < (256 << 20) else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i, (a, b) in enumerate(evs):
        if flush is not None:
            flush.fill_(i & 255)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    rec["l2"] = "flushed before every launch (256 MB write)" if flush is not None else "inputs larger than L2 (no flush)"
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    gbs = nbytes / (ms / 1e3) / 1e9
    rec.update({"kernel": name, "ms": ms, "bytes": nbytes, "GB/s": gbs, "hbm_frac": gbs / hbm,
                "peak_source": peak_src})
    if flops:
        rec.update({"flops": flops, "TFLOP/s": flops / (ms / 1e3) / 1e12,
                    "tc_frac_burst": flops / (ms / 1e3) / 1e12 / tf_burst})
    print(json.dumps(rec), flush=True)


# --------------------------------------------------------------------------
# end-to-end model workload: the 8-layer GQA decoder (d_model 4096, 32/8
# heads, SwiGLU 14336, vocab 32000, bf16), B = 8 prompts at 32k context, the
# full cache held in pinned host memory and swapped in every round while the
# model drafts 32 tokens on its 2-bit caches
# --------------------------------------------------------------------------

M_B, M_HORIZON, M_BITS, M_RESIDUAL = 8, 32, 2, 128
MODEL_WORKLOAD = ("decoder_e2e_{ctx}: 8-layer GQA decoder d4096 32/8 heads hd128 SwiGLU 14336 vocab 32000 bf16 "
                  "(random init N(0,0.02), LM head x20), B8 random prompts of {ctx} tokens, KIVI {bits}-bit g32 R128 "
                  "draft caches, horizon 32, full KV in pinned host memory swapped in every round")


def model_bytes(cfg) -> dict:
    """Algorithmic bytes of the decoder's weights, per GEMM kind."""
    D, F, V = cfg.d_model, cfg.d_ff, cfg.vocab
    qd, kvd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    return {"gemm_qkv": D * (qd + 2 * kvd) * 2, "gemm_o": qd * D * 2, "gemm_gate_up": D * 2 * F * 2,
            "gemm_down": F * D * 2, "gemm_head": D * V * 2}


def decoder_draft_attn_bytes(vc, cfg, ctx: float, bits: int) -> int:
    """Algorithmic bytes of one draft-attention launch of the decoder (all B
    sequences of one layer) at `ctx` cached tokens: the packed records of the
    quantized prefix, the full-precision ring, q and the output."""
    rec_b = vc.vc_record_bytes(bits, cfg.head_dim)
    ng = int((ctx - M_RESIDUAL) // 32)
    n_res = ctx - ng * 32
    per_unit = ng * rec_b + 2 * n_res * cfg.head_dim * 2
    return int(M_B * cfg.n_kv_heads * per_unit + 2 * M_B * cfg.n_heads * cfg.head_dim * 2)


class ModelOracleSample:
    """The oracle (oracle/model.py, fp64, as it stands) on a bounded sample of
    one round of the decoder workload: one draft step of one sequence through
    one decoder layer on a 2-bit KIVI draft cache of `ctx` tokens, one verify
    row of one sequence through one layer over a full cache of `ctx` tokens,
    and one LM-head row.  The weights are one layer of the model's shapes
    drawn by the shared generator, the cached K/V synthetic N(0,1) of the
    workload's shapes (the oracle's cost does not depend on the values)."""

    def __init__(self, cfg, ctx: int, bits: int):
        import dataclasses
        from lossless_draft_verify_gb300 import inputs
        from oracle import model as om
        self.om, self.ctx = om, ctx
        c1 = dataclasses.replace(cfg, n_layers=1)
        W = inputs.decoder_weights_packed(c1, seed=0, device="cpu", dtype=torch.float32)
        qd, kvd, F = c1.n_heads * c1.head_dim, c1.n_kv_heads * c1.head_dim, c1.d_ff
        f = lambda t: t.double().numpy()
        wqkv, wgu = W["wqkv"][0], W["wgu"][0]
        gu = wgu.reshape(c1.d_model, F // 64, 2, 64)        # gate and up interleaved per 64 columns
        weights = {"embed": f(W["embed"]), "lm_head": f(W["lm_head"]),
                   "layers": [{"wq": f(wqkv[:, :qd]), "wk": f(wqkv[:, qd:qd + kvd]), "wv": f(wqkv[:, qd + kvd:]),
                               "wo": f(W["wo"][0]), "wg": f(gu[:, :, 0].reshape(c1.d_model, F)),
                               "wu": f(gu[:, :, 1].reshape(c1.d_model, F)), "wd": f(W["wd"][0])}]}
        del W
        self.m = om.TinyDecoder(weights, c1)
        self.g = np.random.default_rng(0)
        hd, nq = c1.head_dim, (ctx - M_RESIDUAL) // 32 * 32
        self.dc = om.KiviDraftCache(self.m, bits, 32, M_RESIDUAL)
        self.full = om.FullKV(self.m)
        g = self.g
        for h in range(c1.n_kv_heads):
            self.dc.qK[0][h], self.dc.qV[0][h] = g.standard_normal((nq, hd)), g.standard_normal((nq, hd))
            self.dc.rK[0][h] = g.standard_normal((ctx - nq, hd)).astype(np.float32)
            self.dc.rV[0][h] = g.standard_normal((ctx - nq, hd)).astype(np.float32)
            self.full.K[0][h], self.full.V[0][h] = g.standard_normal((ctx, hd)), g.standard_normal((ctx, hd))

    def time_once(self) -> dict:
        """Seconds per draft row-layer, verify row-layer and head row."""
        om, m, ctx = self.om, self.m, self.ctx
        t0 = time.perf_counter()
        om.draft_step(m, self.dc, 1, ctx)                 # one layer + the LM head
        t1 = time.perf_counter()
        om.forward_block(m, self.full, [1], ctx)          # one layer + the LM head
        t2 = time.perf_counter()
        m.logits(self.g.standard_normal(m.cfg.d_model))
        t3 = time.perf_counter()
        self.dc.truncate(ctx)
        self.full.truncate(ctx)
        head = t3 - t2
        return {"draft_row_layer_s": max(t1 - t0 - head, 0.0), "verify_row_layer_s": max(t2 - t1 - head, 0.0),
                "head_row_s": head, "sample_s": t3 - t0}


def model_round_seconds(cfg, s: dict) -> float:
    """Oracle seconds for one round (B sequences, D draft steps through every
    layer and the head, a (D + 1)-row verify pass through every layer and the
    head), from the per-row sample times."""
    nl, D = cfg.n_layers, M_HORIZON
    return (M_B * D * (nl * s["draft_row_layer_s"] + s["head_row_s"]) +
            M_B * (D + 1) * (nl * s["verify_row_layer_s"] + s["head_row_s"]))


def model_cpu_record(cfg, ctx: int, bits: int, tokens_per_round: float, tokens_note: str) -> dict:
    s = ModelOracleSample(cfg, ctx, bits).time_once()
    t_round = model_round_seconds(cfg, s)
    return {"value": tokens_per_round / t_round, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": (f"oracle/model.py in fp64 on one core: one draft row and one verify row through one decoder "
                       f"layer at {ctx} tokens of context and one LM-head row "
                       f"({s['draft_row_layer_s']:.2f} / {s['verify_row_layer_s']:.2f} / {s['head_row_s']:.2f} s), "
                       f"scaled to a round of {M_B}x{M_HORIZON} draft rows and {M_B}x{M_HORIZON + 1} verify rows "
                       f"through {cfg.n_layers} layers plus their head rows ({t_round:.0f} s); {tokens_note}"),
            "sample_seconds": round(s["sample_s"], 2), "round_seconds_estimate": t_round}


def run_model(args, dev, rank, world, barrier, pg):
    from lossless_draft_verify_gb300 import decode, inputs, replicas, vc
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    cfg = inputs.DecoderConfig()
    P = args.prompt
    W = inputs.decoder_weights_packed(cfg, seed=0, device=dev)
    dec = vc.Decoder.from_packed(cfg, W["embed"], W["lm_head"], W["wqkv"], W["wo"], W["wgu"], W["wd"])
    n_tr = 1                                  # traced round
    # K untimed rounds after the timed ones add tokens to the losslessness
    # check (the cache capacity, and so the bytes every swap moves, follow the
    # round count: it is kept at warm-up + traced + 2 K)
    n_extra = args.steps
    total = args.warmup + n_tr + args.steps + n_extra
    max_len = P + total * (M_HORIZON + 1) + 64
    packed = args.swap != "raw"                 # default packed
    run = decode.VeriCacheRunner(dec, M_B, max_len, M_HORIZON, bits=args.bits, residual=M_RESIDUAL, host_cache=True,
                                 prefill_chunk=512, device=dev, rotate=args.rotate, pack_host=packed)
    run.expand_after_draft = not args.expand_during_draft
    prompt = inputs.random_prompts(M_B, P, cfg.vocab, seed=rank, device=dev)
    t_pf = time.perf_counter()
    run.prefill(prompt)
    torch.cuda.synchronize()
    t_pf = time.perf_counter() - t_pf
    packed = run.pack_host                  # False if a prompt row could not be packed
    first = run.x.cpu().tolist()
    log = run.new_log(total)
    for r in range(args.warmup):
        run.round(log, r)
    # per-operation trace (every GEMM and attention call) of one round: the
    # draft steps are captured with tracing on, so their event pairs become
    # nodes of a graph and time the kernels as a graph replay runs them; the
    # verify forward is traced as issued (it is queued behind the draft graph
    # and the swap, so the host is well ahead of the device there)
    ops_per_round = M_HORIZON * (5 * cfg.n_layers + 1) + 5 * cfg.n_layers + 1 + 2 * cfg.n_layers
    trace = vc.DecoderTrace(dec, ops_per_round * n_tr)
    torch.cuda.synchronize()
    ctx_tr = float(run.qc[0].seq_len.float().mean())
    trace.start()
    g_tr = run.capture_draft_graph(keep=False)
    run.round(log, args.warmup, graph=g_tr)
    ops = trace.stop()
    del g_tr
    # the timed rounds replay the draft steps as one CUDA graph
    if not args.no_graph:
        run.capture_draft_graph()
    base0 = args.warmup + n_tr
    # The K timed rounds are timed by two clocks at once.  value: device events
    # around the rounds (tokens / device time).  e2e: the host's wall clock
    # around the same rounds, as a serving loop sees them: each round's emitted
    # tokens (drafts, accepted length, next token) are copied to pinned host
    # memory and read by the host; the next round needs nothing from the host,
    # so round i + 1 is issued before the host waits for round i's tokens.
    # Every round's input, the full cache, comes in from pinned host memory
    # inside the round.  Timing both on the same rounds keeps the host link's
    # drift between runs out of their comparison.
    want_e2e = not args.no_e2e
    n_out = M_B * (M_HORIZON + 2)
    h_out = [torch.empty(n_out, dtype=torch.int32).pin_memory() for _ in range(2)]
    d2h = n_out * 4
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]
    checksum = 0
    evs = [run.new_events() for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    swap_log0 = len(run.swap_rows)
    barrier()
    wall0 = time.perf_counter()
    t0.record()
    torch.cuda.nvtx.range_push("timed_rounds")
    for i in range(args.steps):
        run.round(log, base0 + i, evs[i])
        if want_e2e:
            ho = h_out[i & 1]
            ho[:M_B * M_HORIZON].copy_(run.drafts.view(-1), non_blocking=True)
            ho[M_B * M_HORIZON:M_B * (M_HORIZON + 1)].copy_(run.n_acc, non_blocking=True)
            ho[M_B * (M_HORIZON + 1):].copy_(run.x, non_blocking=True)
            ev_out[i & 1].record()
        if i == args.steps - 1:
            t1.record()
        if want_e2e and i > 0:
            ev_out[(i - 1) & 1].synchronize()              # round i - 1's tokens are on the host
            checksum += int(h_out[(i - 1) & 1].sum())
    if want_e2e:
        ev_out[(args.steps - 1) & 1].synchronize()
        checksum += int(h_out[(args.steps - 1) & 1].sum())
    wall1 = time.perf_counter()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    swap_rows = statistics.mean(run.swap_rows[swap_log0:swap_log0 + args.steps])
    n_acc = log.n_acc[base0:base0 + args.steps].cpu()
    tokens = int((n_acc.long() + 1).sum())
    value, ms_max = replicas.whole_job_rate(tokens, ms, pg, device=dev)
    st = vc.vc_poll_status(run.ws)
    e2e_val = None
    if want_e2e:
        e2e_val, _ = replicas.whole_job_rate(tokens, (wall1 - wall0) * 1e3, pg, device=dev)
    for i in range(n_extra):
        run.round(log, base0 + args.steps + i)
    run.check_packed()                   # every committed row was held by the packed host copy

    # per-phase times and the swap's overlap with drafting, measured as the
    # intersection of the two intervals on the device
    d_ms = statistics.mean(e["d0"].elapsed_time(e["d1"]) for e in evs)
    v_ms = statistics.mean(e["v0"].elapsed_time(e["v1"]) for e in evs)
    c_ms = statistics.mean(e["v1"].elapsed_time(e["c1"]) for e in evs)
    s_ms = statistics.mean(e["swap0"].elapsed_time(e["swap1"]) for e in evs)
    hidden = statistics.mean(
        max(0.0, min(e["swap0"].elapsed_time(e["swap1"]), e["swap0"].elapsed_time(e["d1"]))
            - max(0.0, e["swap0"].elapsed_time(e["d0"]))) / e["swap0"].elapsed_time(e["swap1"]) for e in evs)
    wb = model_bytes(cfg)
    by_kind = {}
    for k, t in ops:
        a = by_kind.setdefault(k, [0, 0.0])
        a[0] += 1
        a[1] += t
    da_bytes = decoder_draft_attn_bytes(vc, cfg, ctx_tr + M_HORIZON / 2, args.bits)
    kernels = {}
    for k, (n, t) in by_kind.items():
        ent = {"launches_per_round": n / n_tr, "ms_per_launch": t / n, "ms_per_round": t / n_tr}
        nb = wb.get(k, da_bytes if k == "draft_attn" else None)
        if nb is not None:
            ent["bytes_per_launch"] = nb
            ent["GB/s"] = nb / (t / n / 1e3) / 1e9
            ent["hbm_frac"] = ent["GB/s"] / hbm
        kernels[k] = ent
    gemm_kinds = [k for k in by_kind if k.startswith("gemm")]
    g_bytes = sum(wb[k] * by_kind[k][0] for k in gemm_kinds)
    g_ms = sum(by_kind[k][1] for k in gemm_kinds)
    da_n, da_t = by_kind.get("draft_attn", (1, float("nan")))
    da_gbs = da_bytes / (da_t / da_n / 1e3) / 1e9
    round_dev_ms = sum(t for _, t in ops) / n_tr
    roof = {"bound": "hbm", "achieved": da_gbs, "peak": hbm, "unit": "GB/s", "frac": da_gbs / hbm,
            "traffic": captured_traffic(DRAFT_TRAFFIC, da_bytes),
            "kernel": "vc_draft_attn inside the decoder's draft steps (draft_kivi_kernel + combine; B8, one layer "
                      "per launch), the hot path's dominant kernel; per-launch times from event pairs captured "
                      "into a replay of the round's draft-step graph",
            "bytes_per_launch": da_bytes, "ms_per_launch": da_t / da_n,
            "peak_source": f"{peak_src} hbm_gbs (copy, burst)"}
    roof_gemm = {"bound": "hbm", "achieved": g_bytes / (g_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                 "frac": g_bytes / (g_ms / 1e3) / 1e9 / hbm,
                 "kernel": "gemm_tc_kernel: the decoder's projections and LM head (weights streamed at M = 8 "
                           "in draft steps, M = 264 in the verify forward); the largest share of device time",
                 "share_of_traced_time": g_ms / n_tr / round_dev_ms}
    del run
    torch.cuda.empty_cache()

    # full-KV baseline and losslessness: the same prompts decoded by plain
    # greedy decoding with the full cache held on the host in the same format
    # and swapped in before every token (one-token forwards); its tokens are
    # the reference the draft-and-verify output must equal, its margins flag
    # near ties, and its token steps time the baseline
    emitted = [[first[b]] + t for b, t in enumerate(log.tokens())]
    n_cmp = max(4, min(min(len(t) for t in emitted), args.check_tokens))
    ref = decode.VeriCacheRunner(dec, M_B, P + n_cmp + 64, M_HORIZON, bits=args.bits, residual=M_RESIDUAL,
                                 host_cache=True, prefill_chunk=512, device=dev, pack_host=packed)
    ref.prefill(prompt)
    margins = torch.zeros(n_cmp, M_B, dtype=torch.float32, device=dev)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_cmp - 1)]
    greedy = ref.greedy(n_cmp, margins=margins, events=sev)
    torch.cuda.synchronize()
    w0 = min(3, n_cmp - 2)
    base_ms = sev[w0][0].elapsed_time(sev[-1][1]) / (n_cmp - 1 - w0)
    base_tps = M_B / (base_ms / 1e3)
    mg = margins.t().cpu().numpy()
    near = mism = mism_near = 0
    for b in range(M_B):
        for t, (a, g) in enumerate(zip(emitted[b][:n_cmp], greedy[b])):
            tie = bool(mg[b, t] < 1e-3)
            near += tie
            if a != g:
                mism += 1
                mism_near += tie
    check = {"tokens_compared": n_cmp * M_B, "mismatches": mism, "near_ties": near,
             "mismatches_at_near_ties": mism_near, "mismatches_elsewhere": mism - mism_near,
             "near_tie_rule": "top-2 logit margin of the reference step below 1e-3",
             "reference": "plain full-KV greedy decoding of the same model and prompts (one-token forwards)"}
    base = {"tokens_per_s": base_tps, "ms_per_token_step": base_ms, "steps_timed": n_cmp - 1 - w0,
            "what": "plain greedy decoding with the full cache in pinned host memory (same format) swapped in "
                    "before every token, one-token forward, argmax, write-back of the new row",
            "speedup_of_draft_and_verify": value / base_tps}
    del ref
    torch.cuda.empty_cache()

    # cross-resource staggering of two request groups (half the batch each):
    # one group's full-cache swap crosses the link while the other drafts and
    # verifies; measured against the unstaggered rounds above
    stag = None if args.no_stagger else run_staggered(args, dec, cfg, prompt, packed, dev, greedy, n_cmp,
                                                      value / world)

    # the one-layer hot path at the configuration of the kernel workloads
    # (B16, 32k): draft attention (2-bit KIVI), verify attention (Dq 33) and
    # acceptance over [16, 33, 151936], timed inside a staggered round
    round_k = None if args.no_round_kernels else round_kernels(dev, hbm, tf_burst)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = model_cpu_record(cfg, P, args.bits, tokens / args.steps,
                               f"tokens per round as measured on the GPU ({tokens / args.steps:.1f})")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights)",
            "config": {"workload": MODEL_WORKLOAD.format(ctx=P, bits=args.bits) +
                       (", keys rotated (Walsh-Hadamard) before quantization" if args.rotate else "") +
                       (", full cache held losslessly packed on the host, expanded on the GPU" if packed else ""),
                       "global_batch": M_B * world,
                       "seq_len": P,
                       "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (no flush)"},
            "roofline": roof,
            "roofline_gemm": roof_gemm,
            "full_kv_baseline": base,
            "lossless_check": check,
            "staggered": stag,
            "phases_ms": {"draft_32_steps": d_ms, "verify_forward": v_ms, "accept_commit_writeback": c_ms,
                          "swap_in": s_ms},
            "swap": {"bytes": run_bytes(cfg, swap_rows, packed),
                     "rows_per_sequence_and_head": swap_rows,
                     "GB/s": run_bytes(cfg, swap_rows, packed) / (s_ms / 1e3) / 1e9,
                     "format": "packed rows (lossless, 208 of 256 bytes)" if packed else "bf16",
                     "hidden_frac": hidden,
                     "hidden_frac_how": "per round, the part of the swap interval inside the drafting interval "
                                        "(device events), over the swap interval"},
            "kernels": kernels,
            "kernels_round_b16_32k": round_k,
            "accepted_per_round_mean": float(n_acc.float().mean()), "tokens_per_round": tokens / args.steps,
            "prefill_s": round(t_pf, 2), "status": st,
            "clocks": clk, "gpu_launches": model_launches_per_round(cfg, vc, packed, args.rotate) * args.steps,
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": run_bytes(cfg, swap_rows, packed),
                    "d2h_bytes_per_step": d2h + model_writeback_bytes(cfg, n_acc, packed),
                    "how": "host wall clock over the same K rounds as value (which uses device events around "
                           "them); each round's tokens are copied to pinned host memory and read by the host while "
                           "the next round runs"},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_staggered(args, dec, cfg, prompt, packed, dev, greedy, n_cmp, unstaggered_tps, cycles: int = 8,
                  warm: int = 3) -> dict:
    """Two half-batch runners ping-ponging on the main stream (decode.StaggeredPair).
    Returns tokens/s, ms per cycle, each swap's overlap with the other group's
    drafting and verify (device events), and the lossless check of both groups
    against the same greedy decoding."""
    from lossless_draft_verify_gb300 import decode
    half = M_B // 2
    P = prompt.shape[1]
    max_len = P + (warm + cycles + 1) * (M_HORIZON + 1) + 64
    mk = lambda: decode.VeriCacheRunner(dec, half, max_len, M_HORIZON, bits=args.bits, residual=M_RESIDUAL,
                                        host_cache=True, prefill_chunk=512, device=dev, pack_host=packed)
    ra, rb = mk(), mk()
    ra.prefill(prompt[:half].contiguous())
    rb.prefill(prompt[half:].contiguous())
    first = ra.x.cpu().tolist() + rb.x.cpu().tolist()
    pair = decode.StaggeredPair(ra, rb)
    la, lb = ra.new_log(warm + cycles), rb.new_log(warm + cycles)
    for i in range(warm):
        pair.cycle(la, lb, i)
    torch.cuda.synchronize()
    ra.capture_draft_graph()
    rb.capture_draft_graph()
    evs = [{k: decode.VeriCacheRunner.new_events() for k in ("A", "B", "A_swap", "B_swap")} for _ in range(cycles)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(cycles):
        pair.cycle(la, lb, warm + i, evs[i])
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    tokens = int((la.n_acc[warm:].long() + 1).sum() + (lb.n_acc[warm:].long() + 1).sum())

    def inside(sw: dict, w0, w1) -> float:
        """Part of the swap interval [swap0, swap1] within [w0, w1], over the swap."""
        span = sw["swap0"].elapsed_time(sw["swap1"])
        lo = max(0.0, sw["swap0"].elapsed_time(w0))
        hi = min(span, sw["swap0"].elapsed_time(w1))
        return max(0.0, hi - lo) / span if span > 0 else 0.0

    ov = []
    for i in range(cycles):
        # A's swap of cycle i runs under B's turn of cycle i, B's under A's turn of cycle i + 1
        ov.append(inside(evs[i]["A_swap"], evs[i]["B"]["d0"], evs[i]["B"]["c1"]))
        if i + 1 < cycles:
            ov.append(inside(evs[i]["B_swap"], evs[i + 1]["A"]["d0"], evs[i + 1]["A"]["c1"]))
    swap_ms = statistics.mean(e[k]["swap0"].elapsed_time(e[k]["swap1"]) for e in evs for k in ("A_swap", "B_swap"))
    turn_ms = statistics.mean(e[k]["d0"].elapsed_time(e[k]["c1"]) for e in evs for k in ("A", "B"))
    draft_ms = statistics.mean(e[k]["d0"].elapsed_time(e[k]["d1"]) for e in evs for k in ("A", "B"))
    emitted = [[first[b]] + t for b, t in enumerate(la.tokens() + lb.tokens())]
    n = min(n_cmp, min(len(t) for t in emitted))
    mism = sum(int(a != g) for b in range(M_B) for a, g in zip(emitted[b][:n], greedy[b][:n]))
    tps = tokens / (ms / 1e3)
    out = {"tokens_per_s": tps, "ms_per_cycle": ms / cycles, "groups": 2, "sequences_per_group": half,
           "swap_ms_per_group": swap_ms, "group_turn_ms": turn_ms, "group_draft_ms": draft_ms,
           "swap_hidden_under_other_group_frac": statistics.mean(ov),
           "vs_unstaggered": tps / unstaggered_tps,
           "lossless_check": {"tokens_compared": n * M_B, "mismatches": mism},
           "what": "two groups of 4 sequences, each its own runner; a group's swap runs while the other group "
                   "drafts and verifies (one link, one main stream); drafting streams the model's weights per "
                   "group, so each group's 32 draft steps cost about what the whole batch's do"}
    del pair, ra, rb
    torch.cuda.empty_cache()
    return out


def model_writeback_bytes(cfg, n_acc, packed: bool) -> int:
    """Bytes per round the write-back stores into the host copy (committed
    rows, K and V, every layer)."""
    row = 16 + 3 * cfg.head_dim // 2 if packed else cfg.head_dim * 2
    rows = float((n_acc.float() + 1).sum(dim=1).mean()) if n_acc.dim() == 2 else float((n_acc.float() + 1).sum())
    return int(2 * cfg.n_layers * cfg.n_kv_heads * rows * row)


def round_kernels(dev, hbm, tf_burst, steps: int = 5, warmup: int = 3) -> dict:
    """Per-kernel numbers of the one-layer round at B16 and 32k context
    (draft attention over the 2-bit cache, verify attention at Dq 33,
    acceptance over [16, 33, 151936] bf16 logits, the packed swap), timed
    with events inside the staggered round."""
    rnd = Round(dev, stagger=2, packed=True)
    for _ in range(warmup):
        rnd.step()
    torch.cuda.synchronize()
    evs = [make_events(HORIZON, rnd.stagger) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        rnd.step(evs[i])
    t1.record()
    torch.cuda.synchronize()
    d_ms = [e["d0"][j].elapsed_time(e["d1"][j]) for e in evs for j in range(HORIZON)]
    d_bytes = [rnd.draft_bytes(j) for _ in evs for j in range(HORIZON)]
    v_ms = [sum(a.elapsed_time(b) for a, b in zip(e["v0"], e["v1"])) for e in evs]
    a_ms = [e["v1"][-1].elapsed_time(e["a1"]) for e in evs]
    s_ms = [e["swap0"].elapsed_time(e["swap1"]) for e in evs]
    draft_gbs = sum(d_bytes) / (sum(d_ms) / 1e3) / 1e9
    ver_tflops = rnd.verify_flops() / (statistics.mean(v_ms) / 1e3) / 1e12
    ver_gbs = rnd.verify_bytes() / (statistics.mean(v_ms) / 1e3) / 1e9
    acc_gbs = (rnd.logits.numel() * 2) / (statistics.mean(a_ms) / 1e3) / 1e9
    out = {
        "what": "one decoder layer's hot path at B16, 32/8 heads, d128, 32768-token context (the draft-attention, "
                "verify-attention and acceptance workloads), timed with events inside the staggered round; these "
                "rounds plant their acceptance in synthetic logits and are not lossless tokens",
        "ms_per_round": t0.elapsed_time(t1) / steps,
        "draft_attn": {"ms": statistics.mean(d_ms), "GB/s": draft_gbs, "hbm_frac": draft_gbs / hbm,
                       "bytes": int(statistics.mean(d_bytes)),
                       "traffic": captured_traffic(DRAFT_TRAFFIC, statistics.mean(d_bytes))},
        "verify_attn_dq33": {"ms": statistics.mean(v_ms), "TFLOP/s": ver_tflops, "tc_frac_burst": ver_tflops / tf_burst,
                             "GB/s": ver_gbs, "hbm_frac": ver_gbs / hbm, "flops": rnd.verify_flops(),
                             "bytes": rnd.verify_bytes()},
        "accept": {"ms": statistics.mean(a_ms), "GB/s": acc_gbs, "hbm_frac": acc_gbs / hbm},
        "swap_in_packed": {"ms": statistics.mean(s_ms), "GB/s": rnd.swap_bytes / (statistics.mean(s_ms) / 1e3) / 1e9,
                           "bytes": rnd.swap_bytes},
    }
    del rnd
    torch.cuda.empty_cache()
    return out


def model_launches_per_round(cfg, vc, packed: bool = False, rotate: bool = False) -> int:
    """Kernels the library launches in one round of the model workload,
    counted from the decoder's sequencing.  A GEMM with more than one K split
    adds a reduction launch when its grid has more than 64 output tiles (fewer
    tiles, or the LM head's argmax epilogue, sum the splits inside the GEMM).
    A packed host cache adds the expansion of K and V per layer.  In draft
    steps RoPE writes the new rows into the compressed cache's ring itself,
    unless the cache rotates its keys (then a ring append follows)."""
    qd, kvd = cfg.n_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    shapes = [(qd + 2 * kvd, cfg.d_model), (cfg.d_model, qd), (2 * cfg.d_ff, cfg.d_model), (cfg.d_model, cfg.d_ff)]

    def g(M, N, K, decode, argmax=False):
        tiles = -(-M // 128) * (N // 128)
        split = vc.vc_gemm_splits(torch.bfloat16, N, K, decode) > 1
        return 1 + int(split and tiles > 64 and not argmax)

    def layer(M, decode, attn_kernels):
        # rmsnorm, qkv, rope, attention, o, rmsnorm, gate_up, silu, down; the
        # SwiGLU runs in the gate|up GEMM's epilogue when that product is unsplit,
        # and in draft steps (M <= 16) the q|k|v and gate|up GEMMs normalise
        # their input rows themselves (no RMSNorm launches)
        fused = vc.vc_gemm_splits(torch.bfloat16, 2 * cfg.d_ff, cfg.d_model, decode) == 1
        norms = 0 if (decode and M <= 16) else 2
        return norms + 1 + sum(g(M, N, K, decode) for N, K in shapes) + (0 if fused else 1) + attn_kernels

    rows_v = M_B * (M_HORIZON + 1)
    # embed, layers (+ append with rotated keys), LM head (argmax, normalising its rows), acceptance,
    # scatter, status fold
    draft = 1 + cfg.n_layers * (layer(M_B, True, 1) + int(rotate)) + g(M_B, cfg.vocab, cfg.d_model, True, True) + 3
    # embed, layers (verify attention + its combine), rmsnorm, LM head (argmax), acceptance, status fold
    verify = 1 + cfg.n_layers * layer(rows_v, False, 2) + 1 + g(rows_v, cfg.vocab, cfg.d_model, False, True) + 2
    # + the commit (one append per layer) and the host write-back
    return M_HORIZON * draft + verify + cfg.n_layers + 1 + (2 * cfg.n_layers if packed else 0)


def run_bytes(cfg, rows: float, packed: bool = False) -> float:
    """Bytes of one full-cache swap-in of `rows` rows per (sequence, kv head)
    (K and V, every layer), bf16 or packed rows."""
    row = 16 + 3 * cfg.head_dim // 2 if packed else cfg.head_dim * 2
    return 2 * cfg.n_layers * M_B * cfg.n_kv_heads * rows * row


def full_kv_step_ms(rnd, steps: int, warmup: int) -> float:
    """Plain decoding with the full cache held on the host: every decoded token
    needs the whole cache swapped in, then a one-query verify pass and the
    argmax (the full-KV baseline of the pages' comparison).  Returns ms per
    token step for all B sequences."""
    vc, main = rnd.vc, torch.cuda.current_stream()
    q1 = rnd.q_ver[:, :1].contiguous()
    o1 = torch.empty_like(q1)
    lg1 = rnd.logits[:, :1].contiguous()
    ws = vc.Workspace(vc.vc_verify_attn_workspace_bytes(torch.bfloat16, B, 1, HQ, HKV, D_HEAD, CTX), device=rnd.dev)
    ev = torch.cuda.Event()

    def one():
        rnd.side.wait_stream(main)
        for t, h in ((rnd.kfull, rnd.kfull_host), (rnd.vfull, rnd.vfull_host)):
            if rnd.link_gbps:
                vc.vc_swap_in_paced(t, h, rnd.link_gbps, rnd.pace_ws, stream=rnd.side, done_event=ev)
            else:
                vc.vc_swap_in(t, h, stream=rnd.side, done_event=ev)
        main.wait_event(ev)
        vc.vc_verify_attn(q1, rnd.kfull, rnd.vfull, rnd.ctx, CTX, rnd.scale, o1, ws)
        vc.vc_accept(lg1, None, rnd.n_acc, rnd.next_tok, rnd.ws_a)
    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        one()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def run_sweep(args, dev):
    """Draft-horizon sweep of the round workload (pages: draft horizon against
    throughput; the divergence point of each sequence is uniform in [0, D]).
    One JSON line per horizon: tokens per round, round time, drafting and swap
    times.  Not the benchmark's contract line."""
    if args.sweep == "budget":
        # compressed-cache budget: code width and full-precision window; bytes
        # the draft step reads per token of context, against round time
        for cfg in args.sweep_budgets.split(","):
            bits, res = (int(x) for x in cfg.split("/"))
            rnd = Round(dev, stagger=args.stagger, bits=bits, residual=res)
            for _ in range(args.warmup):
                rnd.step()
            torch.cuda.synchronize()
            evs = [make_events(rnd.D, rnd.stagger) for _ in range(args.steps)]
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for i in range(args.steps):
                rnd.step(evs[i])
            t1.record()
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1) / args.steps
            tokens = rnd.tokens_per_round()
            d_ms = statistics.mean(sum(e["d0"][j].elapsed_time(e["d1"][j]) for j in range(rnd.D)) for e in evs)
            per_step = rnd.draft_bytes(0)
            full = 2 * B * HKV * CTX * D_HEAD * 2
            print(json.dumps({"sweep": "budget", "bits": bits, "residual": res,
                              "draft_bytes_per_step": per_step, "fraction_of_full_kv": per_step / full,
                              "draft_attn_ms_per_round": d_ms, "draft_GB/s": rnd.D * per_step / d_ms / 1e6,
                              "ms_per_round": ms, "tokens_per_round": tokens,
                              "tokens_per_s": tokens / (ms / 1e3)}), flush=True)
            del rnd
            torch.cuda.empty_cache()
        return
    if args.sweep == "link":
        # the full cache behind slower stores (remote prefix caching): draft and
        # verify against the full-KV baseline at each source rate
        for r in args.sweep_links.split(","):
            gbps = None if r == "native" else float(r)
            rnd = Round(dev, stagger=args.stagger, link_gbps=gbps)
            for _ in range(args.warmup):
                rnd.step()
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(args.steps):
                rnd.step()
            t1.record()
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1) / args.steps
            tokens = rnd.tokens_per_round()
            base_ms = full_kv_step_ms(rnd, max(2, args.steps // 2), 2)
            vt, bt = tokens / (ms / 1e3), B / (base_ms / 1e3)
            print(json.dumps({"sweep": "link", "source_gbps": r, "ms_per_round": ms, "tokens_per_round": tokens,
                              "tokens_per_s": vt, "full_kv_ms_per_token_step": base_ms, "full_kv_tokens_per_s": bt,
                              "speedup": vt / bt}), flush=True)
            del rnd
            torch.cuda.empty_cache()
        return
    for D in [int(x) for x in args.sweep_horizons.split(",")]:
        rnd = Round(dev, stagger=args.stagger, horizon=D)
        for _ in range(args.warmup):
            rnd.step()
        torch.cuda.synchronize()
        evs = [make_events(D, rnd.stagger) for _ in range(args.steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for i in range(args.steps):
            rnd.step(evs[i])
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / args.steps
        tokens = rnd.tokens_per_round()
        d_ms = statistics.mean(sum(e["d0"][j].elapsed_time(e["d1"][j]) for j in range(D)) for e in evs)
        s_ms = statistics.mean(e["swap0"].elapsed_time(e["swap1"]) for e in evs)
        print(json.dumps({"sweep": "horizon", "horizon": D, "tokens_per_round": tokens, "ms_per_round": ms,
                          "tokens_per_s": tokens / (ms / 1e3), "draft_attn_ms_per_round": d_ms,
                          "swap_ms": s_ms, "stagger": rnd.stagger}), flush=True)
        del rnd
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernel", default=None,
                    help="time one kernel alone: draft, verify, verify_h2o, accept, quantize, drop, dense_draft, "
                         "dense_draft_h2o, gemm, unpack, swap")
    ap.add_argument("--dq", type=int, default=32, help="verify block size for --kernel verify")
    ap.add_argument("--batch", type=int, default=B, help="sequences for --kernel draft/verify")
    ap.add_argument("--ctx", type=int, default=CTX, help="context tokens for --kernel draft/quantize")
    ap.add_argument("--chunks", type=int, default=1, help="side streams for --kernel swap")
    ap.add_argument("--stagger", type=int, default=2, choices=[1, 2],
                    help="round workload: swap and verify per half batch (2) or whole batch (1)")
    ap.add_argument("--swap", default=None, choices=["packed", "raw"],
                    help="the full cache on the host packed (lossless rows of 16 + 3d/2 bytes, expanded on the "
                         "GPU after each swap; the default) or as plain bf16")
    ap.add_argument("--workload", default="model", choices=["round", "model"],
                    help="model (default): the 8-layer decoder end to end, lossless tokens/s; round: one layer's "
                         "hot path at 32k (B16) with planted acceptance")
    ap.add_argument("--no-round-kernels", action="store_true",
                    help="--workload model: skip the one-layer B16 round that reports the kernel workloads")
    ap.add_argument("--no-stagger", action="store_true",
                    help="--workload model: skip the staggered two-group measurement")
    ap.add_argument("--prompt", type=int, default=32768, help="prompt tokens per sequence (--workload model)")
    ap.add_argument("--no-check", action="store_true", help="skip the lossless check (--workload model)")
    ap.add_argument("--check-tokens", type=int, default=256, help="tokens per sequence compared by the check")
    ap.add_argument("--bits", type=int, default=2, choices=[2, 4], help="draft cache bits (--workload model)")
    ap.add_argument("--expand-during-draft", action="store_true",
                    help="model workload: expand the packed swap as each layer lands, during the draft steps "
                         "(default: after them)")
    ap.add_argument("--no-graph", action="store_true",
                    help="--workload model: launch the draft steps one by one instead of replaying a CUDA graph")
    ap.add_argument("--rotate", action="store_true",
                    help="draft caches with rotated keys (--workload model; the RotateKV-style variant)")
    ap.add_argument("--sweep", default=None, choices=["horizon", "link", "budget"],
                    help="print a sweep instead of the contract line")
    ap.add_argument("--sweep-links", default="native,100,50,25,12.5", help="source rates in GB/s for --sweep link")
    ap.add_argument("--sweep-horizons", default="8,16,32,64,96,128")
    ap.add_argument("--sweep-budgets", default="2/128,2/1024,2/4096,4/128,4/1024,4/4096",
                    help="bits/residual pairs for --sweep budget")
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.kernel:
        torch.cuda.set_device(local)
        from lossless_draft_verify_gb300 import build
        build.build()
        run_kernel(args, torch.device("cuda", local))
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    from lossless_draft_verify_gb300 import build, replicas
    build.build()

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    if args.sweep:
        run_sweep(args, dev)
        return
    if args.workload == "model":
        run_model(args, dev, rank, world, barrier, pg)
        if pg is not None:
            pg.destroy_process_group()
        return
    rnd = Round(dev, stagger=args.stagger, packed=args.swap != "raw")      # default packed

    for _ in range(args.warmup):
        rnd.step()
    barrier()
    evs = [make_events(HORIZON, rnd.stagger) for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0.record()
    for i in range(args.steps):
        rnd.step(evs[i])
    t1.record()
    barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    st = rnd.vc.vc_poll_status(rnd.ws_d) | rnd.vc.vc_poll_status(rnd.ws_v)
    tokens = rnd.tokens_per_round()
    value, ms_max = replicas.whole_job_rate(tokens * args.steps, ms, pg, device=dev)

    # per-kernel times from the events
    d_ms = [e["d0"][j].elapsed_time(e["d1"][j]) for e in evs for j in range(HORIZON)]
    d_bytes = [rnd.draft_bytes(j) for _ in evs for j in range(HORIZON)]
    v_ms = [sum(a.elapsed_time(b) for a, b in zip(e["v0"], e["v1"])) for e in evs]
    a_ms = [e["v1"][-1].elapsed_time(e["a1"]) for e in evs]
    s_ms = [e["swap0"].elapsed_time(e["swap1"]) for e in evs]
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    draft_gbs = sum(d_bytes) / (sum(d_ms) / 1e3) / 1e9
    ver_tflops = rnd.verify_flops() / (statistics.mean(v_ms) / 1e3) / 1e12
    ver_gbs = rnd.verify_bytes() / (statistics.mean(v_ms) / 1e3) / 1e9
    acc_gbs = (rnd.logits.numel() * 2) / (statistics.mean(a_ms) / 1e3) / 1e9
    swap_gbs = rnd.swap_bytes / (statistics.mean(s_ms) / 1e3) / 1e9
    draft_total = sum(d_ms) / args.steps
    overlap = min(1.0, draft_total / statistics.mean(s_ms)) if s_ms else None

    # end-to-end: same round with host inputs copied in and results read back
    e2e_val = None
    if not args.no_e2e:
        for _ in range(2):
            rnd.step(e2e=True)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            rnd.step(e2e=True)
        e1.record()
        barrier()
        e2e_val, _ = replicas.whole_job_rate(tokens * args.steps, e0.elapsed_time(e1), pg, device=dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_record(rnd, tokens)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_PACKED if rnd.packed else WORKLOAD, "global_batch": B * world,
                       "seq_len": CTX,
                       "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (no flush)",
                       "stagger": rnd.stagger,
                       "swap": ("full cache held packed on the host (lossless, 208 of 256 bytes a row), "
                                "expanded on the GPU" if rnd.packed else "full bf16 cache")},
            "roofline": {"bound": "hbm", "achieved": draft_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": draft_gbs / hbm,
                         "traffic": captured_traffic(DRAFT_TRAFFIC, statistics.mean(d_bytes)),
                         "kernel": "vc_draft_attn (draft_kivi_kernel + combine)",
                         "peak_source": f"{peak_src} hbm_gbs"},
            "kernels": {
                "draft_attn": {"ms": statistics.mean(d_ms), "GB/s": draft_gbs, "hbm_frac": draft_gbs / hbm,
                               "bytes": int(statistics.mean(d_bytes)), "launches_per_step": HORIZON},
                "verify_attn": {"ms": statistics.mean(v_ms), "TFLOP/s": ver_tflops,
                                "tc_frac_burst": ver_tflops / tf_burst, "GB/s": ver_gbs, "hbm_frac": ver_gbs / hbm,
                                "flops": rnd.verify_flops(), "bytes": rnd.verify_bytes()},
                "accept": {"ms": statistics.mean(a_ms), "GB/s": acc_gbs, "hbm_frac": acc_gbs / hbm},
                "swap_in": {"ms": statistics.mean(s_ms), "GB/s": swap_gbs, "bytes": rnd.swap_bytes,
                            "hidden_frac": overlap},
            },
            "tokens_per_round": tokens, "status": st,
            "clocks": clk, "gpu_launches": rnd.launches_per_step * args.steps,
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": rnd.h2d_bytes,
                    "d2h_bytes_per_step": rnd.d2h_bytes},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
