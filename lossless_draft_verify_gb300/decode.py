"""Host-side sequencing of VeriCache decoding on one GPU: prefill, plain
full-KV greedy decoding, and draft-and-verify rounds.

Every computation is a call into libvc.so (vc.py); this module only orders
the calls on CUDA streams and moves bookkeeping tensors with plain copies
(paper page, "What the paper found": draft on the compressed cache, swap the
full cache in from host memory at the same time, verify the drafted block on
the full cache, keep the longest prefix that matches).

A round for B sequences whose pending token x sits at position P (its K/V
not yet cached):
  1. the full cache is copied in from pinned host memory on a side stream
     (when the cache lives on the host);
  2. D draft steps on the compressed per-layer caches, each appending the
     input's K/V to the ring and producing the greedy draft token;
  3. one forward of [x, d1..dD] at positions P..P+D over the full cache (the
     verify pass, waiting for the copy), writing the block's K/V;
  4. acceptance: n = longest prefix with argmax(row i) == d(i+1), next =
     argmax(row n) (by default from the LM head's argmax epilogue, so the
     verify logits are never written; fused_head=False writes them and scans);
  5. the compressed caches roll back to P and take the verify pass's K/V of
     the n + 1 committed rows (re-quantized); the host copy of the full cache
     receives the same rows.
The round emits d1..dn and next.
"""
from __future__ import annotations

import contextlib
import dataclasses

import torch

from . import vc


@dataclasses.dataclass
class RoundLog:
    drafts: torch.Tensor        # [R][B][D] int32 (device)
    n_acc: torch.Tensor         # [R][B]
    nxt: torch.Tensor           # [R][B]

    def tokens(self) -> list[list[int]]:
        """Emitted tokens per sequence (host lists), in order."""
        d, n, x = self.drafts.cpu(), self.n_acc.cpu(), self.nxt.cpu()
        R, B, _ = d.shape
        out = [[] for _ in range(B)]
        for r in range(R):
            for b in range(B):
                k = int(n[r, b])
                out[b].extend(int(t) for t in d[r, b, :k])
                out[b].append(int(x[r, b]))
        return out

    def accepted(self) -> list[list[int]]:
        return self.n_acc.cpu().t().tolist()


class VeriCacheRunner:
    """Caches, workspaces and buffers of one decoding job (B sequences)."""

    def __init__(self, dec: vc.Decoder, B: int, max_len: int, horizon: int, bits: int = 2, group: int = 32,
                 residual: int = 128, host_cache: bool = False, prefill_chunk: int = 512, device="cuda",
                 fused_head: bool = True, rotate: bool = False, use_graph: bool = False, pack_host: bool = False):
        cfg = dec.cfg
        self.dec, self.B, self.D, self.device = dec, B, horizon, device
        # use_graph: after one eager round, the round's D draft steps (about a
        # hundred short launches each) are captured once as a CUDA graph and
        # replayed every round; every buffer they touch is fixed, so the graph
        # stays valid for the runner's lifetime
        self.use_graph = use_graph
        self._graph = None
        self._rounds = 0
        # fused_head: draft steps and the verify pass take the greedy tokens
        # from the LM head's argmax epilogue (no logits written)
        self.fused_head = fused_head
        self.dtype = dec.dtype
        self.L_stride = max_len + horizon + 1
        nl, hkv, hd = cfg.n_layers, cfg.n_kv_heads, cfg.head_dim
        shape = (nl, B, hkv, self.L_stride, hd)
        self.k_full = torch.zeros(shape, dtype=self.dtype, device=device)
        self.v_full = torch.zeros_like(self.k_full)
        self.host_cache = host_cache
        # pack_host: the host copy is held packed (vc_kv_pack rows); each round
        # moves the packed bytes into a device staging buffer and expands them
        # into the full cache, and the write-back packs the committed rows
        self.pack_host = host_cache and pack_host
        if self.pack_host:
            assert self.dtype == torch.bfloat16
            pshape = shape[:-1] + (vc.vc_kv_packed_row_bytes(hd),)
            self.k_host = torch.zeros(pshape, dtype=torch.uint8).pin_memory()
            self.v_host = torch.zeros(pshape, dtype=torch.uint8).pin_memory()
            self.k_pack = torch.zeros(pshape, dtype=torch.uint8, device=device)
            self.v_pack = torch.zeros_like(self.k_pack)
            self.n_over = torch.zeros(1, dtype=torch.int32, device=device)
            # layer l is expanded on its own stream while layer l + 1 is on
            # the link
            self.unpack_stream = torch.cuda.Stream(device=device)
            self.ev_layer = [torch.cuda.Event() for _ in range(nl)]
        elif host_cache:
            self.k_host = torch.zeros(shape, dtype=self.dtype).pin_memory()
            self.v_host = torch.zeros(shape, dtype=self.dtype).pin_memory()
        maxg = self.L_stride // group + 1
        res_cap = ((residual + group + horizon + 1 + 15) // 16) * 16
        # rotate: draft caches with rotated keys (vc_quant_cfg.rotate)
        self.qc = [vc.QCache(B, hkv, hd, bits, maxg, res_cap, residual, group=group, res_dtype=self.dtype,
                             device=device, rotate=rotate) for _ in range(nl)]
        self.qc_arr = vc.qcache_array(self.qc)
        self.k_blk = torch.zeros(nl, B, hkv, horizon + 1, hd, dtype=self.dtype, device=device)
        self.v_blk = torch.zeros_like(self.k_blk)
        self.prefill_chunk = prefill_chunk
        rows = max(prefill_chunk, horizon + 1)
        self.ws = vc.Workspace(dec.workspace_bytes(B, rows, self.L_stride - rows, self.qc[0]), device=device)
        self.logits_d = torch.zeros(B, cfg.vocab, dtype=self.dtype, device=device)
        self.logits_v = torch.zeros(B, horizon + 1, cfg.vocab, dtype=self.dtype, device=device)
        self.ws_acc = vc.Workspace(vc.vc_accept_workspace_bytes(B, horizon, cfg.vocab), device=device)
        self.x = torch.zeros(B, dtype=torch.int32, device=device)          # pending token
        self.next_d = torch.zeros(B, dtype=torch.int32, device=device)
        self.drafts = torch.zeros(B, horizon, dtype=torch.int32, device=device)
        self.n_acc = torch.zeros(B, dtype=torch.int32, device=device)
        self.round_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.ctx = torch.zeros(B, dtype=torch.int32, device=device)
        self.ctx_bound = 0
        self.side = torch.cuda.Stream(device=device)
        self.ev_swap = torch.cuda.Event()
        # ev_ready[l]: layer l of the swapped-in cache is resident (copied, and
        # expanded when packed); a forward over the full cache waits on it
        # before touching layer l, so the verify pass overlaps the swap's tail
        self.ev_ready = [torch.cuda.Event() for _ in range(nl)] if host_cache else None
        # expand_after_draft: in round(), packed rows are expanded after the
        # draft steps instead of while they run
        self.expand_after_draft = True
        self.ev_drafted = torch.cuda.Event()
        self.swap_rows: list[int] = []    # rows per (sequence, head) each swap copied

    # ------------------------------------------------------------ prefill --
    def prefill(self, prompt: torch.Tensor):
        """prompt: [B][P] int32 on the device.  Fills the full cache (and its
        host copy), quantizes it into the draft caches, sets the pending
        token to the greedy continuation."""
        B, P = prompt.shape
        assert B == self.B and P + 1 <= self.L_stride
        prompt = prompt.to(torch.int32).contiguous()
        C = self.prefill_chunk
        starts = list(range(0, P, C))
        ctxs = torch.tensor([[s] * B for s in starts], dtype=torch.int32, device=self.device)
        last = torch.zeros(B, self.dec.cfg.vocab, dtype=self.dtype, device=self.device)
        for ci, s in enumerate(starts):
            n = min(C, P - s)
            vc.vc_decoder_forward(self.dec, None, prompt[:, s:], P, B, n, ctxs[ci], s, self.k_full, self.v_full,
                                  last, self.ws, last_only=True)
        vc.vc_accept(last.view(B, 1, -1), None, self.n_acc, self.x, self.ws_acc)
        self.last_logits = last
        for l, q in enumerate(self.qc):
            vc.vc_quantize_kv(self.k_full[l], self.v_full[l], q, L=P)
        if self.pack_host:
            vc.vc_kv_pack(self.k_full, self.k_pack, self.n_over)
            vc.vc_kv_pack(self.v_full, self.v_pack, self.n_over)
            if int(self.n_over.item()):
                # a prompt row the packed format cannot hold: keep a bf16 host copy
                self.pack_host = False
                del self.k_pack, self.v_pack, self.unpack_stream, self.ev_layer
                self.k_host = torch.empty(self.k_full.shape, dtype=self.dtype).pin_memory()
                self.v_host = torch.empty(self.v_full.shape, dtype=self.dtype).pin_memory()
            else:
                self.k_host.copy_(self.k_pack)
                self.v_host.copy_(self.v_pack)
        if self.host_cache and not self.pack_host:
            self.k_host.copy_(self.k_full)
            self.v_host.copy_(self.v_full)
        self.ctx.fill_(P)
        self.ctx_bound = P
        self.round_len.copy_(self.qc[0].seq_len)
        return self.x

    def check_packed(self):
        """Raise if a committed row could not be packed into the host copy (a
        row with more than 7 values far below its largest one): the copy is
        then unusable.  (A prompt row that cannot be packed makes prefill keep a
        bf16 host copy instead.)"""
        if self.pack_host and int(self.n_over.item()):
            raise RuntimeError(f"{int(self.n_over.item())} K/V rows cannot be held packed; use pack_host=False")

    # ------------------------------------------------------- plain greedy --
    def greedy(self, n_new: int, margins: torch.Tensor | None = None, events: list | None = None
               ) -> list[list[int]]:
        """Plain full-KV greedy decoding from the pending token: n_new tokens
        per sequence, the first being the pending token itself.

        With a host cache this is full-KV inference over an offloaded cache
        (the baseline the paper page compares against, "What the paper
        found"): the whole cache is swapped in before every token, and each
        token's K/V row is written back to the host copy.
        margins: optional device fp32 [n_new][B]; row t receives the gap
        between the largest and second-largest logit of the step that chose
        token t (row 0: the prefill's last row).  events: optional list of
        n_new - 1 (start, end) CUDA event pairs around the token steps."""
        B = self.B
        main = torch.cuda.current_stream()
        out = torch.zeros(n_new, B, dtype=torch.int32, device=self.device)
        out[0].copy_(self.x)
        if margins is not None:
            margins[0].copy_(self._top2_margin(self.last_logits))
        if self.host_cache:
            nl, hkv, hd = self.dec.cfg.n_layers, self.dec.cfg.n_kv_heads, self.dec.cfg.head_dim
            k1 = torch.zeros(nl, B, hkv, 1, hd, dtype=self.dtype, device=self.device)
            v1 = torch.zeros_like(k1)
            zero = torch.zeros(B, dtype=torch.int32, device=self.device)
        for t in range(1, n_new):
            if events is not None:
                events[t - 1][0].record(main)
            if self.host_cache:
                self._swap_in(main)
                with self._layer_arrivals():
                    vc.vc_decoder_forward(self.dec, self.x, None, 0, B, 1, self.ctx, self.ctx_bound, self.k_full,
                                          self.v_full, self.logits_d, self.ws, k_blk=k1, v_blk=v1, last_only=True)
            else:
                vc.vc_decoder_forward(self.dec, self.x, None, 0, B, 1, self.ctx, self.ctx_bound, self.k_full,
                                      self.v_full, self.logits_d, self.ws, last_only=True)
            vc.vc_accept(self.logits_d.view(B, 1, -1), None, self.n_acc, self.x, self.ws_acc)
            if self.host_cache:
                main.wait_event(self.ev_swap)          # the copy has read the host copy
                self._write_back(k1, v1, zero, self.ctx)
            if events is not None:
                events[t - 1][1].record(main)
            if margins is not None:
                margins[t].copy_(self._top2_margin(self.logits_d))
            out[t].copy_(self.x)
            self.ctx += 1
            self.ctx_bound += 1
        return out.t().cpu().tolist()

    @contextlib.contextmanager
    def _layer_arrivals(self):
        """While enqueuing a forward over the swapped-in cache: the decoder
        waits on this runner's per-layer arrival events (the decoder object
        may be shared with other runners, so they are cleared afterwards)."""
        if not self.host_cache:
            yield
            return
        vc.vc_decoder_set_layer_events(self.dec, self.ev_ready)
        try:
            yield
        finally:
            vc.vc_decoder_set_layer_events(self.dec, None)

    @staticmethod
    def _top2_margin(logits: torch.Tensor) -> torch.Tensor:
        """Per row, largest minus second-largest logit (bookkeeping of the
        losslessness check, not part of decoding)."""
        top = torch.topk(logits.float(), 2, dim=-1).values
        return top[..., 0] - top[..., 1]

    def _swap_copies(self, ev: dict | None = None):
        """The link part of the swap: the host copy of the full cache (the rows
        that can hold tokens) into the device, layer by layer on the side stream (packed rows into the
        staging buffer, each layer marked by ev_layer[l]; bf16 rows straight
        into the cache, each layer marked by ev_ready[l]).  ev["swap0"] and
        ev["swap1"] bracket the transfer."""
        if ev is not None:
            ev["swap0"].record(self.side)
        # every sequence holds at most ctx_bound tokens, and a forward writes its
        # own rows before reading them: the rows past the bound stay behind
        rows = min(self.ctx_bound, self.L_stride)
        self.swap_rows.append(rows)
        for l in range(len(self.qc)):
            if self.pack_host:
                vc.vc_swap_in_rows(self.k_pack[l], self.k_host[l], rows, stream=self.side)
                vc.vc_swap_in_rows(self.v_pack[l], self.v_host[l], rows, stream=self.side,
                                   done_event=self.ev_layer[l])
            else:
                vc.vc_swap_in_rows(self.k_full[l], self.k_host[l], rows, stream=self.side)
                vc.vc_swap_in_rows(self.v_full[l], self.v_host[l], rows, stream=self.side,
                                   done_event=self.ev_ready[l])
        if ev is not None:
            ev["swap1"].record(self.side)
        if not self.pack_host:
            self.ev_swap.record(self.side)

    def _swap_expand(self, after: torch.cuda.Event | None = None):
        """Packed rows: each layer expanded into the bf16 cache on the unpack
        stream once its copy has landed (and after `after` when given);
        ev_ready[l] marks layer l, self.ev_swap the whole cache."""
        if not self.pack_host:
            return
        if after is not None:
            self.unpack_stream.wait_event(after)
        for l in range(len(self.qc)):
            self.unpack_stream.wait_event(self.ev_layer[l])
            vc.vc_kv_unpack(self.k_pack[l], self.k_full[l], stream=self.unpack_stream)
            vc.vc_kv_unpack(self.v_pack[l], self.v_full[l], stream=self.unpack_stream)
            self.ev_ready[l].record(self.unpack_stream)
        self.ev_swap.record(self.unpack_stream)

    def _swap_in(self, main: torch.cuda.Stream, ev: dict | None = None, wait_main: bool = True):
        """Copy the host copy of the full cache into the device cache on the
        side stream, packed rows expanded layer by layer on a second stream as
        they land; self.ev_swap marks the end.  wait_main: the copy waits for
        everything issued on `main` so far (else the caller has ordered it)."""
        if wait_main:
            self.side.wait_stream(main)
        self._swap_copies(ev)
        self._swap_expand()

    def _write_back(self, k_blk, v_blk, n_acc, ctx_len):
        """Committed rows (i <= n_acc[b]) of a block into the host copy at
        ctx_len[b] + i."""
        if self.pack_host:
            vc.vc_kv_writeback_packed(k_blk, v_blk, n_acc, ctx_len, self.k_host, self.v_host, self.n_over)
        else:
            vc.vc_kv_writeback(k_blk, v_blk, n_acc, ctx_len, self.k_host, self.v_host)

    # --------------------------------------------------- draft and verify --
    def round(self, log: RoundLog | None = None, r: int = 0, ev: dict | None = None,
              graph: torch.cuda.CUDAGraph | None = None):
        """One draft-and-verify round (enqueued; no host synchronization).
        graph: a recording of the draft steps to replay instead of the
        runner's own (e.g. one captured with tracing on)."""
        main = torch.cuda.current_stream()
        self.round_len.copy_(self.qc[0].seq_len)
        defer = self.host_cache and self.pack_host and self.expand_after_draft
        if self.host_cache:
            self.side.wait_stream(main)
            if defer:
                self._swap_copies(ev)
            else:
                self.swap_phase(ev)
        self.draft_phase(ev, graph)
        if defer:
            # the packed rows are expanded once the draft steps have run, so
            # the expansion's HBM traffic does not slow them (the link copies
            # still overlap them); layer l's verify waits for layer l only
            self.ev_drafted.record(main)
            self._swap_expand(after=self.ev_drafted)
        self.verify_phase(log, r, ev)

    def swap_phase(self, ev: dict | None = None, after: torch.cuda.Event | None = None):
        """Copy the host copy of the full cache in on the side stream (after
        `after` when given); self.ev_swap marks its end."""
        if after is not None:
            self.side.wait_event(after)
        self._swap_in(torch.cuda.current_stream(), ev, wait_main=False)

    def draft_phase(self, ev: dict | None = None, graph: torch.cuda.CUDAGraph | None = None):
        """The round's D draft steps on the compressed caches (main stream)."""
        main = torch.cuda.current_stream()
        if self.use_graph and self._graph is None and self._rounds >= 1:
            self.capture_draft_graph()
        if ev is not None:
            ev["d0"].record(main)
        if graph is not None:
            graph.replay()
        elif self._graph is not None:
            self._graph.replay()
        else:
            self._draft_steps()
        if ev is not None:
            ev["d1"].record(main)

    def verify_phase(self, log: RoundLog | None = None, r: int = 0, ev: dict | None = None):
        """Verify forward of [x, d1..dD] over the full cache (after the swap),
        acceptance, commit to the compressed caches and write-back to the host
        copy (main stream)."""
        B, D = self.B, self.D
        main = torch.cuda.current_stream()
        if ev is not None:
            ev["v0"].record(main)
        max_ctx = min(self.ctx_bound, self.L_stride - (D + 1))
        if self.fused_head:
            # verify pass and acceptance in one call; next token overwrites x
            with self._layer_arrivals():
                vc.vc_decoder_verify(self.dec, self.x, self.drafts, D, B, self.round_len, max_ctx, self.k_full,
                                     self.v_full, self.n_acc, self.x, self.ws, k_blk=self.k_blk, v_blk=self.v_blk)
            if ev is not None:
                ev["v1"].record(main)
        else:
            with self._layer_arrivals():
                vc.vc_decoder_forward(self.dec, self.x, self.drafts, D, B, D + 1, self.round_len, max_ctx,
                                      self.k_full, self.v_full, self.logits_v, self.ws, k_blk=self.k_blk,
                                      v_blk=self.v_blk)
            if ev is not None:
                ev["v1"].record(main)
            vc.vc_accept(self.logits_v, self.drafts, self.n_acc, self.x, self.ws_acc)
        for l, q in enumerate(self.qc):
            vc.vc_qcache_commit(q, self.k_blk[l], self.v_blk[l], self.round_len, self.n_acc)
        if self.host_cache:
            main.wait_event(self.ev_swap)              # the copy has read the host copy
            self._write_back(self.k_blk, self.v_blk, self.n_acc, self.round_len)
        if ev is not None:
            ev["c1"].record(main)
        if log is not None:
            log.drafts[r].copy_(self.drafts)
            log.n_acc[r].copy_(self.n_acc)
            log.nxt[r].copy_(self.x)
        self.ctx_bound += D + 1
        self._rounds += 1
        # the next round's lengths (a copy on the main stream, after the commit)
        self.round_len.copy_(self.qc[0].seq_len)

    def _draft_steps(self):
        """The round's D greedy draft steps on the compressed caches."""
        tok = self.x
        logits_d = None if self.fused_head else self.logits_d
        for j in range(self.D):
            vc.vc_decoder_draft_step(self.dec, tok, self.qc_arr, logits_d, self.next_d, self.ws,
                                     drafts_out=self.drafts[:, j], drafts_stride=self.D)
            tok = self.next_d

    def capture_draft_graph(self, keep: bool = True) -> torch.cuda.CUDAGraph:
        """Record the D draft steps as one CUDA graph (nothing runs while it
        is recorded); with keep, round() replays it from then on."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self._draft_steps()
        if keep:
            self._graph = g
        return g

    @staticmethod
    def new_events() -> dict:
        mk = lambda: torch.cuda.Event(enable_timing=True)
        return {k: mk() for k in ("swap0", "swap1", "d0", "d1", "v0", "v1", "c1")}

    def new_log(self, rounds: int) -> RoundLog:
        B, D = self.B, self.D
        z = lambda *s: torch.zeros(*s, dtype=torch.int32, device=self.device)
        return RoundLog(z(rounds, B, D), z(rounds, B), z(rounds, B))

    def generate(self, n_new: int, max_rounds: int | None = None) -> tuple[list[list[int]], list[list[int]]]:
        """Draft-and-verify until every sequence has n_new tokens (the first
        being the pending token after prefill).  Returns (tokens, accepted
        lengths per round) per sequence."""
        first = self.x.cpu().tolist()
        max_rounds = max_rounds or n_new
        log = self.new_log(max_rounds)
        have = [1] * self.B
        r = 0
        while min(have) < n_new and r < max_rounds:
            self.round(log, r)
            na = log.n_acc[r].cpu().tolist()
            self.check_packed()              # before the next round's swap reads the host copy
            have = [h + k + 1 for h, k in zip(have, na)]
            r += 1
        used = RoundLog(log.drafts[:r], log.n_acc[:r], log.nxt[:r])
        toks = [[first[b]] + t for b, t in enumerate(used.tokens())]
        return [t[:n_new] for t in toks], used.accepted()


class StaggeredPair:
    """Cross-resource staggering of two request groups (paper page, "What the
    paper found"): each group is a runner of half the batch with its own caches
    and side streams, and the two ping-pong on the main stream, so that one
    group's full-cache swap crosses the link while the other group drafts and
    verifies.  A cycle: A drafts, A verifies (after its swap), A's next swap is
    issued; then B drafts, B verifies (after its swap), B's next swap is issued.
    Each group's tokens are those of its own runner (greedy decoding of its
    sequences)."""

    def __init__(self, a: VeriCacheRunner, b: VeriCacheRunner):
        self.a, self.b = a, b
        self.started = False

    def _start(self):
        main = torch.cuda.current_stream()
        for g in (self.a, self.b):
            g.side.wait_stream(main)
            g.swap_phase()
        self.started = True

    def cycle(self, log_a: RoundLog | None = None, log_b: RoundLog | None = None, r: int = 0,
              evs: dict | None = None):
        """One cycle (enqueued).  evs: optional {"A", "B", "A_swap", "B_swap"}
        event dicts (new_events()): each group's phases in this cycle, and the
        swap each group issues at the end of its turn."""
        if not self.started:
            self._start()
        main = torch.cuda.current_stream()
        for name, g, log in (("A", self.a, log_a), ("B", self.b, log_b)):
            ev = evs[name] if evs else None
            g.draft_phase(ev)
            g.verify_phase(log, r, ev)
            done = torch.cuda.Event()
            done.record(main)
            g.swap_phase(evs[name + "_swap"] if evs else None, after=done)

