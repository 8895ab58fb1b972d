/*
 * vc.h -- C ABI of the GB300 (sm_103a) draft-and-verify hot path.
 *
 * The method ("VeriCache: Turning Lossy KV Cache into Lossless LLM Inference",
 * paper page, "What the paper found" and abstract): the target model itself
 * drafts tokens while reading a lossy (quantized or token-dropped) copy of its
 * KV state; the HBM-bound drafting runs while the interconnect-bound copy of
 * the exact KV state comes in; one causal pass over the exact state then
 * checks the whole drafted block, and only the prefix whose verify argmax
 * agrees with the drafts is kept, so the emitted tokens are those of plain
 * greedy decoding.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are caller-owned.  "device" pointers are CUDA device
 *    memory of the current device; "pinned host" pointers are page-locked host
 *    memory.  The library never allocates, frees or retains memory.
 *  - Layouts are dense, row-major, in the element type named by a vc_dtype
 *    argument (VC_BF16: bfloat16, VC_F32: binary32).
 *  - Every call validates its host-side arguments first and returns
 *    VC_ERR_INVALID (bad size, null pointer, misalignment) or
 *    VC_ERR_UNSUPPORTED (valid but not implemented) without touching the
 *    stream.  On success the work is enqueued on `stream` and VC_OK is
 *    returned; the call does not synchronize.  Errors raised later on the
 *    device surface at the caller's next synchronization, or through
 *    vc_check().
 *  - Calls keep no state between invocations and may be issued from several
 *    host threads on different streams.  Calls that share a workspace or a
 *    cache must be ordered by the caller.
 *  - Stream order holds as for any CUDA work.  Most kernels are launched with
 *    programmatic dependent launch: such a kernel may begin while the
 *    previous kernel on `stream` is still running, but it reads nothing
 *    before that kernel has completed and its writes are visible.  The one
 *    exception is the decoder's weights (vc_decoder_create), which must not
 *    change while a decoder call is pending: its projections may start
 *    reading them early.  The environment variable VC_PDL=0 turns this off.
 *  - Workspaces: entry points that combine partial results take a device
 *    workspace `ws` of at least the size returned by the matching
 *    *_workspace_bytes() query, 256-byte aligned.  The first 256 bytes of every
 *    workspace are a status block; kernels whose waits are bounded record a
 *    timeout there (read and cleared by vc_poll_status()).  A new workspace
 *    must be zero-filled once before first use (vc_workspace_init()).
 */
#ifndef VC_H
#define VC_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vc_status {
    VC_OK = 0,
    VC_ERR_INVALID = 1,      /* bad argument: null pointer, size, alignment */
    VC_ERR_UNSUPPORTED = 2,  /* valid request outside what is implemented */
    VC_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    VC_ERR_TIMEOUT = 4       /* a bounded device-side wait gave up */
} vc_status;

typedef enum vc_dtype {
    VC_BF16 = 0,
    VC_F32 = 1
} vc_dtype;

/* Human-readable text for a status code (static storage). */
const char *vc_status_str(vc_status s);

/* Library version string and the device architecture it was built for. */
const char *vc_version(void);

/* Synchronize `stream` and report any asynchronous CUDA error as VC_ERR_CUDA. */
vc_status vc_check(cudaStream_t stream);

/* Zero-fill a new workspace (ws_bytes bytes) on `stream`. */
vc_status vc_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronize `stream`, read the status block of `ws`, clear it.  Returns
 * VC_ERR_TIMEOUT if a kernel that used this workspace gave up on a wait
 * (its outputs are then undefined), VC_OK otherwise. */
vc_status vc_poll_status(void *ws, cudaStream_t stream);

/*
 * vc_wait_probe -- exercises the failure path of the bounded waits (no
 * counterpart in the paper; it makes that path testable without faulting a
 * GPU): one CTA waits on an mbarrier that nothing completes, the wait gives
 * up after 2 s of wall time, records a timeout in the
 * status block of `ws` (>= 256 bytes, 256-byte aligned) and the kernel
 * returns.  vc_poll_status(ws) then reports VC_ERR_TIMEOUT and the context
 * stays usable.
 */
vc_status vc_wait_probe(void *ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (1) KIVI-style quantized draft cache                                      */
/* ------------------------------------------------------------------------ */
/*
 * KIVI (named among the compressors on the paper page, "What the paper
 * found"; ref [42] on pith.science): K is quantized per channel over groups of
 * `group` consecutive tokens, V per token over groups of `group` consecutive
 * channels; every group stores an fp16 scale s and zero-point z and b-bit
 * codes, x^ = code * s + z.  The most recent tokens stay full precision.
 *
 * Rounding rule (the pages give only the name; this is the library's reading):
 *   z = fp16 round-down(min), s = fp16 round-up((max - z) / (2^b - 1)) with
 *   the fp32 subtraction and division rounded upward, code =
 *   clamp(round-half-even((x - z) / s), 0, 2^b - 1) in fp32 round-to-nearest
 *   (code = 0 when s = 0).  Hence z <= min, z + (2^b-1) s >= max and
 *   |x - x^| <= s/2 (up to the rounding of the fp32 quotient).
 *
 * Storage.  Quantized token groups live in fixed-size records, one per
 * (sequence, kv head, group), at
 *   records + ((b * Hkv + h) * max_groups + g) * vc_record_bytes(bits, d).
 * A record is [K codes | V codes | K meta | V meta]:
 *   Code sections (group*d*bits/8 bytes each).  Lane l in [0,32) of the draft
 *     kernel owns W = d*bits/32 little-endian 32-bit words; word w of lane l
 *     sits at byte 16*(32*(w/4) + l) + 4*(w%4) of the section.  A lane's d/2
 *     code pairs follow the m16n8k16 operand fragments: pair (mt, ks, r)
 *     holds elements hh = 0, 1 of fragment register r (row = l/4 + 8*(r&1),
 *     col = 2*(l%4) + hh + 8*(r>>1)):
 *       K: token 16 mt + row, channel 16 ks + col (mt < 2, ks < d/16),
 *          class kappa = 2 ks + (r>>1), member mu = 2 mt + (r&1);
 *       V: channel 16 mt + row, token 16 ks + col (mt < d/16, ks < 2),
 *          class kappa = 2 mt + (r&1), member mu = 2 ks + (r>>1).
 *     Pair (kappa, mu) sits in word `word` at slot `slot` (first element at
 *     bit bits*slot, second at bit 16 + bits*slot):
 *       2-bit, h = W/2, q = W/4: if kappa < 3h: word = 2 (kappa % h) + mu/2,
 *         slot = kappa/h + 5 (mu % 2); else k2 = kappa - 3h: word =
 *         4 (k2 % q) + mu, slot = 3 + k2/q.
 *       4-bit, h = W/2: word = 2 (kappa % h) + mu/2, slot = kappa/h + 2 (mu % 2).
 *     (Every class keeps one power-of-two factor through the draft kernel's
 *     shift-free unpacking; the kernel cancels it per channel.)
 *   K meta section (4d bytes): for lane quad j in [0,4) and k-step ks in
 *     [0, d/16), the 16 bytes at 16*(4 ks + j) hold, for rr = 0 then rr = 1,
 *     the fp16 zero-point pair (z[c0], z[c0+1]) and then the scale pair
 *     (s[c0], s[c0+1]), c0 = 16 ks + 2 j + 8 rr (zero pair at + 8 rr, scale
 *     pair at + 8 rr + 4): one 16-byte load is both the scales of a k-step and
 *     the operand of the draft kernel's zero-point MMA.
 *   V meta section (4d bytes): fp16 pair n of quad j at byte
 *     16*(4*(n/4) + j) + 4*(n%4), zero-point pair at the same offset + 2d;
 *     n = (2 ks + rr)*(d/32) + gc holds (s[t0][gc], s[t0+1][gc]),
 *     t0 = 16 ks + 2 j + 8 rr.
 * Rotated cache (rotate = 1; RotateKV, named among the compressors on the
 * paper page, "What the paper found"; the library's reading is a fixed
 * rotation, the pages describe no adaptive part): every key row x, quantized
 * or in the ring, is stored as res_dtype(W(x) * 2^-ceil(log2(d)/2)), W the
 * binary32 Walsh-Hadamard butterfly network (stages h = 1, 2, ..., d/2, the
 * pair (i, i + h), i mod 2h < h, becoming (a + b, a - b), each rounded to
 * binary32); vc_draft_attn applies W(q) * 2^-floor(log2(d)/2) to the queries,
 * so rotated dot products equal the plain ones.  Values are not rotated.
 * Appends and commits rotate the new key rows the same way.
 *
 * Full-precision tokens (positions n_groups[b]*group .. seq_len[b]-1) live in
 * a ring: position p of (b, h) at k_res/v_res + ((b * Hkv + h) * res_cap +
 * p % res_cap) * d elements.
 * Supported: bits in {2, 4}, group == 32, d in {64, 128}.
 */
typedef struct vc_quant_cfg {
    int32_t bits;        /* 2 or 4 */
    int32_t group;       /* 32 */
    int32_t residual;    /* R: tokens kept full precision (the newest R..R+group-1) */
    int32_t rotate;      /* 1: rotated cache (below), 0: plain */
} vc_quant_cfg;

typedef struct vc_qcache {
    void *records;        /* device, [B][Hkv][max_groups] records, 256-B aligned */
    void *k_res;          /* device, [B][Hkv][res_cap][d] in res_dtype */
    void *v_res;          /* device, same */
    int32_t *n_groups;    /* device [B]: quantized groups of sequence b */
    int32_t *seq_len;     /* device [B]: cached tokens of sequence b */
    int32_t *status;      /* device, 1 word: bits 0-1 set by a ring overflow, bit 2 by a
                             prefill staging wait that gave up (bounded, about 2 s) */
    int32_t B, Hkv, d;
    vc_quant_cfg cfg;
    int32_t max_groups;   /* record capacity per (b, h) */
    int32_t res_cap;      /* ring capacity per (b, h), >= cfg.residual + group */
    vc_dtype res_dtype;
} vc_qcache;

/* Bytes of one group record: 2*group*d*bits/8 + 8*d (group = 32). */
size_t vc_record_bytes(int bits, int d);

/*
 * vc_quantize_kv -- compress a prefill K/V cache into `cache`.
 * k, v: device [B][Hkv][L_stride][d] in dt (dt must equal cache->res_dtype);
 * tokens 0..L-1 are used.  With n_q = floor(max(L - R, 0) / group) groups,
 * writes records 0..n_q-1 of every (b, h), copies positions n_q*group..L-1
 * into the ring, and sets n_groups[b] = n_q, seq_len[b] = L.
 * Requires n_q <= max_groups and L - n_q*group <= res_cap.
 */
vc_status vc_quantize_kv(const void *k, const void *v, vc_dtype dt, int B, int Hkv,
                         int L, int L_stride, int d, vc_qcache *cache,
                         cudaStream_t stream);

/*
 * vc_qcache_append -- append new tokens to the cache (draft steps and the
 * commit after verification).
 * k_new, v_new: device [B][Hkv][max_new][d] in cache->res_dtype; sequence b
 * appends its first n_new[b] rows (device int32 [B], 0 <= n_new[b] <= max_new)
 * at positions seq_len[b].., then seq_len[b] += n_new[b].  With requantize != 0
 * every complete group that has left the residual window ((g+1)*group <=
 * seq_len[b] - R) is quantized into record g and n_groups[b] advances.  A
 * ring overflow (tokens that would overwrite unquantized ones) sets
 * *cache->status and drops the excess tokens.
 * Rolling back drafted tokens is a plain rewrite of seq_len by the caller.
 */
vc_status vc_qcache_append(vc_qcache *cache, const void *k_new, const void *v_new,
                           const int32_t *n_new, int max_new, int requantize,
                           cudaStream_t stream);

/*
 * vc_qcache_commit -- the end of a draft-and-verify round for the draft cache
 * (paper page: the drafted tokens are verified against the full cache; the
 * compressed cache then carries on from the verified output).  For every
 * sequence b: roll back to round_len[b] (the length before drafting), append
 * the first n_acc[b] + 1 rows of the verify block k_blk, v_blk (device
 * [B][Hkv][Dq][d] in cache->res_dtype: the verify pass's K/V of the pending
 * token and the accepted drafts), and re-quantize every group that left the
 * residual window.  round_len, n_acc: device int32 [B] (n_acc as written by
 * vc_accept, 0 <= n_acc[b] < Dq).
 */
vc_status vc_qcache_commit(vc_qcache *cache, const void *k_blk, const void *v_blk,
                           const int32_t *round_len, const int32_t *n_acc, int Dq,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (2) token-dropping compressor                                             */
/* ------------------------------------------------------------------------ */
/*
 * Token dropping by accumulated attention score (H2O, source 3 on the
 * podparley page; KVzip 4x on the paper page, "What the paper found"): per
 * (b, h) keep the `keep_recent` newest tokens and the `keep_top` best of the
 * older ones, ranked by score descending, ties by position ascending, and
 * compact them in ascending position order.
 */
typedef struct vc_drop_cfg {
    int64_t keep_top;
    int64_t keep_recent;
} vc_drop_cfg;

/* Kept tokens per (b, h): min(keep_top, max(L - R, 0)) + min(R, L). */
int64_t vc_drop_kept_count(int64_t L, vc_drop_cfg cfg);

size_t vc_drop_tokens_workspace_bytes(int B, int H, int L);

/*
 * scores: device fp32 [B][H][L] (finite); k, v: device [B][H][L][d] in dt.
 * kept_idx: device int32 [B][H][n_keep] (ascending positions);
 * k_out, v_out: device [B][H][n_keep][d] in dt, the gathered rows.
 * Selection and compaction are exact: kept_idx is unique for given scores.
 */
vc_status vc_drop_tokens(const float *scores, const void *k, const void *v, vc_dtype dt,
                         int B, int H, int L, int d, vc_drop_cfg cfg,
                         int32_t *kept_idx, void *k_out, void *v_out,
                         void *ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (3) draft decode attention over the compressed cache                      */
/* ------------------------------------------------------------------------ */
/*
 * Drafting runs the target model on the compressed cache (paper page, "What
 * the paper found"); this is its attention: one query per sequence and query
 * head, o = softmax(q K^T * sm_scale) V over every cached token, with query
 * head hq reading kv head hq / (Hq / Hkv).
 */
typedef enum vc_cache_kind {
    VC_CACHE_KIVI = 0,    /* quantized records + full-precision ring */
    VC_CACHE_DENSE = 1    /* plain K/V rows (a compacted dropped cache, or full) */
} vc_cache_kind;

typedef struct vc_cache_view {
    vc_cache_kind kind;
    const vc_qcache *kivi;       /* VC_CACHE_KIVI */
    const void *k, *v;           /* VC_CACHE_DENSE: device [B][Hkv][L_stride][d] */
    vc_dtype dt;                 /* VC_CACHE_DENSE element type */
    const int32_t *seq_len;      /* VC_CACHE_DENSE: device [B], tokens of sequence b */
    int32_t B, Hkv, d;           /* VC_CACHE_DENSE shape */
    int32_t L_stride;            /* VC_CACHE_DENSE row stride per (b, h) */
    int32_t max_len;             /* VC_CACHE_DENSE: upper bound of seq_len (grid sizing) */
    int32_t flags;               /* VC_VIEW_* bits; zero-initialise the view (0: none) */
} vc_cache_view;

/* VC_CACHE_KIVI: the caller guarantees that the kernel launched just before on
 * the stream writes neither the cache's records nor its n_groups (it may write
 * the ring and seq_len, as a draft step's RoPE does), so the draft kernel may
 * start copying records before that kernel has finished (programmatic
 * dependent launch).  Without the flag every read waits for it. */
#define VC_VIEW_RECORDS_STABLE 1

size_t vc_draft_attn_workspace_bytes(const vc_cache_view *view, int Hq);

/*
 * q: device [B][Hq][d] in q_dt; out: device [B][Hq][d] in q_dt.
 * Hq must be a multiple of Hkv with Hq / Hkv <= 8 (<= 4 for VC_CACHE_KIVI).
 * Sequences with no cached token produce zeros.
 */
vc_status vc_draft_attn(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq,
                        float sm_scale, void *out, void *ws, size_t ws_bytes,
                        cudaStream_t stream);

/*
 * vc_draft_attn_h2o -- vc_draft_attn over a dense bf16 view that also
 * accumulates attention scores for token dropping (H2O, source 3 on the
 * podparley page: tokens are ranked by the attention mass they have received
 * so far).  For kv unit u = b*Hkv + h and cached row j < seq_len[b]:
 *   scores[u * scores_stride + pos] += sum over the Hq/Hkv query heads of h
 *       of softmax_j(q . k_j * sm_scale),   pos = kept_idx ? kept_idx[u * kept_stride + j] : j
 * (kept_idx maps rows of a compacted cache back to original positions, as
 * vc_drop_tokens writes it).  The probabilities are those of this call's
 * attention: each head's scores are stored in fp32 and normalised by the
 * head's final max and sum after the split merge.  scores: device fp32, rows
 * of one unit distinct positions.  Workspace: vc_draft_attn_h2o_workspace_bytes
 * (the attention's plus 16 bytes per cached row).
 * Views: dense bf16 (q bf16), or KIVI (q bf16 or fp32; the mass of the
 * dequantized cache x^ and of the ring; kept_idx must be NULL, the rows being
 * the positions, and scores_stride >= max_groups * group + res_cap).
 * VC_ERR_UNSUPPORTED for dense fp32 views.
 */
size_t vc_draft_attn_h2o_workspace_bytes(const vc_cache_view *view, int Hq);
vc_status vc_draft_attn_h2o(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq, float sm_scale,
                            void *out, float *scores, int scores_stride, const int32_t *kept_idx, int kept_stride,
                            void *ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (4) verify attention over the full cache                                  */
/* ------------------------------------------------------------------------ */
/*
 * Verification re-runs the drafted block against the full KV cache (paper
 * page, "What the paper found"): a causal block of Dq queries.  Query i of
 * sequence b sits at position ctx_len[b] + i and attends keys
 * 0 .. ctx_len[b] + i; the block's own K/V must already be written at
 * positions ctx_len[b] .. ctx_len[b] + Dq - 1 of k, v.
 * q: device [B][Dq][Hq][d]; k, v: device [B][Hkv][L_stride][d];
 * out: device [B][Dq][Hq][d]; all in dt.  ctx_len: device int32 [B] with
 * ctx_len[b] + Dq <= L_stride and ctx_len[b] <= max_ctx.
 * bf16 with d = 128 and Hq / Hkv in {1, 2, 4, 8} runs on the tensor cores
 * (TMA + tcgen05, fp32 accumulation); other supported shapes (fp32, d = 64)
 * run an fp32 CUDA-core kernel.
 */
size_t vc_verify_attn_workspace_bytes(vc_dtype dt, int B, int Dq, int Hq, int Hkv, int d,
                                      int max_ctx);

vc_status vc_verify_attn(const void *q, const void *k, const void *v, vc_dtype dt,
                         const int32_t *ctx_len, int B, int Dq, int Hq, int Hkv, int d,
                         int L_stride, int max_ctx, float sm_scale, void *out,
                         void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * vc_verify_attn_h2o -- vc_verify_attn that also accumulates attention
 * scores for token dropping (H2O, source 3 on the podparley page: tokens are
 * ranked by the attention mass they have received).  For kv unit
 * u = b*Hkv + h and key j < ctx_len[b] + Dq:
 *   scores[u * scores_stride + j] += sum over the block's rows (query i,
 *       query head of h) with j <= ctx_len[b] + i of softmax_j(q . k_j * sm_scale)
 * The probabilities use each row's final max and sum from the verify pass;
 * a second pass over K recomputes the scores on the tensor cores.
 * Shapes: bf16, d = 128, Hq / Hkv in {1, 2, 4, 8}, Dq * Hq / Hkv <= 272;
 * VC_ERR_UNSUPPORTED otherwise.  scores: device fp32 with
 * scores_stride >= max_ctx + Dq.  Workspace: vc_verify_attn_h2o_workspace_bytes
 * (the verify pass's plus 8 bytes per row).
 */
size_t vc_verify_attn_h2o_workspace_bytes(int B, int Dq, int Hq, int Hkv, int d, int max_ctx);

vc_status vc_verify_attn_h2o(const void *q, const void *k, const void *v, const int32_t *ctx_len, int B,
                             int Dq, int Hq, int Hkv, int d, int L_stride, int max_ctx, float sm_scale,
                             void *out, float *scores, int scores_stride, void *ws, size_t ws_bytes,
                             cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (5) greedy acceptance                                                     */
/* ------------------------------------------------------------------------ */
/*
 * The greedy rule of speculative decoding (source 2 on the podparley page),
 * which makes the output identical to full-KV greedy decoding (paper page,
 * "What the paper found"): with a_i = argmax of verify logits row i (lowest
 * index on ties, -0 == +0), n = first i in [0, D) with a_i != drafts[i], else
 * D; next = a_n.  The round emits drafts[0..n-1] and next.
 * logits: device [B][D+1][V] in dt (finite values); drafts: device int32
 * [B][D]; n_acc, next_tok: device int32 [B].  Limits: D <= 1024 and
 * B * (D + 1) <= 65535 rows; larger requests return VC_ERR_INVALID and
 * enqueue nothing.  The workspace's per-sequence counters are left at zero
 * by every call, so a workspace zero-filled once serves any number of calls.
 */
size_t vc_accept_workspace_bytes(int B, int D, int V);

vc_status vc_accept(const void *logits, vc_dtype dt, const int32_t *drafts, int B, int D,
                    int V, int32_t *n_acc, int32_t *next_tok, void *ws, size_t ws_bytes,
                    cudaStream_t stream);

/*
 * vc_accept_tiles -- vc_accept from the tile maxima of the LM head's argmax
 * epilogue (vc_gemm_argmax) instead of the logits: row (b, i), i = 0..D, has
 * n_tiles entries tile_max[(b (D+1) + i) n_tiles + t] (the largest bf16 value
 * of columns 128 t .. 128 t + 127, as float) and tile_idx[...] (its lowest
 * column); the row's argmax is the largest value, the lowest column on ties,
 * exactly the argmax vc_accept takes over the bf16 logits.  Device buffers; no
 * workspace.  Same outputs as vc_accept.
 */
vc_status vc_accept_tiles(const float *tile_max, const int32_t *tile_idx, int n_tiles, const int32_t *drafts,
                          int B, int D, int32_t *n_acc, int32_t *next_tok, cudaStream_t stream);

/*
 * vc_accept_noalloc -- vc_accept for callers that cannot allocate device
 * memory (no counterpart in the paper: this is a library convenience).
 * Some callers have no way to provide the workspace vc_accept needs: code
 * running inside another framework that owns all device memory through its
 * own pool, plugin hosts that expose no allocator, and latency-critical loops
 * where cudaMalloc/cudaFree would synchronize the device.  This entry point
 * takes the same inputs and outputs as vc_accept and computes the same
 * results, but keeps its scratch in a static device buffer inside the library
 * (about 516 KiB, held by every GPU that loads the library until the process
 * exits); it calls no allocator.
 * Limits: B <= 1024 and B * (D + 1) <= 16384; larger requests return
 * VC_ERR_INVALID and enqueue nothing.
 * The first call on a device (made with that device current) looks up the
 * buffer's device address; make that first call before any stream capture.
 * The address belongs to the CUDA context the call ran in: after a
 * cudaDeviceReset, or when the caller switches to another context on the
 * same device, the next call looks it up again and must also be made outside
 * a stream capture.
 * All calls on one device share the buffer, so calls that may run
 * concurrently on the GPU (different streams without ordering) race and
 * must be serialized by the caller.  Each call clears the part of the buffer
 * that must start at zero; the rest keeps the previous call's contents.
 */
vc_status vc_accept_noalloc(const void *logits, vc_dtype dt, const int32_t *drafts, int B,
                            int D, int V, int32_t *n_acc, int32_t *next_tok,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (6) full-KV swap-in                                                       */
/* ------------------------------------------------------------------------ */
/*
 * The exact KV state lives in host memory between rounds and is brought in
 * for verification while drafting runs (abstract on the paper page; the
 * cross-resource staggering of "What the paper found").  Copies `bytes` from pinned host memory to the
 * device with one asynchronous copy on `side_stream` and, if `done` is not
 * NULL, records `done` on that stream after it; the caller makes the verify
 * stream wait on `done`.  Returns VC_ERR_INVALID if src is not page-locked
 * host memory (a pageable source would serialize the copy), or if the range
 * [src, src + bytes) or [dst, dst + bytes) does not end inside memory of its
 * kind (checked at its first and last byte).
 */
vc_status vc_swap_in(void *dst_dev, const void *src_pinned_host, size_t bytes,
                     cudaStream_t side_stream, cudaEvent_t done);

/*
 * vc_swap_in_rows -- vc_swap_in of the used prefix of a blocked cache: src and
 * dst hold `blocks` blocks of `pitch_rows` rows of `row_bytes` bytes each
 * ([blocks][pitch_rows][row_bytes], e.g. one layer's [B][Hkv][L_stride] rows);
 * the first `rows` rows of every block are copied by one 2-D asynchronous copy
 * on `side_stream` (a cache whose sequences hold at most `rows` tokens needs
 * nothing past them), then `done` is recorded as for vc_swap_in.  Returns
 * VC_ERR_INVALID if rows > pitch_rows, or if src is not page-locked host
 * memory or dst not device memory at the first and the last byte copied.
 */
vc_status vc_swap_in_rows(void *dst_dev, const void *src_pinned_host, size_t row_bytes, size_t rows,
                          size_t pitch_rows, size_t blocks, cudaStream_t side_stream, cudaEvent_t done);

/*
 * vc_swap_in_paced -- vc_swap_in as if the source produced data at `gbps`
 * (GB/s): the emulation of a full cache held by a slower store, e.g. a remote
 * prefix cache behind a network (paper page, "Key results": remote prefix
 * caching).  The copy is cut into chunks of chunk_bytes; chunk i starts no
 * earlier than i * chunk_bytes / gbps after the first, by a one-thread kernel
 * on side_stream that sleeps until that time (never more than 30 s).  The rate
 * is an upper bound: a link slower than gbps gives its own rate.  pace_ws:
 * 16 device bytes, 16-byte aligned, used by this call until `done`.
 */
vc_status vc_swap_in_paced(void *dst_dev, const void *src_pinned_host, size_t bytes, double gbps,
                           size_t chunk_bytes, void *pace_ws, cudaStream_t side_stream, cudaEvent_t done);

/*
 * Packed full cache for the host link.  The swap-in above is bound by the
 * link (paper page, "What the paper found": the exact KV state comes in over
 * the interconnect while drafting runs), so the host may hold the full cache
 * losslessly packed; it then moves 16 + 3d/2 bytes per row of d bf16 values
 * instead of 2d (208 instead of 256 at d = 128) and vc_kv_unpack restores
 * every bit on the GPU.  Packed row (d even):
 *   byte 0           base = E - 14, or 0 when E < 14, E = the row's largest
 *                    bf16 exponent field (bits 14..7)
 *   byte 1           n_esc in 0..7, or 255: the row needs more than 7
 *                    escapes and cannot be held (its other bytes are then
 *                    unspecified)
 *   bytes 2..15      7 escape slots (value index, exponent field), ascending
 *                    index order, unused slots zero
 *   16 .. 16 + d/2   4-bit codes: value i in the low nibble of byte i/2 for
 *                    even i, the high nibble for odd i; code = field - base
 *                    when that lies in 0..14, else 15 (the field is in a slot)
 *   last d bytes     sign << 7 | 7 mantissa bits of value i, in byte i
 * Rows are independent and 16-byte multiples, so a [B][Hkv][L][d] cache packs
 * to [B][Hkv][L][16 + 3d/2] and appended rows pack on their own.
 */
size_t vc_kv_packed_row_bytes(int d);   /* 16 + 3d/2 for d in {64, 128}, else 0 */

/*
 * Pack `rows` rows of d bf16 values.  src_bf16: device, [rows][d], 8-byte
 * aligned; dst_packed: device (or mapped pinned host), [rows][16 + 3d/2],
 * 16-byte aligned.  n_over: device int32 or NULL; the number of rows marked
 * 255 is added to it (a row so marked cannot be unpacked: keep the raw copy
 * for that cache).  VC_ERR_UNSUPPORTED for d outside {64, 128}.
 */
vc_status vc_kv_pack(const void *src_bf16, void *dst_packed, int64_t rows, int d, int32_t *n_over,
                     cudaStream_t stream);

/*
 * Unpack `rows` packed rows (none marked 255) into bf16.  src_packed: device,
 * 16-byte aligned; dst_bf16: device, [rows][d], 8-byte aligned.  Bit-exact
 * inverse of vc_kv_pack.
 */
vc_status vc_kv_unpack(const void *src_packed, void *dst_bf16, int64_t rows, int d, cudaStream_t stream);

/*
 * vc_kv_writeback_packed -- vc_kv_writeback for a packed host cache: the
 * committed rows (i <= n_acc[b]) of the verify block, every layer, K and V,
 * packed into k_host_packed / v_host_packed [n_layers][B][Hkv][L_stride]
 * [16 + 3d/2] at position ctx_len[b] + i.  k_blk, v_blk: device bf16
 * [n_layers][B][Hkv][Dq][d], 8-byte aligned; the host buffers pinned and
 * 16-byte aligned.  Rows that cannot be packed are counted in n_over (device
 * int32, or NULL) and marked: the caller must then stop using the packed copy.
 */
vc_status vc_kv_writeback_packed(const void *k_blk, const void *v_blk, int n_layers, int B, int Hkv, int Dq, int d,
                                 const int32_t *n_acc, const int32_t *ctx_len, void *k_host_packed,
                                 void *v_host_packed, int L_stride, int32_t *n_over, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* (7) target decoder around the hot path                                    */
/* ------------------------------------------------------------------------ */
/*
 * The pages run the method inside a trained LLM; the drafting and the
 * verification are forward passes of that one model (paper page, "What the
 * paper found": the target model drafts for itself).  This section is the
 * model around the six calls above: a Llama-style decoder (pre-RMSNorm with
 * unit weight, rotate-half RoPE applied to q and k before caching, grouped
 * query attention with q head h reading kv head h / (Hq/Hkv), SwiGLU MLP,
 * final RMSNorm, untied LM head, no biases).  Its attention is vc_draft_attn
 * over a vc_qcache (drafting) or vc_verify_attn over the full cache (verify,
 * prefill, plain decoding); its projections are the library's own GEMMs.
 *
 * Row independence: every kernel of a forward pass computes a token's row
 * with an operation order fixed by the model's shapes, the key positions and
 * the device, never by how many rows or sequences share the launch.  A verify
 * pass over [x, d1..dD] therefore gives, row for row and bit for bit, the
 * logits that D+1 one-token passes give, which makes draft-and-verify
 * decoding equal plain greedy decoding exactly (not only up to rounding).
 */
typedef struct vc_decoder_cfg {
    int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ff, vocab;
    float norm_eps;       /* RMSNorm epsilon */
    float rope_theta;     /* RoPE base */
    vc_dtype dt;          /* weights, activations, caches, logits */
} vc_decoder_cfg;

/* Device pointers, row-major, each matrix stored [in][out] (y = x W).  The
 * per-layer arrays are host arrays of n_layers device pointers; they are
 * copied by vc_decoder_create.  bf16 weights with N % 128 == 0 and K % 64 == 0
 * use the tensor-core GEMM; 16-byte aligned. */
typedef struct vc_decoder_weights {
    const void *embed;                /* [vocab][d_model] */
    const void *lm_head;              /* [d_model][vocab] */
    const void *const *w_qkv;         /* [d_model][(Hq + 2 Hkv) head_dim]: q | k | v columns */
    const void *const *w_o;           /* [Hq head_dim][d_model] */
    const void *const *w_gate_up;     /* [d_model][2 d_ff]: gate and up columns interleaved per 64
                                         (column 128 t + j is gate column 64 t + j, column 128 t + 64 + j
                                         up column 64 t + j), so that a 128-column GEMM tile holds the
                                         gate and up halves of 64 activations (d_ff % 64 == 0) */
    const void *const *w_down;        /* [d_ff][d_model] */
} vc_decoder_weights;

typedef struct vc_decoder vc_decoder;   /* host object: configuration + weight pointers */

/* Validate and record the model; no device memory is allocated.
 * Supported: head_dim in {64, 128}, n_heads % n_kv_heads == 0 with at most 4
 * q heads per kv head (the draft kernel), d_ff % 64 == 0, bf16 or fp32. */
vc_status vc_decoder_create(const vc_decoder_cfg *cfg, const vc_decoder_weights *w, vc_decoder **out);
void vc_decoder_destroy(vc_decoder *dec);

/*
 * Tracing (measurement aid): after vc_decoder_set_trace, the decoder records
 * events[2k] and events[2k+1] on the call's stream around its k-th operation
 * whose kind bit (1 << kind) is set in kind_mask, writes the kind to
 * kinds[k], and stops recording once `capacity` operations are traced.  The
 * arrays are caller-owned (events created by the caller); capacity 0 turns
 * tracing off.  Tracing mutates the decoder object: traced calls must not run
 * concurrently on one vc_decoder.  A GEMM operation includes its split-K
 * reduction.  Calls enqueued while their stream is being captured into a
 * CUDA graph put the events into the graph as external event-record nodes:
 * they are recorded each time the graph is replayed.
 */
typedef enum vc_trace_kind {
    VC_TRACE_GEMM_QKV = 0, VC_TRACE_GEMM_O = 1, VC_TRACE_GEMM_GATE_UP = 2, VC_TRACE_GEMM_DOWN = 3,
    VC_TRACE_GEMM_HEAD = 4, VC_TRACE_DRAFT_ATTN = 5, VC_TRACE_VERIFY_ATTN = 6
} vc_trace_kind;
vc_status vc_decoder_set_trace(vc_decoder *dec, cudaEvent_t *events, int32_t *kinds, int capacity, int kind_mask);
int vc_decoder_trace_count(const vc_decoder *dec);

/*
 * Per-layer arrival of a full cache that is being copied in (the swap-in
 * overlapped with the rest of the round, paper page "What the paper found"):
 * after vc_decoder_set_layer_events(dec, events, n_layers), vc_decoder_forward
 * and vc_decoder_verify make their stream wait on events[l]
 * (cudaStreamWaitEvent) before their first access to layer l of k_cache and
 * v_cache, so layer l's work starts once that layer is resident instead of
 * once the whole cache is.  The caller records events[l] on the copying
 * stream after layer l's copy (and expansion) is enqueued, before it enqueues
 * the forward; an event never recorded is no wait.  The handles are copied
 * (the caller owns the events and keeps them alive while set); n = 0 clears
 * them.  Like tracing, this mutates the decoder object: a change of the
 * events must not race with another host thread's call on the same
 * vc_decoder.  Not for calls enqueued while their stream is being captured.
 * Errors: VC_ERR_INVALID for dec NULL, n < 0, or n > 0 with events NULL, a
 * NULL handle or n != n_layers.
 */
vc_status vc_decoder_set_layer_events(vc_decoder *dec, const cudaEvent_t *events, int n);

/* Workspace for calls with up to B sequences of up to max_rows rows each and
 * contexts up to max_ctx tokens; draft_cache (may be NULL when only
 * vc_decoder_forward is used) is a cache of the geometry later passed to
 * vc_decoder_draft_step.  Zero-fill once (vc_workspace_init); the status
 * block of every kernel the decoder launches is folded into its first word
 * (vc_poll_status). */
size_t vc_decoder_workspace_bytes(const vc_decoder *dec, int B, int max_rows, int max_ctx,
                                  const vc_qcache *draft_cache);

/*
 * vc_decoder_forward -- causal forward of Dq tokens per sequence against the
 * full KV cache: prefill (ctx_len = 0 or a chunk start), the verify pass
 * (paper page: the drafted block checked against the full cache) and plain
 * one-token decoding (Dq = 1).
 * Tokens: row (b, i) takes first_tok[b] for i = 0 when first_tok is not
 * NULL, else tokens[b * tok_stride + i - (first_tok ? 1 : 0)] (device int32).
 * Row (b, i) sits at position ctx_len[b] + i (device int32 [B], every value
 * <= max_ctx).  k_cache, v_cache: device [n_layers][B][Hkv][L_stride][head_dim]
 * (L_stride >= max_ctx + Dq); the pass writes its own K/V at those positions
 * and, when k_blk/v_blk are not NULL, also to [n_layers][B][Hkv][Dq][head_dim]
 * (the rows vc_qcache_commit consumes).  logits: device [B][Dq][vocab], or
 * [B][vocab] for row Dq-1 only when logits_last_only != 0.
 * Token ids outside [0, vocab) read row 0 and set the status block.
 */
vc_status vc_decoder_forward(const vc_decoder *dec, const int32_t *first_tok, const int32_t *tokens,
                             int tok_stride, int B, int Dq, const int32_t *ctx_len, int max_ctx,
                             void *k_cache, void *v_cache, int L_stride, void *k_blk, void *v_blk,
                             int logits_last_only, void *logits, void *ws, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * vc_decoder_verify -- the verify pass and greedy acceptance in one call,
 * without logits: the forward of [first_tok[b], drafts[b][0..D-1]] at
 * positions ctx_len[b] .. ctx_len[b] + D over the full cache (as
 * vc_decoder_forward with tokens = drafts, tok_stride = D), the LM head with
 * the argmax epilogue, then vc_accept_tiles: n_acc[b], next_tok[b] are those
 * vc_accept gives on the logits vc_decoder_forward would write.  D in
 * [0, 1024]; workspace from vc_decoder_workspace_bytes with max_rows >= D + 1.
 */
vc_status vc_decoder_verify(const vc_decoder *dec, const int32_t *first_tok, const int32_t *drafts, int D, int B,
                            const int32_t *ctx_len, int max_ctx, void *k_cache, void *v_cache, int L_stride,
                            void *k_blk, void *v_blk, int32_t *n_acc, int32_t *next_tok, void *ws, size_t ws_bytes,
                            cudaStream_t stream);

/*
 * vc_decoder_draft_step -- one draft step on the compressed caches (one
 * vc_qcache per layer, host array of n_layers, all of one geometry): token
 * tok[b] sits at position caches[l].seq_len[b]; its K/V are appended to every
 * layer's ring (no re-quantization: drafted tokens are rolled back by
 * vc_qcache_commit), attention is vc_draft_attn over the cache, and the
 * greedy draft token argmax(logits[b]) (lowest index on ties) is written to
 * next_tok[b] and, when drafts_out is not NULL, to drafts_out[b * drafts_stride].
 * logits: device [B][vocab] (written), or NULL: the LM head then runs with the
 * argmax epilogue and no logits are written (same next_tok).
 */
vc_status vc_decoder_draft_step(const vc_decoder *dec, const int32_t *tok, int B, vc_qcache *caches,
                                void *logits, int32_t *next_tok, int32_t *drafts_out, int drafts_stride,
                                void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * vc_kv_writeback -- after acceptance, store the verify pass's K/V of the
 * n_acc[b] + 1 committed rows of every layer into the host-resident full cache
 * (pinned memory, written directly by the GPU): row i of sequence b goes to
 * position ctx_len[b] + i.  k_blk, v_blk: device [n_layers][B][Hkv][Dq][d];
 * k_host, v_host: pinned [n_layers][B][Hkv][L_stride][d]; dt of both.
 * Returns VC_ERR_INVALID if the host buffers are not page-locked.
 */
vc_status vc_kv_writeback(const void *k_blk, const void *v_blk, vc_dtype dt, int n_layers, int B, int Hkv,
                          int Dq, int d, const int32_t *n_acc, const int32_t *ctx_len, void *k_host,
                          void *v_host, int L_stride, cudaStream_t stream);

/*
 * vc_gemm -- out = x W (+ resid) with the decoder's GEMM: x [M][K], W [K][N],
 * resid and out [M][N] (resid may equal out), dt for all; fp32 accumulation.
 * The summation order of every output element depends on (N, K), the plan and
 * the device only.  ws: vc_gemm_workspace_bytes(dt, M, N, K) bytes (may be 0),
 * zero-filled once before first use (it holds per-tile counters that every
 * call leaves at zero).
 */
size_t vc_gemm_workspace_bytes(vc_dtype dt, int M, int N, int K);
/* Number of K splits of the decoder's GEMM for (N, K): decode_plan != 0 gives
 * the plan of vc_decoder_draft_step (M <= 128, chosen to fill whole waves),
 * 0 the row-invariant plan of vc_gemm and vc_decoder_forward.  0 on bad input. */
int vc_gemm_splits(vc_dtype dt, int N, int K, int decode_plan);
vc_status vc_gemm(const void *x, const void *w, const void *resid, void *out, vc_dtype dt, int M, int N, int K,
                  void *ws, size_t ws_bytes, cudaStream_t stream);
/*
 * vc_gemm_argmax -- the LM head of greedy decoding with an argmax epilogue:
 * the product x W (bf16, N a multiple of 128, K of 64) is rounded to bf16
 * element by element exactly as vc_gemm_ex with the same plan would store it,
 * and every (row m, tile t of 128 columns) yields tile_max[m (N/128) + t] and
 * tile_idx[...], the value and lowest column of the tile's maximum; the
 * product itself is never written (paper page, "What the paper found": only
 * the greedy token of each verify row is needed).  ws as for vc_gemm.
 * VC_ERR_UNSUPPORTED for other shapes or types.
 */
vc_status vc_gemm_argmax(const void *x, const void *w, vc_dtype dt, int M, int N, int K, int decode_plan,
                         float *tile_max, int32_t *tile_idx, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * vc_gemm_swiglu -- the decoder's gate|up projection with its SwiGLU in the
 * GEMM epilogue: with g, u the bf16-rounded products x W of a gate column and
 * its up column (w_gate_up [K][2F] in the decoder's interleaved layout, see
 * vc_decoder_weights), act [M][F] (row-major) receives bf16(g / (1 + exp(-g))
 * * u), the value a separate pass over the stored bf16 product gives.  For
 * bf16 products the plan (decode_plan as for vc_gemm_ex) leaves unsplit,
 * F % 64 == 0, K % 64 == 0; VC_ERR_UNSUPPORTED otherwise.  No workspace.
 */
vc_status vc_gemm_swiglu(const void *x, const void *w_gate_up, void *act, vc_dtype dt, int M, int F, int K,
                         int decode_plan, cudaStream_t stream);

/*
 * vc_gemm_rms -- the draft-step product of RMS-normalised rows, as the
 * decoder's draft steps compute it: out = rmsnorm(x) W with rmsnorm(x)[m] =
 * x[m] / sqrt(mean_k x[m][k]^2 + eps) (no gain), x [M][K], W [K][N], out
 * [M][N]; or with swiglu != 0 the SwiGLU of that product (W [K][N] in the
 * interleaved gate|up layout of vc_decoder_weights, out = act [M][N/2]).  The
 * GEMM reads x itself and scales each output row by 1 / sqrt(mean x^2 + eps)
 * in its epilogue (fp32), so the result is within fp32 rounding of the
 * two-pass product, not bit-identical to it.  bf16, 1 <= M <= 16, K % 64 == 0,
 * N % 128 == 0 (swiglu: the unsplit products of vc_gemm_swiglu);
 * VC_ERR_UNSUPPORTED otherwise.  ws as for vc_gemm (the decode plan).
 */
vc_status vc_gemm_rms(const void *x, const void *w, void *out, vc_dtype dt, int M, int N, int K, float eps, int swiglu,
                      void *ws, size_t ws_bytes, cudaStream_t stream);

/* vc_gemm with the split plan chosen explicitly: decode_plan != 0 runs the plan
 * of vc_decoder_draft_step (for M <= 16 it loads only 16 rows of x per K slice
 * and keeps six slices of W in flight); 0 is vc_gemm.  The workspace size from
 * vc_gemm_workspace_bytes covers both plans. */
vc_status vc_gemm_ex(const void *x, const void *w, const void *resid, void *out, vc_dtype dt, int M, int N, int K,
                     int decode_plan, void *ws, size_t ws_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VC_H */
