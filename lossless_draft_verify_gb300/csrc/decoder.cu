// decoder.cu -- the target model around the draft-and-verify hot path: token
// embedding, RMSNorm, RoPE with the K/V scatter into the caches, SwiGLU, the
// LM head, and the host-side sequencing of one forward pass (prefill, verify
// block, plain decoding) or one draft step (paper page, "What the paper
// found": the target model drafts on its compressed cache and verifies on the
// full one).
//
// Every kernel here keeps a row's arithmetic independent of the other rows
// of the launch (one CTA per row where a row reduces; fixed reduction trees),
// and so do the GEMMs (gemm.cu) and the fixed-split verify attention.  A
// verify pass therefore reproduces one-token decoding bit for bit.
#include <cuda.h>

#include <algorithm>
#include <new>
#include <cmath>
#include <vector>

#include "vc_common.cuh"
#include "vc_internal.h"

struct RopeFreq {
    double inv_freq[64];          // theta^(-2j / head_dim), j < head_dim / 2
};

struct vc_decoder {
    vc_decoder_cfg c;
    RopeFreq rope;
    const void *embed, *head;
    std::vector<const void *> wqkv, wo, wgu, wd;
    // optional trace: event pairs around selected operations (caller-owned)
    mutable cudaEvent_t *tr_ev = nullptr;
    mutable int32_t *tr_kind = nullptr;
    mutable int tr_cap = 0, tr_n = 0, tr_mask = 0;
    // optional: one event per layer, recorded when that layer's full cache is
    // resident; a forward waits on event l before it touches layer l's cache
    std::vector<cudaEvent_t> layer_ev;
};

namespace vc {
namespace {

// Verify attention inside the decoder uses key splits of a fixed 4096 keys.
constexpr int kSplitTiles = 64;
constexpr int kRowThreads = 256;
constexpr int kBadToken = 1 << 1;       // status bit: a token id outside [0, vocab)
constexpr int kBadPosition = 1 << 2;    // status bit: a position outside the cache

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }
int rope_blocks(const vc_decoder_cfg &c) { return (c.n_heads + 2 * c.n_kv_heads + 3) / 4; }
size_t esize(vc_dtype dt) { return dt == VC_BF16 ? 2 : 4; }

// ------------------------------------------------------------------ kernels --
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
embed_kernel(const int32_t *__restrict__ first_tok, const int32_t *__restrict__ toks, int tok_stride,
             int rows_per_seq, const T *__restrict__ E, int vocab, int D, T *__restrict__ x, int32_t *status,
             uint32_t *z0 = nullptr, int z0_words = 0, uint32_t *z1 = nullptr, int z1_words = 0)
{
    pdl_wait();
    pdl_trigger();
    // a draft step's scratch words that later kernels of the step expect at
    // zero (draft attention's status and arrival counters, RoPE's arrivals)
    if (blockIdx.x == 0) {
        for (int j = threadIdx.x; j < z0_words; j += kRowThreads) z0[j] = 0u;
        for (int j = threadIdx.x; j < z1_words; j += kRowThreads) z1[j] = 0u;
    }
    const int m = blockIdx.x;
    const int b = m / rows_per_seq, i = m % rows_per_seq;
    int t;
    if (first_tok)
        t = i == 0 ? first_tok[b] : toks[(size_t)b * tok_stride + i - 1];
    else
        t = toks[(size_t)b * tok_stride + i];
    if (t < 0 || t >= vocab) {
        if (threadIdx.x == 0) atomicOr(status, kBadToken);
        t = 0;
    }
    const T *src = E + (size_t)t * D;
    T *dst = x + (size_t)m * D;
    for (int j = threadIdx.x; j < D; j += kRowThreads) dst[j] = src[j];
}

// y[r] = x[r*in_step + in_off] / sqrt(mean(x^2) + eps): one CTA per row, the
// sum of squares over a fixed thread/warp tree.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
rmsnorm_kernel(const T *__restrict__ x, int D, int in_step, int in_off, float eps, T *__restrict__ y)
{
    pdl_wait();
    pdl_trigger();
    __shared__ float wsum[kRowThreads / 32];
    const int r = blockIdx.x;
    const T *xr = x + ((size_t)r * in_step + in_off) * D;
    float ss = 0.f;
    for (int j = threadIdx.x; j < D; j += kRowThreads) {
        const float v = Elem<T>::to_f(xr[j]);
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kRowThreads / 32; ++w) tot += wsum[w];
    const float inv = 1.0f / sqrtf(tot / (float)D + eps);
    T *yr = y + (size_t)r * D;
    for (int j = threadIdx.x; j < D; j += kRowThreads) yr[j] = Elem<T>::from_f(Elem<T>::to_f(xr[j]) * inv);
}

// RoPE (rotate-half: pair (j, j + hd/2) turned by pos * theta^(-2j/hd)) on the
// q and k parts of one qkv row, q to q_out, k and v scattered to up to two
// destinations [.][Hkv][stride][hd]: dst1 at row (pos1 ? pos : 0) + i (the
// cache), dst2 at row i (the block copy).  Angles in fp64 (positions reach
// 10^5 radians), reduced modulo 2 pi in fp64, cos/sin in fp32.
struct RopeDst {
    void *k1, *v1;
    size_t bstride1;   // elements between sequences
    int stride1, pos1; // rows per (sequence, head); row = pos when pos1 else i
    void *k2, *v2;
    size_t bstride2;
    int stride2;
    // Draft steps (one row per sequence): the new K and V rows go straight
    // into the compressed cache's ring of unquantized tokens at slot
    // pos % res_cap, and the last CTA of a sequence advances its length, as
    // the ring append would (no rotation, no re-quantization).  kr null: off.
    void *kr, *vr;     // [B][Hkv][res_cap][hd]
    int res_cap;
    int32_t *len, *ngroups, *qstatus;   // the cache's seq_len, n_groups, status
    unsigned int *arrive;               // [B] CTA arrivals, zero between launches
};
constexpr int kQGroup = 32;   // tokens per quantized group of the compressed cache

// One CTA per (row, block of kRopeHeads heads of q|k|v), one thread per
// rotated pair (j, j + hd/2).  The inverse frequencies are fp64 (tabulated
// once per decoder); the angle pos * inv_freq is formed and reduced modulo
// 2 pi in fp64 (positions reach 10^5 radians), then cos/sin of the small
// remainder in fp32.
constexpr int kRopeHeads = 4;

template <typename T>
__global__ void __launch_bounds__(kRopeHeads * 64)
rope_kernel(const T *__restrict__ qkv, int rows_per_seq, int Hq, int Hkv, int hd, const int32_t *__restrict__ pos_base,
            RopeFreq fr, T *__restrict__ q_out, RopeDst dst, int32_t *status)
{
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x;
    const int b = m / rows_per_seq, i = m % rows_per_seq;
    // the position is read once per CTA: in ring mode the sequence's last CTA
    // to arrive advances the length that pos_base points to
    __shared__ int s_pos;
    if (threadIdx.x == 0) s_pos = pos_base[b] + i;
    __syncthreads();
    const int pos = s_pos;
    const int half = hd / 2;
    bool ring_ok = false;
    if (dst.kr) {
        const int unq = pos - dst.ngroups[b] * kQGroup;   // unquantized tokens before this one
        ring_ok = unq >= 0 && unq < dst.res_cap;
        if (threadIdx.x == 0) {
            if (blockIdx.y == 0 && !ring_ok) atomicOr(dst.qstatus, unq < 0 ? 2 : 1);
            if (atomicAdd(&dst.arrive[b], 1u) == gridDim.y - 1) {
                if (ring_ok) dst.len[b] = pos + 1;
                dst.arrive[b] = 0u;
            }
        }
    }
    const int row1 = dst.pos1 ? pos : i;
    if (row1 < 0 || row1 >= dst.stride1) {
        // a position outside the cache: record it, write nothing
        if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(status, kBadPosition);
        return;
    }
    const int hh = blockIdx.y * kRopeHeads + threadIdx.x / half;   // head among q | k | v
    const int j = threadIdx.x % half;
    if (threadIdx.x >= kRopeHeads * half || hh >= Hq + 2 * Hkv) return;
    const T *row = qkv + (size_t)m * (Hq + 2 * Hkv) * hd;
    const T *src = row + (size_t)hh * hd;
    if (hh >= Hq + Hkv) {
        // v: copied into the cache (and the block copy)
        const int h = hh - Hq - Hkv;
        const T v0 = src[j], v1 = src[j + half];
        if (dst.kr) {
            if (ring_ok) {
                T *r = (T *)dst.vr + (((size_t)b * Hkv + h) * dst.res_cap + pos % dst.res_cap) * hd;
                r[j] = v0;
                r[j + half] = v1;
            }
            return;
        }
        T *d1 = (T *)dst.v1 + b * dst.bstride1 + ((size_t)h * dst.stride1 + row1) * hd;
        d1[j] = v0;
        d1[j + half] = v1;
        if (dst.v2) {
            T *d2 = (T *)dst.v2 + b * dst.bstride2 + ((size_t)h * dst.stride2 + i) * hd;
            d2[j] = v0;
            d2[j + half] = v1;
        }
        return;
    }
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    const double ang = (double)pos * fr.inv_freq[j];
    const double red = fma(-rint(ang * (1.0 / kTwoPi)), kTwoPi, ang);
    float sn, cs;
    sincosf((float)red, &sn, &cs);
    const float x1 = Elem<T>::to_f(src[j]), x2 = Elem<T>::to_f(src[j + half]);
    const T y1 = Elem<T>::from_f(x1 * cs - x2 * sn);
    const T y2 = Elem<T>::from_f(x2 * cs + x1 * sn);
    if (hh < Hq) {
        T *qo = q_out + (size_t)m * Hq * hd + (size_t)hh * hd;
        qo[j] = y1;
        qo[j + half] = y2;
    } else if (dst.kr) {
        if (ring_ok) {
            T *r = (T *)dst.kr + (((size_t)b * Hkv + (hh - Hq)) * dst.res_cap + pos % dst.res_cap) * hd;
            r[j] = y1;
            r[j + half] = y2;
        }
    } else {
        const int h = hh - Hq;
        T *k1 = (T *)dst.k1 + b * dst.bstride1 + ((size_t)h * dst.stride1 + row1) * hd;
        k1[j] = y1;
        k1[j + half] = y2;
        if (dst.k2) {
            T *k2 = (T *)dst.k2 + b * dst.bstride2 + ((size_t)h * dst.stride2 + i) * hd;
            k2[j] = y1;
            k2[j + half] = y2;
        }
    }
}

// act = silu(gate) * up from a [M][2F] row whose columns hold gate and up
// interleaved per 64 (columns 128 t + j: gate 64 t + j; 128 t + 64 + j: up
// 64 t + j), the layout of the decoder's gate|up weight.
template <typename T>
__global__ void silu_mul_kernel(const T *__restrict__ gu, int M, int F, T *__restrict__ act)
{
    pdl_wait();
    pdl_trigger();
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)M * F) return;
    const size_t m = idx / F, j = idx % F;
    const size_t gc = (j / 64) * 128 + j % 64;
    const float g = Elem<T>::to_f(gu[m * 2 * F + gc]);
    const float u = Elem<T>::to_f(gu[m * 2 * F + gc + 64]);
    act[idx] = Elem<T>::from_f((g / (1.0f + expf(-g))) * u);
}

__global__ void scatter_tokens_kernel(const int32_t *__restrict__ src, int B, int32_t *dst, int stride)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) dst[(size_t)b * stride] = src[b];
}

// OR the status words of the sub-workspaces into the decoder's, clear them.
__global__ void fold_status_kernel(int32_t *main, int32_t *a, int32_t *b, int32_t *c)
{
    pdl_wait();
    pdl_trigger();
    int32_t v = 0;
    if (a) { v |= *a; *a = 0; }
    if (b) { v |= *b; *b = 0; }
    if (c) { v |= *c; *c = 0; }
    if (v) atomicOr(main, v);
}

// One CTA per (row i, sequence-head bh, layer); rows i <= n_acc[b] copied.
template <typename T>
__global__ void writeback_kernel(const T *__restrict__ kb, const T *__restrict__ vb, int B, int Hkv, int Dq, int d,
                                 const int32_t *__restrict__ n_acc, const int32_t *__restrict__ ctx, T *kh, T *vh,
                                 int L_stride)
{
    const int i = blockIdx.x, bh = blockIdx.y, layer = blockIdx.z;
    const int b = bh / Hkv;
    if (i > n_acc[b] || ctx[b] + i >= L_stride) return;
    const size_t src = (((size_t)layer * B * Hkv + bh) * Dq + i) * d;
    const size_t dst = (((size_t)layer * B * Hkv + bh) * L_stride + ctx[b] + i) * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        kh[dst + c] = kb[src + c];
        vh[dst + c] = vb[src + c];
    }
}

// ------------------------------------------------------------------ layout --
struct Layout {
    size_t x, h, qkv, q, att, gu, act, kvn, hl, part, dws, vws, aws, nacc, tmax, tidx, lsc, rarr, total;
    bool fused_head;      // LM head with the argmax epilogue (else logits staged in lsc)
};

Layout layout_of(const vc_decoder *d, int B, int max_rows, int max_ctx, size_t draft_ws)
{
    const vc_decoder_cfg &c = d->c;
    const size_t es = esize(c.dt);
    const size_t M = (size_t)B * max_rows;
    const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
    const int nqkv = qd + 2 * kvd;
    Layout L;
    size_t o = kStatusBytes + kGemmCounterBytes;   // GEMM tile counters: same place in every call
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += a256(bytes);
        return at;
    };
    L.x = take(M * c.d_model * es);
    L.h = take(M * c.d_model * es);
    L.qkv = take(M * nqkv * es);
    L.q = take(M * qd * es);
    L.att = take(M * qd * es);
    L.gu = take(M * 2 * (size_t)c.d_ff * es);
    L.act = take(M * (size_t)c.d_ff * es);
    L.kvn = take(2 * (size_t)B * kvd * es);
    L.hl = take((size_t)B * c.d_model * es);
    size_t part = 0;
    auto gp = [&](int rows, int N, int K) {
        part = std::max(part, gemm_ws_bytes(c.dt, rows, N, K, kGemmRowInvariant));
        part = std::max(part, gemm_ws_bytes(c.dt, std::min(rows, B), N, K, kGemmDecode));
    };
    gp((int)M, nqkv, c.d_model);
    gp((int)M, c.d_model, qd);
    gp((int)M, 2 * c.d_ff, c.d_model);
    gp((int)M, c.d_model, c.d_ff);
    gp((int)M, c.vocab, c.d_model);
    L.part = take(part);
    L.dws = take(draft_ws);
    L.vws = take(verify_ws_bytes(c.dt, B, max_rows, c.n_heads, c.n_kv_heads, c.head_dim, max_ctx, kSplitTiles));
    L.aws = take(accept_ws_bytes(B, max_rows - 1, c.vocab));
    L.nacc = take((size_t)B * 4);
    // greedy heads without a logits output: tile maxima of the argmax
    // epilogue, or (no tensor-core head for this shape) staged logits
    L.fused_head = gemm_argmax_ok(c.dt, (int)M, c.vocab, c.d_model, kGemmRowInvariant, true) &&
                   gemm_argmax_ok(c.dt, B, c.vocab, c.d_model, kGemmDecode, true);
    const size_t nt = c.vocab / kGemmTileN;
    L.tmax = take(L.fused_head ? M * nt * 4 : 0);
    L.tidx = take(L.fused_head ? M * nt * 4 : 0);
    L.lsc = take(L.fused_head ? 0 : M * (size_t)c.vocab * es);
    L.rarr = take((size_t)B * 4);         // RoPE's per-sequence arrivals in draft steps
    L.total = o;
    return L;
}

size_t draft_ws_of(const vc_decoder *d, const vc_qcache *cache)
{
    if (!cache) return 0;
    vc_cache_view v{};
    v.kind = VC_CACHE_KIVI;
    v.kivi = const_cast<vc_qcache *>(cache);
    return draft_ws_bytes(&v, d->c.n_heads);
}

// ------------------------------------------------------------ sequencing --
struct Ctx {
    const vc_decoder *d;
    uint8_t *ws;
    Layout L;
    cudaStream_t st;
    int plan;          // GEMM split plan: row-invariant (forward) or decode (draft), + kGemmEarlyWeights
    int32_t *status() const { return (int32_t *)ws; }
    unsigned int *counters() const { return (unsigned int *)(ws + kStatusBytes); }
    template <typename P = void> P *at(size_t off) const { return reinterpret_cast<P *>(ws + off); }
};

// A trace event on the call's stream.  While the stream is being captured
// into a CUDA graph the event becomes an event-record node of the graph
// (external), so it is recorded each time the graph is replayed.
inline void trace_record(cudaEvent_t ev, cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, st);
}

// Record the trace events around op() when its kind is selected.
template <typename F>
cudaError_t traced(const Ctx &C, int kind, F &&op)
{
    const vc_decoder *d = C.d;
    const bool on = d->tr_ev && (d->tr_mask & (1 << kind)) && d->tr_n < d->tr_cap;
    if (on) trace_record(d->tr_ev[2 * d->tr_n], C.st);
    const cudaError_t e = op();
    if (on) {
        trace_record(d->tr_ev[2 * d->tr_n + 1], C.st);
        d->tr_kind[d->tr_n] = kind;
        ++d->tr_n;
    }
    return e;
}

#define VC_TRY(expr)                                \
    do {                                            \
        cudaError_t e_ = (expr);                    \
        if (e_ != cudaSuccess) return e_;           \
    } while (0)

template <typename T>
cudaError_t rmsnorm(const Ctx &C, const void *x, int rows, int in_step, int in_off, void *y)
{
    return launch_pdl(rmsnorm_kernel<T>, dim3(rows), dim3(kRowThreads), 0, C.st, (const T *)x, C.d->c.d_model,
                      in_step, in_off, C.d->c.norm_eps, (T *)y);
}

// The MLP and attention-output half of a layer, shared by both passes:
// x += att Wo; x += silu(x' Wg) (x' Wu) Wd with x' = rmsnorm(x).  In draft
// steps the gate|up GEMM takes x itself and scales its rows by 1 / rms (no
// separate normalisation launch); forward passes keep the separate RMSNorm, so
// a block's rows take the arithmetic of one-token forwards.
template <typename T>
cudaError_t layer_tail(const Ctx &C, int l, int M)
{
    const vc_decoder_cfg &c = C.d->c;
    const int qd = c.n_heads * c.head_dim;
    void *x = C.at(C.L.x), *h = C.at(C.L.h), *part = C.at(C.L.part);
    VC_TRY(traced(C, VC_TRACE_GEMM_O, [&] {
        return gemm(C.at(C.L.att), C.d->wo[l], x, x, c.dt, M, c.d_model, qd, qd, part, C.counters(), C.status(),
                    C.st, C.plan);
    }));
    if (gemm_swiglu_ok(c.dt, c.d_ff, c.d_model, C.plan) &&
        gemm_rms_ok(c.dt, M, 2 * c.d_ff, c.d_model, c.d_model, C.plan)) {
        VC_TRY(traced(C, VC_TRACE_GEMM_GATE_UP, [&] {
            return gemm_swiglu(x, C.d->wgu[l], C.at(C.L.act), c.dt, M, c.d_ff, c.d_model, c.d_model, C.status(),
                               C.st, C.plan, c.norm_eps);
        }));
    } else if (gemm_swiglu_ok(c.dt, c.d_ff, c.d_model, C.plan)) {
        VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
        // gate|up product and SwiGLU in one launch (the tensor-core epilogue)
        VC_TRY(traced(C, VC_TRACE_GEMM_GATE_UP, [&] {
            return gemm_swiglu(h, C.d->wgu[l], C.at(C.L.act), c.dt, M, c.d_ff, c.d_model, c.d_model, C.status(),
                               C.st, C.plan);
        }));
    } else {
        VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
        VC_TRY(traced(C, VC_TRACE_GEMM_GATE_UP, [&] {
            return gemm(h, C.d->wgu[l], nullptr, C.at(C.L.gu), c.dt, M, 2 * c.d_ff, c.d_model, c.d_model, part,
                        C.counters(), C.status(), C.st, C.plan);
        }));
        const size_t n = (size_t)M * c.d_ff;
        VC_TRY(launch_pdl(silu_mul_kernel<T>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, C.st,
                          C.at<const T>(C.L.gu), M, c.d_ff, C.at<T>(C.L.act)));
    }
    return traced(C, VC_TRACE_GEMM_DOWN, [&] {
        return gemm(C.at(C.L.act), C.d->wd[l], x, x, c.dt, M, c.d_model, c.d_ff, c.d_ff, part, C.counters(),
                    C.status(), C.st, C.plan);
    });
}

// The LM head of greedy decoding without a logits output: argmax epilogue and
// acceptance over the tile maxima, or (no tensor-core head) staged logits and
// the logits scan.  Rows [B][D+1]; drafts [B][D] (null for D = 0).  rms_eps
// >= 0: h is the raw residual stream, normalised inside the head's GEMM.
cudaError_t greedy_head(const Ctx &C, const void *h, int B, int D, const int32_t *drafts, int32_t *n_acc,
                        int32_t *next_tok, float rms_eps = -1.f)
{
    const vc_decoder_cfg &c = C.d->c;
    const int M = B * (D + 1);
    if (C.L.fused_head) {
        const int nt = c.vocab / kGemmTileN;
        VC_TRY(traced(C, VC_TRACE_GEMM_HEAD, [&] {
            return gemm(h, C.d->head, nullptr, nullptr, c.dt, M, c.vocab, c.d_model, c.d_model, C.at(C.L.part),
                        C.counters(), C.status(), C.st, C.plan, C.at<float>(C.L.tmax), C.at<int32_t>(C.L.tidx),
                        rms_eps);
        }));
        return accept_tiles(C.at<float>(C.L.tmax), C.at<int32_t>(C.L.tidx), nt, drafts, B, D, n_acc, next_tok, C.st);
    }
    VC_TRY(traced(C, VC_TRACE_GEMM_HEAD, [&] {
        return gemm(h, C.d->head, nullptr, C.at(C.L.lsc), c.dt, M, c.vocab, c.d_model, c.d_model, C.at(C.L.part),
                    C.counters(), C.status(), C.st, C.plan);
    }));
    // the workspace layout depends on the call's shape, so other buffers may
    // have used these bytes since the last acceptance: clear its counters
    return accept(C.at(C.L.lsc), c.dt, drafts, B, D, c.vocab, n_acc, next_tok, C.at(C.L.aws), C.st, true);
}

template <typename T>
cudaError_t forward_impl(const Ctx &C, const int32_t *first_tok, const int32_t *toks, int tok_stride, int B,
                         int Dq, const int32_t *ctx, int max_ctx, void *kc, void *vcache, int L_stride, void *kb,
                         void *vb, int last_only, void *logits, int32_t *n_acc = nullptr,
                         int32_t *next_tok = nullptr)
{
    const vc_decoder_cfg &c = C.d->c;
    const int M = B * Dq;
    const int hd = c.head_dim, qd = c.n_heads * hd, nqkv = qd + 2 * c.n_kv_heads * hd;
    const size_t layer_cache = (size_t)B * c.n_kv_heads * L_stride * hd;
    const size_t layer_blk = (size_t)B * c.n_kv_heads * Dq * hd;
    void *x = C.at(C.L.x), *h = C.at(C.L.h), *part = C.at(C.L.part);
    const float scale = 1.0f / sqrtf((float)hd);
    // the attention's status block sits where other calls keep activations
    VC_TRY(cudaMemsetAsync(C.at(C.L.vws), 0, kStatusBytes, C.st));
    // a plain launch after the memset; the kernels after it start early
    // (programmatic dependent launch) and wait for their inputs on the device
    embed_kernel<T><<<M, kRowThreads, 0, C.st>>>(first_tok, toks, tok_stride, Dq, (const T *)C.d->embed, c.vocab,
                                                 c.d_model, (T *)x, C.status());
    VC_TRY(cudaGetLastError());
    for (int l = 0; l < c.n_layers; ++l) {
        VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
        VC_TRY(traced(C, VC_TRACE_GEMM_QKV, [&] {
            return gemm(h, C.d->wqkv[l], nullptr, C.at(C.L.qkv), c.dt, M, nqkv, c.d_model, c.d_model, part,
                        C.counters(), C.status(), C.st, C.plan);
        }));
        if (!C.d->layer_ev.empty()) VC_TRY(cudaStreamWaitEvent(C.st, C.d->layer_ev[l], 0));
        RopeDst dst{};
        dst.k1 = (T *)kc + l * layer_cache;
        dst.v1 = (T *)vcache + l * layer_cache;
        dst.bstride1 = (size_t)c.n_kv_heads * L_stride * hd;
        dst.stride1 = L_stride;
        dst.pos1 = 1;
        dst.k2 = kb ? (void *)((T *)kb + l * layer_blk) : nullptr;
        dst.v2 = vb ? (void *)((T *)vb + l * layer_blk) : nullptr;
        dst.bstride2 = (size_t)c.n_kv_heads * Dq * hd;
        dst.stride2 = Dq;
        VC_TRY(launch_pdl(rope_kernel<T>, dim3(M, rope_blocks(c)), dim3(kRopeHeads * 64), 0, C.st,
                          C.at<const T>(C.L.qkv), Dq, c.n_heads, c.n_kv_heads, hd, ctx, C.d->rope, C.at<T>(C.L.q),
                          dst, C.status()));
        VC_TRY(traced(C, VC_TRACE_VERIFY_ATTN, [&] {
            return verify_attn(C.at(C.L.q), dst.k1, dst.v1, c.dt, ctx, B, Dq, c.n_heads, c.n_kv_heads, hd, L_stride,
                               max_ctx, scale, C.at(C.L.att), C.at(C.L.vws), C.st, kSplitTiles);
        }));
        VC_TRY(layer_tail<T>(C, l, M));
    }
    if (!logits) {
        // verify: the head's argmax feeds acceptance directly (tokens after
        // the first are the drafts)
        VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
        VC_TRY(greedy_head(C, h, B, Dq - 1, toks, n_acc, next_tok));
    } else if (last_only) {
        VC_TRY(rmsnorm<T>(C, x, B, Dq, Dq - 1, C.at(C.L.hl)));
        VC_TRY(traced(C, VC_TRACE_GEMM_HEAD, [&] {
            return gemm(C.at(C.L.hl), C.d->head, nullptr, logits, c.dt, B, c.vocab, c.d_model, c.d_model, part,
                        C.counters(), C.status(), C.st, C.plan);
        }));
    } else {
        VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
        VC_TRY(traced(C, VC_TRACE_GEMM_HEAD, [&] {
            return gemm(h, C.d->head, nullptr, logits, c.dt, M, c.vocab, c.d_model, c.d_model, part, C.counters(),
                        C.status(), C.st, C.plan);
        }));
    }
    return launch_pdl(fold_status_kernel, dim3(1), dim3(1), 0, C.st, C.status(), C.at<int32_t>(C.L.vws),
                      (int32_t *)nullptr, (int32_t *)nullptr);
}

template <typename T>
cudaError_t draft_impl(const Ctx &C, const int32_t *tok, int B, vc_qcache *caches, void *logits, int32_t *next_tok,
                       int32_t *drafts_out, int drafts_stride)
{
    const vc_decoder_cfg &c = C.d->c;
    const int M = B;
    const int hd = c.head_dim, qd = c.n_heads * hd, kvd = c.n_kv_heads * hd, nqkv = qd + 2 * kvd;
    void *x = C.at(C.L.x), *h = C.at(C.L.h), *part = C.at(C.L.part);
    T *kn = C.at<T>(C.L.kvn), *vn = kn + (size_t)B * kvd;
    const float scale = 1.0f / sqrtf((float)hd);
    // the draft kernel's status block and arrival counters (zero between its
    // calls) share the workspace with regions that forward passes overwrite:
    // the embedding launch clears them, and RoPE's arrivals, first (a kernel
    // rather than memset nodes, so the chain of programmatic dependent
    // launches runs on from one draft step into the next)
    VC_TRY(launch_pdl(embed_kernel<T>, dim3(M), dim3(kRowThreads), 0, C.st, tok, (const int32_t *)nullptr, 0, 1,
                      (const T *)C.d->embed, c.vocab, c.d_model, (T *)x, C.status(), C.at<uint32_t>(C.L.dws),
                      (int)((kStatusBytes + a256((size_t)B * c.n_kv_heads * 4)) / 4), C.at<uint32_t>(C.L.rarr), B));
    // the q|k|v and LM-head products take x itself and normalise its rows in
    // their epilogue (no RMSNorm launches in a draft step) when the shape allows
    const bool rms_qkv = gemm_rms_ok(c.dt, M, nqkv, c.d_model, c.d_model, C.plan);
    const bool rms_head = !logits && C.L.fused_head && gemm_rms_ok(c.dt, M, c.vocab, c.d_model, c.d_model, C.plan);
    for (int l = 0; l < c.n_layers; ++l) {
        if (!rms_qkv) VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
        VC_TRY(traced(C, VC_TRACE_GEMM_QKV, [&] {
            return gemm(rms_qkv ? x : h, C.d->wqkv[l], nullptr, C.at(C.L.qkv), c.dt, M, nqkv, c.d_model, c.d_model,
                        part, C.counters(), C.status(), C.st, C.plan, nullptr, nullptr, rms_qkv ? c.norm_eps : -1.f);
        }));
        RopeDst dst{};
        dst.k1 = kn;
        dst.v1 = vn;
        dst.bstride1 = (size_t)kvd;
        dst.stride1 = 1;
        dst.pos1 = 0;
        dst.k2 = dst.v2 = nullptr;
        dst.bstride2 = 0;
        dst.stride2 = 1;
        // the new row straight into the ring (one launch less per layer),
        // unless the cache rotates its keys on the way in
        const vc_qcache &qc = caches[l];
        const bool ring = !qc.cfg.rotate && qc.d == hd && qc.Hkv == c.n_kv_heads && qc.B >= B &&
                          (qc.res_dtype == VC_BF16) == (sizeof(T) == 2);
        if (ring) {
            dst.kr = qc.k_res;
            dst.vr = qc.v_res;
            dst.res_cap = qc.res_cap;
            dst.len = qc.seq_len;
            dst.ngroups = qc.n_groups;
            dst.qstatus = qc.status;
            dst.arrive = C.at<unsigned int>(C.L.rarr);
        }
        VC_TRY(launch_pdl(rope_kernel<T>, dim3(M, rope_blocks(c)), dim3(kRopeHeads * 64), 0, C.st,
                          C.at<const T>(C.L.qkv), 1, c.n_heads, c.n_kv_heads, hd, (const int32_t *)caches[l].seq_len,
                          C.d->rope, C.at<T>(C.L.q), dst, C.status()));
        if (!ring) VC_TRY(qcache_append(&caches[l], kn, vn, nullptr, nullptr, nullptr, 1, 0, C.st));
        vc_cache_view view{};
        view.kind = VC_CACHE_KIVI;
        view.kivi = &caches[l];
        // in a draft step the kernel before draft attention (RoPE, or the ring
        // append) writes only the ring and the length: the records are stable
        view.flags = VC_VIEW_RECORDS_STABLE;
        VC_TRY(traced(C, VC_TRACE_DRAFT_ATTN, [&] {
            return draft_attn(C.at(C.L.q), c.dt, &view, c.n_heads, scale, C.at(C.L.att), C.at(C.L.dws), C.st);
        }));
        VC_TRY(layer_tail<T>(C, l, M));
    }
    if (!rms_head) VC_TRY(rmsnorm<T>(C, x, M, 1, 0, h));
    if (logits) {
        VC_TRY(traced(C, VC_TRACE_GEMM_HEAD, [&] {
            return gemm(h, C.d->head, nullptr, logits, c.dt, M, c.vocab, c.d_model, c.d_model, part, C.counters(),
                        C.status(), C.st, C.plan);
        }));
        VC_TRY(accept(logits, c.dt, nullptr, B, 0, c.vocab, C.at<int32_t>(C.L.nacc), next_tok, C.at(C.L.aws),
                      C.st, true));
    } else if (rms_head) {
        VC_TRY(greedy_head(C, x, B, 0, nullptr, C.at<int32_t>(C.L.nacc), next_tok, c.norm_eps));
    } else {
        VC_TRY(greedy_head(C, h, B, 0, nullptr, C.at<int32_t>(C.L.nacc), next_tok));
    }
    if (drafts_out) {
        VC_TRY(launch_pdl(scatter_tokens_kernel, dim3((B + 127) / 128), dim3(128), 0, C.st, (const int32_t *)next_tok,
                          B, drafts_out, drafts_stride));
    }
    return launch_pdl(fold_status_kernel, dim3(1), dim3(1), 0, C.st, C.status(), C.at<int32_t>(C.L.dws),
                      (int32_t *)nullptr, (int32_t *)nullptr);
}

vc_status to_status(cudaError_t e)
{
    if (e == cudaSuccess) return VC_OK;
    cudaGetLastError();
    return e == cudaErrorInvalidValue ? VC_ERR_INVALID : VC_ERR_CUDA;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace vc

using namespace vc;

extern "C" {

vc_status vc_decoder_create(const vc_decoder_cfg *cfg, const vc_decoder_weights *w, vc_decoder **out)
{
    if (!cfg || !w || !out) return VC_ERR_INVALID;
    *out = nullptr;
    const vc_decoder_cfg &c = *cfg;
    if (c.n_layers <= 0 || c.d_model <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.d_ff <= 0 || c.vocab <= 0)
        return VC_ERR_INVALID;
    if (c.dt != VC_BF16 && c.dt != VC_F32) return VC_ERR_INVALID;
    if (c.n_heads % c.n_kv_heads || c.n_heads / c.n_kv_heads > 4) return VC_ERR_UNSUPPORTED;
    if (c.head_dim != 64 && c.head_dim != 128) return VC_ERR_UNSUPPORTED;
    if (c.d_model % 8 || c.d_ff % 64 || c.vocab % 8) return VC_ERR_UNSUPPORTED;   // gate|up interleaved per 64
    if (!(c.norm_eps >= 0.f) || !(c.rope_theta > 0.f)) return VC_ERR_INVALID;
    if (!w->embed || !w->lm_head || !w->w_qkv || !w->w_o || !w->w_gate_up || !w->w_down) return VC_ERR_INVALID;
    if (!aligned16(w->embed) || !aligned16(w->lm_head)) return VC_ERR_INVALID;
    vc_decoder *d = new (std::nothrow) vc_decoder;
    if (!d) return VC_ERR_INVALID;
    d->c = c;
    for (int j = 0; j < c.head_dim / 2; ++j)
        d->rope.inv_freq[j] = std::pow((double)c.rope_theta, -2.0 * j / (double)c.head_dim);
    d->embed = w->embed;
    d->head = w->lm_head;
    for (int l = 0; l < c.n_layers; ++l) {
        const void *p[4] = {w->w_qkv[l], w->w_o[l], w->w_gate_up[l], w->w_down[l]};
        for (const void *q : p)
            if (!q || !aligned16(q)) {
                delete d;
                return VC_ERR_INVALID;
            }
        d->wqkv.push_back(p[0]);
        d->wo.push_back(p[1]);
        d->wgu.push_back(p[2]);
        d->wd.push_back(p[3]);
    }
    *out = d;
    return VC_OK;
}

void vc_decoder_destroy(vc_decoder *dec) { delete dec; }

vc_status vc_decoder_set_trace(vc_decoder *dec, cudaEvent_t *events, int32_t *kinds, int capacity, int kind_mask)
{
    if (!dec || capacity < 0 || (capacity > 0 && (!events || !kinds))) return VC_ERR_INVALID;
    dec->tr_ev = capacity > 0 ? events : nullptr;
    dec->tr_kind = kinds;
    dec->tr_cap = capacity;
    dec->tr_n = 0;
    dec->tr_mask = kind_mask;
    return VC_OK;
}

int vc_decoder_trace_count(const vc_decoder *dec) { return dec ? dec->tr_n : 0; }

vc_status vc_decoder_set_layer_events(vc_decoder *dec, const cudaEvent_t *events, int n)
{
    if (!dec || n < 0) return VC_ERR_INVALID;
    if (n == 0) {
        dec->layer_ev.clear();
        return VC_OK;
    }
    if (!events || n != dec->c.n_layers) return VC_ERR_INVALID;
    for (int l = 0; l < n; ++l)
        if (!events[l]) return VC_ERR_INVALID;
    dec->layer_ev.assign(events, events + n);
    return VC_OK;
}

size_t vc_decoder_workspace_bytes(const vc_decoder *dec, int B, int max_rows, int max_ctx,
                                  const vc_qcache *draft_cache)
{
    if (!dec || B <= 0 || max_rows <= 0 || max_ctx < 0) return 0;
    return layout_of(dec, B, max_rows, max_ctx, draft_ws_of(dec, draft_cache)).total;
}

vc_status vc_decoder_forward(const vc_decoder *dec, const int32_t *first_tok, const int32_t *tokens,
                             int tok_stride, int B, int Dq, const int32_t *ctx_len, int max_ctx,
                             void *k_cache, void *v_cache, int L_stride, void *k_blk, void *v_blk,
                             int logits_last_only, void *logits, void *ws, size_t ws_bytes,
                             cudaStream_t stream)
{
    if (!dec || !ctx_len || !k_cache || !v_cache || !logits || !ws) return VC_ERR_INVALID;
    if (B <= 0 || Dq <= 0 || max_ctx < 0 || L_stride < max_ctx + Dq) return VC_ERR_INVALID;
    if ((k_blk == nullptr) != (v_blk == nullptr)) return VC_ERR_INVALID;
    if (!first_tok && !tokens) return VC_ERR_INVALID;
    if (tokens && tok_stride < (first_tok ? Dq - 1 : Dq)) return VC_ERR_INVALID;
    if (first_tok && !tokens && Dq > 1) return VC_ERR_INVALID;
    if (((uintptr_t)ws & 255u) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(logits))
        return VC_ERR_INVALID;
    const Layout L = layout_of(dec, B, Dq, max_ctx, 0);
    if (ws_bytes < L.total) return VC_ERR_INVALID;
    Ctx C{dec, (uint8_t *)ws, L, stream, kGemmRowInvariant | kGemmEarlyWeights};
    const cudaError_t e =
        dec->c.dt == VC_BF16
            ? forward_impl<__nv_bfloat16>(C, first_tok, tokens, tok_stride, B, Dq, ctx_len, max_ctx, k_cache, v_cache,
                                          L_stride, k_blk, v_blk, logits_last_only, logits)
            : forward_impl<float>(C, first_tok, tokens, tok_stride, B, Dq, ctx_len, max_ctx, k_cache, v_cache,
                                  L_stride, k_blk, v_blk, logits_last_only, logits);
    return to_status(e);
}

vc_status vc_decoder_draft_step(const vc_decoder *dec, const int32_t *tok, int B, vc_qcache *caches,
                                void *logits, int32_t *next_tok, int32_t *drafts_out, int drafts_stride,
                                void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!dec || !tok || !caches || !next_tok || !ws || B <= 0) return VC_ERR_INVALID;
    if (drafts_out && drafts_stride <= 0) return VC_ERR_INVALID;
    if (((uintptr_t)ws & 255u) || (logits && !aligned16(logits))) return VC_ERR_INVALID;
    const vc_decoder_cfg &c = dec->c;
    for (int l = 0; l < c.n_layers; ++l) {
        const vc_qcache &q = caches[l];
        if (!q.records || !q.k_res || !q.v_res || !q.n_groups || !q.seq_len) return VC_ERR_INVALID;
        if (q.B != B || q.Hkv != c.n_kv_heads || q.d != c.head_dim || q.res_dtype != c.dt) return VC_ERR_INVALID;
        if (q.max_groups != caches[0].max_groups || q.res_cap != caches[0].res_cap ||
            q.cfg.bits != caches[0].cfg.bits || q.cfg.residual != caches[0].cfg.residual)
            return VC_ERR_INVALID;
    }
    const Layout L = layout_of(dec, B, 1, 0, draft_ws_of(dec, &caches[0]));
    if (ws_bytes < L.total) return VC_ERR_INVALID;
    Ctx C{dec, (uint8_t *)ws, L, stream, kGemmDecode | kGemmEarlyWeights};
    const cudaError_t e =
        c.dt == VC_BF16
            ? draft_impl<__nv_bfloat16>(C, tok, B, caches, logits, next_tok, drafts_out, drafts_stride)
            : draft_impl<float>(C, tok, B, caches, logits, next_tok, drafts_out, drafts_stride);
    return to_status(e);
}

vc_status vc_kv_writeback(const void *k_blk, const void *v_blk, vc_dtype dt, int n_layers, int B, int Hkv, int Dq,
                          int d, const int32_t *n_acc, const int32_t *ctx_len, void *k_host, void *v_host,
                          int L_stride, cudaStream_t stream)
{
    if (!k_blk || !v_blk || !n_acc || !ctx_len || !k_host || !v_host) return VC_ERR_INVALID;
    if ((dt != VC_BF16 && dt != VC_F32) || n_layers <= 0 || B <= 0 || Hkv <= 0 || Dq <= 0 || d <= 0 ||
        L_stride < Dq)
        return VC_ERR_INVALID;
    void *kd = nullptr, *vd = nullptr;
    if (cudaHostGetDevicePointer(&kd, k_host, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&vd, v_host, 0) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_INVALID;
    }
    dim3 grid(Dq, B * Hkv, n_layers);
    if (dt == VC_BF16)
        writeback_kernel<__nv_bfloat16><<<grid, 64, 0, stream>>>(
            (const __nv_bfloat16 *)k_blk, (const __nv_bfloat16 *)v_blk, B, Hkv, Dq, d, n_acc, ctx_len,
            (__nv_bfloat16 *)kd, (__nv_bfloat16 *)vd, L_stride);
    else
        writeback_kernel<float><<<grid, 64, 0, stream>>>((const float *)k_blk, (const float *)v_blk, B, Hkv, Dq, d,
                                                         n_acc, ctx_len, (float *)kd, (float *)vd, L_stride);
    return to_status(cudaGetLastError());
}

int vc_gemm_splits(vc_dtype dt, int N, int K, int decode_plan)
{
    if ((dt != VC_BF16 && dt != VC_F32) || N <= 0 || K <= 0) return 0;
    if (!gemm_uses_tensor_cores(dt, N, K)) return 1;
    return gemm_splits(N, K, decode_plan ? kGemmDecode : kGemmRowInvariant);
}

size_t vc_gemm_workspace_bytes(vc_dtype dt, int M, int N, int K)
{
    if ((dt != VC_BF16 && dt != VC_F32) || M <= 0 || N <= 0 || K <= 0) return 0;
    const size_t p = std::max(gemm_ws_bytes(dt, M, N, K, kGemmRowInvariant), gemm_ws_bytes(dt, M, N, K, kGemmDecode));
    return p ? p + kGemmCounterBytes : 0;
}

vc_status vc_gemm_ex(const void *x, const void *w, const void *resid, void *out, vc_dtype dt, int M, int N, int K,
                     int decode_plan, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!x || !w || !out || (dt != VC_BF16 && dt != VC_F32) || M <= 0 || N <= 0 || K <= 0) return VC_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (resid && !aligned16(resid))) return VC_ERR_INVALID;
    const int plan = decode_plan ? kGemmDecode : kGemmRowInvariant;
    const size_t need = gemm_ws_bytes(dt, M, N, K, plan);
    if (need && (!ws || ws_bytes < need + kGemmCounterBytes || !aligned16(ws))) return VC_ERR_INVALID;
    return to_status(gemm(x, w, resid, out, dt, M, N, K, K, need ? (uint8_t *)ws + kGemmCounterBytes : nullptr,
                          need ? (unsigned int *)ws : nullptr, nullptr, stream, plan));
}

vc_status vc_gemm(const void *x, const void *w, const void *resid, void *out, vc_dtype dt, int M, int N, int K,
                  void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return vc_gemm_ex(x, w, resid, out, dt, M, N, K, 0, ws, ws_bytes, stream);
}

vc_status vc_gemm_rms(const void *x, const void *w, void *out, vc_dtype dt, int M, int N, int K, float eps, int swiglu,
                      void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!x || !w || !out || M <= 0 || N <= 0 || K <= 0 || !(eps >= 0.f)) return VC_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out)) return VC_ERR_INVALID;
    if (!gemm_rms_ok(dt, M, N, K, K, kGemmDecode)) return VC_ERR_UNSUPPORTED;
    if (swiglu) {
        if (N % 2 || !gemm_swiglu_ok(dt, N / 2, K, kGemmDecode)) return VC_ERR_UNSUPPORTED;
        return to_status(gemm_swiglu(x, w, out, dt, M, N / 2, K, K, nullptr, stream, kGemmDecode, eps));
    }
    const size_t need = gemm_ws_bytes(dt, M, N, K, kGemmDecode);
    if (need && (!ws || ws_bytes < need + kGemmCounterBytes || !aligned16(ws))) return VC_ERR_INVALID;
    return to_status(gemm(x, w, nullptr, out, dt, M, N, K, K, need ? (uint8_t *)ws + kGemmCounterBytes : nullptr,
                          need ? (unsigned int *)ws : nullptr, nullptr, stream, kGemmDecode, nullptr, nullptr, eps));
}

vc_status vc_gemm_swiglu(const void *x, const void *w_gate_up, void *act, vc_dtype dt, int M, int F, int K,
                         int decode_plan, cudaStream_t stream)
{
    if (!x || !w_gate_up || !act || M <= 0 || F <= 0 || K <= 0) return VC_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_gate_up) || !aligned16(act)) return VC_ERR_INVALID;
    const int plan = decode_plan ? kGemmDecode : kGemmRowInvariant;
    if (!gemm_swiglu_ok(dt, F, K, plan)) return VC_ERR_UNSUPPORTED;
    return to_status(gemm_swiglu(x, w_gate_up, act, dt, M, F, K, K, nullptr, stream, plan));
}

vc_status vc_gemm_argmax(const void *x, const void *w, vc_dtype dt, int M, int N, int K, int decode_plan,
                         float *tile_max, int32_t *tile_idx, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!x || !w || !tile_max || !tile_idx || M <= 0 || N <= 0 || K <= 0) return VC_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w)) return VC_ERR_INVALID;
    const int plan = decode_plan ? kGemmDecode : kGemmRowInvariant;
    if (!gemm_argmax_ok(dt, M, N, K, plan, true)) return VC_ERR_UNSUPPORTED;
    const size_t need = gemm_ws_bytes(dt, M, N, K, plan);
    if (need && (!ws || ws_bytes < need + kGemmCounterBytes || !aligned16(ws))) return VC_ERR_INVALID;
    return to_status(gemm(x, w, nullptr, nullptr, dt, M, N, K, K, need ? (uint8_t *)ws + kGemmCounterBytes : nullptr,
                          need ? (unsigned int *)ws : nullptr, nullptr, stream, plan, tile_max, tile_idx));
}

vc_status vc_decoder_verify(const vc_decoder *dec, const int32_t *first_tok, const int32_t *drafts, int D, int B,
                            const int32_t *ctx_len, int max_ctx, void *k_cache, void *v_cache, int L_stride,
                            void *k_blk, void *v_blk, int32_t *n_acc, int32_t *next_tok, void *ws, size_t ws_bytes,
                            cudaStream_t stream)
{
    if (!dec || !first_tok || !ctx_len || !k_cache || !v_cache || !n_acc || !next_tok || !ws) return VC_ERR_INVALID;
    if (B <= 0 || D < 0 || D > 1024 || (D > 0 && !drafts)) return VC_ERR_INVALID;
    const int Dq = D + 1;
    if (max_ctx < 0 || L_stride < max_ctx + Dq) return VC_ERR_INVALID;
    if ((k_blk == nullptr) != (v_blk == nullptr)) return VC_ERR_INVALID;
    if (((uintptr_t)ws & 255u) || !aligned16(k_cache) || !aligned16(v_cache)) return VC_ERR_INVALID;
    const Layout L = layout_of(dec, B, Dq, max_ctx, 0);
    if (ws_bytes < L.total) return VC_ERR_INVALID;
    Ctx C{dec, (uint8_t *)ws, L, stream, kGemmRowInvariant | kGemmEarlyWeights};
    const int32_t *toks = D > 0 ? drafts : nullptr;
    const cudaError_t e =
        dec->c.dt == VC_BF16
            ? forward_impl<__nv_bfloat16>(C, first_tok, toks, D, B, Dq, ctx_len, max_ctx, k_cache, v_cache,
                                          L_stride, k_blk, v_blk, 0, nullptr, n_acc, next_tok)
            : forward_impl<float>(C, first_tok, toks, D, B, Dq, ctx_len, max_ctx, k_cache, v_cache, L_stride, k_blk,
                                  v_blk, 0, nullptr, n_acc, next_tok);
    return to_status(e);
}

}  // extern "C"
