// draft_attn.cu -- single-query decode attention over the compressed draft
// cache (VeriCache drafts on the compressed cache; drafting is
// HBM-bandwidth-bound, paper page "What the paper found").
//
// KIVI cache kernel.  Grid = (split, kv unit); each CTA streams a contiguous
// range of 32-token group records through per-warp shared-memory rings filled
// by cp.async.bulk (one bulk copy per pair of records, mbarrier completion).
// A warp owns pairs of groups and computes, for the Hq/Hkv <= 4 query heads of
// its kv head, the scores and the weighted values with m16n8k16 tensor-core
// MMAs on the integer codes themselves: the per-channel K scale is folded into
// the query (q' = q * s), the per-token V scale into the probabilities
// (p' = p * s), and the K zero-point enters through one small MMA whose
// operand is the padding head columns 4..7 (n = 8), the V zero-point through
// another.  Codes become exact fp16 operands with a single AND per pair: the
// masked bits are an fp16 subnormal code * 2^(b e) * 2^-24, the slot factor
// 2^(b e) being fixed per channel by the record layout and cancelled in q (K)
// or per output row (V).  Online softmax in the exp2 domain with lazy
// rescaling.  The residual window (the most recent tokens, full precision):
// a bf16 window is cut into 16-token tiles that run on bf16 MMAs inside the
// quantized splits, continuing the warps' softmax state; an fp32 window is
// one or more extra splits of fp32 CUDA-core math.  The last CTA of each kv
// unit (device-scope counter in the workspace, returned to zero after use)
// merges the split partials.
//
// Dense cache kernels (compacted dropped cache, or an uncompressed cache):
// bf16 caches use the same MMA structure with the K/V tiles as operands
// (ldmatrix from padded rows); fp32 caches use CUDA-core math over 32-token
// tiles staged by cp.async.bulk.
//
// Every ring stage is read with ordinary loads and refilled by a bulk copy
// (async proxy): each reading lane fences (fence.proxy.async) before the
// stage is released.  The kernels wait on griddepcontrol.wait before their
// first global access (programmatic dependent launch).
#include <algorithm>
#include <type_traits>

#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int G = 32;
constexpr int NW = 4;                    // warps per CTA
constexpr int kThreads = NW * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;
constexpr float kLazy = 8.0f;            // rescale only when the max grows by > 2^8

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// partial record per (unit, split): m[4], l[4], o[4][D] (fp32, unnormalized)
__host__ __device__ constexpr int part_floats(int D) { return 8 + 4 * D; }
// the CTA merge's shared buffer: every warp's (m, l, o), then the warps' weights and the maxima
__host__ __device__ constexpr int merge_floats(int D) { return NW * part_floats(D) + NW * 4 + 4; }

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

constexpr uint32_t kOnes = 0x3C003C00u;    // half2(1, 1)

// ------------------------------------------------------------ KIVI kernel --
// Position of code pair (kappa, mu) of a lane (record format, include/vc.h)
// and the power-of-two factor its slot gives the unpacked value:
// lop3(word >> sh, mask << b*slot, 0x6400) = fp16(1024 + code * 2^(b*e)).
template <int BITS, int D>
struct Pairs {
    static constexpr int W = D * BITS / 32;        // words per lane per section
    struct Pos {
        int word, slot, e;
    };
    static constexpr Pos pos(int kappa, int mu)
    {
        if (BITS == 2) {
            const int h = W / 2, q = W / 4;
            if (kappa < 3 * h) return {2 * (kappa % h) + mu / 2, kappa / h + 5 * (mu % 2), kappa / h};
            const int k2 = kappa - 3 * h;
            return {4 * (k2 % q) + mu, 3 + k2 / q, 3 + k2 / q};
        } else {
            const int h = W / 2;
            return {2 * (kappa % h) + mu / 2, kappa / h + 2 * (mu % 2), kappa / h};
        }
    }
    // exponent of class kappa: the unpacked code carries a factor 2^(BITS*e)
    static constexpr int exp_of(int kappa) { return pos(kappa, 0).e; }
};

// Unpack pair (kappa, mu) from the lane's words w0 (as stored) and w1 (the
// words shifted right so that the high slots land at the bottom).  Masking
// the two codes in place yields two fp16 subnormals of exact value
// code * 2^(b e) * 2^-24: the MMA multiplies them exactly and the caller
// removes the 2^24 and 2^(b e) factors once.
template <int BITS, int D>
__device__ __forceinline__ uint32_t unpack(const uint32_t *w0, const uint32_t *w1, int kappa, int mu)
{
    constexpr uint32_t base = BITS == 2 ? 0x00030003u : 0x000F000Fu;
    constexpr int split = BITS == 2 ? 5 : 2;       // slots >= split come from the shifted words
    const auto p = Pairs<BITS, D>::pos(kappa, mu);
    const uint32_t src = p.slot < split ? w0[p.word] : w1[p.word];
    const int sl = p.slot < split ? p.slot : p.slot - split;
    return src & (base << (BITS * sl));
}

constexpr float kTwo24 = 16777216.0f;          // undoes the subnormal 2^-24

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int BITS, int D>
struct KiviGeom {
    static constexpr int KS = D / 16;                  // QK k-steps, PV m-tiles
    static constexpr int NG = D / 32;                  // V channel groups
    static constexpr int CODE_BYTES = G * D * BITS / 8;
    static constexpr int W = D * BITS / 32;            // code words per lane per section
    static constexpr int KM = 2 * CODE_BYTES;          // K meta offset
    static constexpr int VM = KM + 4 * D;              // V meta offset
    static constexpr int REC = VM + 4 * D;             // record bytes
    static constexpr int SHIFT = BITS == 2 ? 10 : 8;   // high-slot shift
    static constexpr int NST = 2;                      // ring stages per warp (2 records each)
};

struct KiviParams {
    const void *q;
    const uint8_t *records;
    const void *kres, *vres;
    const int32_t *n_groups, *seq_len;
    float *part;
    unsigned int *counters;                            // [units], zero between calls
    void *out;
    int32_t *status;
    int Hkv, Hq, grp, max_groups, res_cap, n_split_q;
    int n_split_r, res_per_split;                      // ring splits and ring tokens per split
    float qscale;                                      // sm_scale * log2(e)
    float *raw;                                        // optional [units][raw_stride][4] log2-domain scores (H2O)
    float *ml;                                         // optional [units][8]: each head's final max and sum
    int raw_stride;
    int early_records;   // records and n_groups stable: the first record copies precede the grid-dependency wait
};

template <typename TQ, int D>
__device__ __forceinline__ float load_q(const TQ *q, int idx) { return Elem<TQ>::to_f(q[idx]); }

// q[idx], q[idx + 1] for even idx, one load when the pair is aligned
template <typename TQ, int D>
__device__ __forceinline__ float2 load_q2(const TQ *q, int idx, bool pairs)
{
    if (pairs) {
        if constexpr (std::is_same<TQ, float>::value) {
            return *reinterpret_cast<const float2 *>(q + idx);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(q + idx);
            return make_float2(bf16_lo(w), bf16_hi(w));
        }
    }
    return make_float2(load_q<TQ, D>(q, idx), load_q<TQ, D>(q, idx + 1));
}

// Merge the NW warps' (m, l, o) of this CTA in shared memory and store the
// CTA partial.  Every warp has written wm[w][h], wl[w][h], wo[w][h][c].
template <int D>
__device__ void cta_merge_store(float *wbuf, float *dst, int grp)
{
    __syncthreads();
    float *wm = wbuf;                       // [NW][4]
    float *wl = wbuf + NW * 4;              // [NW][4]
    float *wo = wbuf + NW * 8;              // [NW][4][D]
    float *ww = wo + NW * 4 * D;            // [NW][4] weights 2^(m_w - M), then [4] M
    if (threadIdx.x < NW * 4) {
        const int h = threadIdx.x & 3;
        float M = kNegBig;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * 4 + h]);
        ww[threadIdx.x] = exp2f(wm[threadIdx.x] - M);
        if (threadIdx.x < 4) ww[NW * 4 + h] = M;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * D; i += kThreads) {
        const int h = i / D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) o += wo[(w * 4 + h) * D + (i % D)] * ww[w * 4 + h];
        dst[8 + i] = h < grp ? o : 0.f;
    }
    if (threadIdx.x < 4) {
        const int h = threadIdx.x;
        float L = 0.f;
        for (int w = 0; w < NW; ++w) L += wl[w * 4 + h] * ww[w * 4 + h];
        dst[h] = ww[NW * 4 + h];
        dst[4 + h] = h < grp ? L : 0.f;
    }
}

// The last CTA of a kv unit to finish merges the unit's split partials and
// writes the normalised output rows out[h][D] (h < grp); the counter is left
// at zero for the next call.  The per-split weights 2^(m_s - M) / L are
// computed once in shared memory, so each output element is a sum of
// independent loads.
constexpr int kMaxSplit = 64;

template <typename TO, int D>
__device__ void last_cta_combine(const float *unit_part, int n_split, unsigned int *counter, int grp,
                                 TO *out, float *ml_out = nullptr)
{
    __shared__ bool is_last;
    __shared__ float wgt[4][kMaxSplit];      // the splits' m, then their weights
    __shared__ float lsp[4][kMaxSplit];      // the splits' l
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(counter, 1u) == (unsigned int)(n_split - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // every split's (m, l) in one round of independent loads
    for (int i = threadIdx.x; i < 4 * n_split; i += kThreads) {
        const int s = i >> 2, h = i & 3;
        const float *q = unit_part + (size_t)s * part_floats(D);
        wgt[h][s] = __ldcg(q + h);
        lsp[h][s] = __ldcg(q + 4 + h);
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        const int h = threadIdx.x;
        float M = kNegBig;
        for (int s = 0; s < n_split; ++s) M = fmaxf(M, wgt[h][s]);
        float L = 0.f;
        for (int s = 0; s < n_split; ++s) {
            const float w = exp2f(wgt[h][s] - M);
            wgt[h][s] = w;
            L += lsp[h][s] * w;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int s = 0; s < n_split; ++s) wgt[h][s] *= inv;
        if (ml_out) {
            ml_out[h] = M;
            ml_out[4 + h] = L;
        }
    }
    __syncthreads();
    // four consecutive channels per thread (the split rows are 16-byte aligned)
    static_assert(part_floats(D) % 4 == 0 && D % 4 == 0, "float4 partial rows");
    for (int i = 4 * threadIdx.x; i < grp * D; i += 4 * kThreads) {
        const int h = i / D, c = i % D;
        const float *q = unit_part + 8 + h * D + c;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int s = 0; s < n_split; ++s) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(q + (size_t)s * part_floats(D)));
            const float w = wgt[h][s];
            O.x = fmaf(x.x, w, O.x);
            O.y = fmaf(x.y, w, O.y);
            O.z = fmaf(x.z, w, O.z);
            O.w = fmaf(x.w, w, O.w);
        }
        out[h * D + c] = Elem<TO>::from_f(O.x);
        out[h * D + c + 1] = Elem<TO>::from_f(O.y);
        out[h * D + c + 2] = Elem<TO>::from_f(O.z);
        out[h * D + c + 3] = Elem<TO>::from_f(O.w);
    }
    if (threadIdx.x == 0) *counter = 0u;
}

// Scores of one group: sc[mt][4] (rows = tokens 16 mt + gid (+8), columns =
// heads 2 tig + {0,1}) with the zero-point term folded in.
// kmeta: this lane quad's K meta chunks (the record's, or fp16 ones for the
// head copies 4..7 on lanes gid >= 4).  The chunk of k-step ks is
// {z pair rr=0, s pair rr=0, z pair rr=1, s pair rr=1}: as loaded it is the
// A operand of the zero-point MMA (rows gid: the zero-points, rows gid + 8:
// the scales, whose products land in output rows that are never read), and
// its scale pairs scale q into the B operand.
template <int BITS, int D>
__device__ __forceinline__ void group_scores(const uint8_t *rec, const uint8_t *kmeta,
                                             const uint32_t (&qf)[D / 16][2], int lane, int tig,
                                             float (&sc)[2][4])
{
    using Gm = KiviGeom<BITS, D>;
    constexpr int KS = Gm::KS;
    uint32_t w0[Gm::W], w1[Gm::W];
#pragma unroll
    for (int c = 0; c < Gm::W / 4; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(rec + 16 * (32 * c + lane));
        w0[4 * c] = u.x; w0[4 * c + 1] = u.y; w0[4 * c + 2] = u.z; w0[4 * c + 3] = u.w;
    }
#pragma unroll
    for (int i = 0; i < Gm::W; ++i) w1[i] = w0[i] >> Gm::SHIFT;
    float cb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const uint4 m = *reinterpret_cast<const uint4 *>(kmeta + 16 * (4 * ks + tig));
        const uint32_t b0 = hmul2(qf[ks][0], m.y);
        const uint32_t b1 = hmul2(qf[ks][1], m.w);
        const uint32_t ab[4] = {m.x, m.y, m.z, m.w};
        mma16816(cb, ab, b0, b1);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            uint32_t a[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) a[r] = unpack<BITS, D>(w0, w1, 2 * ks + (r >> 1), 2 * mt + (r & 1));
            mma16816(sc[mt], a, b0, b1);
        }
    }
    // rows 0..3 of the bias tile, columns 4..7 = sum of z * q for heads 0..3
    // (columns 2 tig + {0, 1} of a lane are one register pair: packed FMAs)
    const int t1 = tig & 1;
    const float2 bias = make_float2(__shfl_sync(0xffffffffu, cb[0], 6 + t1), __shfl_sync(0xffffffffu, cb[1], 6 + t1));
    const float2 k24 = make_float2(kTwo24, kTwo24);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 4; r += 2) {
            const float2 v = fma2(make_float2(sc[mt][r], sc[mt][r + 1]), k24, bias);
            sc[mt][r] = v.x;
            sc[mt][r + 1] = v.y;
        }
}

// O += V^T p' for one group, plus the zero-point accumulator.
template <int BITS, int D>
__device__ __forceinline__ void group_values(const uint8_t *rec, const uint8_t *zvsrc, const uint32_t (&pb)[2][2],
                                             int lane, int tig, float (&o_acc)[D / 16][4], float (&vb_acc)[4])
{
    using Gm = KiviGeom<BITS, D>;
    constexpr int NG = Gm::NG;
    uint32_t w0[Gm::W], w1[Gm::W];
    const uint8_t *vsec = rec + Gm::CODE_BYTES;
#pragma unroll
    for (int c = 0; c < Gm::W / 4; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(vsec + 16 * (32 * c + lane));
        w0[4 * c] = u.x; w0[4 * c + 1] = u.y; w0[4 * c + 2] = u.z; w0[4 * c + 3] = u.w;
    }
#pragma unroll
    for (int i = 0; i < Gm::W; ++i) w1[i] = w0[i] >> Gm::SHIFT;
    // scale pairs of quad tig: n = (2 ks + rr) * NG + gc
    uint32_t sv[4 * NG];
    const uint8_t *vmeta = rec + Gm::VM;
#pragma unroll
    for (int c = 0; c < NG; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(vmeta + 16 * (4 * c + tig));
        sv[4 * c] = u.x; sv[4 * c + 1] = u.y; sv[4 * c + 2] = u.z; sv[4 * c + 3] = u.w;
    }
    // zero-point rows gc = lane/4 (< NG): pairs n = (2 ks + rr) * NG + gc;
    // rows gid + 8 are ones, so accumulator rows 8..15 sum the probabilities
    // (the softmax denominator, over the fp16 p the MMAs multiply)
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const int gid = lane >> 2;
        const int n0 = (2 * ks) * NG + (gid & (NG - 1)), n1 = (2 * ks + 1) * NG + (gid & (NG - 1));
        const uint32_t z0 = *reinterpret_cast<const uint32_t *>(zvsrc + 16 * (4 * (n0 >> 2) + tig) + 4 * (n0 & 3));
        const uint32_t z1 = *reinterpret_cast<const uint32_t *>(zvsrc + 16 * (4 * (n1 >> 2) + tig) + 4 * (n1 & 3));
        const uint32_t az[4] = {z0, kOnes, z1, kOnes};
        mma16816(vb_acc, az, pb[ks][0], pb[ks][1]);
#pragma unroll
        for (int gc = 0; gc < NG; ++gc) {
            const uint32_t b0 = hmul2(pb[ks][0], sv[(2 * ks) * NG + gc]);
            const uint32_t b1 = hmul2(pb[ks][1], sv[(2 * ks + 1) * NG + gc]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int mt = 2 * gc + half;
                uint32_t a[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) a[r] = unpack<BITS, D>(w0, w1, 2 * mt + (r & 1), 2 * ks + (r >> 1));
                mma16816(o_acc[mt], a, b0, b1);
            }
        }
    }
}

// Rotated-cache queries: rq[h][c] = W(q_h)[c] * 2^-floor(log2(D)/2) for the
// CTA's kv head (W the binary32 Walsh-Hadamard butterfly of the cache's key
// rotation, stages h = 1, ..., D/2, pair (i, i + h) -> (a + b, a - b)); rows
// h >= grp are zero.  Block-uniform call.
template <typename TQ, int D>
__device__ void rotate_queries(const TQ *qg, int grp, float *rq)
{
    for (int i = threadIdx.x; i < 4 * D; i += kThreads) rq[i] = i / D < grp ? Elem<TQ>::to_f(qg[i]) : 0.f;
    __syncthreads();
    for (int h = 1; h < D; h <<= 1) {
        for (int p = threadIdx.x; p < 4 * (D / 2); p += kThreads) {
            const int r = p / (D / 2), kk = p % (D / 2);
            const int i = r * D + (kk / h) * 2 * h + (kk % h);
            const float a = rq[i], b = rq[i + h];
            rq[i] = a + b;
            rq[i + h] = a - b;
        }
        __syncthreads();
    }
    constexpr float kScale = 0.125f;     // 2^-floor(log2(D)/2) for D = 128 and D = 64
    for (int i = threadIdx.x; i < 4 * D; i += kThreads) rq[i] *= kScale;
    __syncthreads();
}

// Full-precision window tokens of a bf16 ring with bf16 tensor-core MMAs,
// continuing a warp's online-softmax state (m, per-lane partial l, o in plain
// units; rows = channels 16 mt + gid (+8), columns = heads 2 tig + {0,1}).
// The window's positions [ng G, len) are cut into 16-token tiles; tile j goes
// to split j % n_split and, within it, to warp NW - 1 - (j / n_split) % NW
// (the last warps hold the fewest group pairs of a split).  A tile's
// rows are bulk-copied from their ring slots (pos % res_cap) into the warp's
// idle stream stage with a padded pitch (conflict-free ldmatrix); rows past the
// window's end are zeroed (their p is 0 and their V must be finite).
// S = K q (A = K rows, B = q in bf16), O^T += V^T P (A = V^T via
// ldmatrix.trans).  Returns false when a bounded wait gave up.
template <int D, typename TQ, bool ROT>
__device__ bool ring_tiles_mma(const KiviParams &P, int unit, int b, int split, int warp, int lane, const TQ *qg,
                               const float *rq, uint8_t *stage, uint64_t *bar, uint32_t phase, float (&m_run)[2],
                               float (&l_run)[2], float (&o)[D / 16][4])
{
    constexpr int KS = D / 16, PITCH = 2 * D + 16, TILE = 16 * PITCH, ROW = 2 * D;
    const int gid = lane >> 2, tig = lane & 3;
    const int len = P.seq_len[b];
    const int r0 = min(P.n_groups[b], P.max_groups) * G;
    const int r1 = min(len, r0 + P.res_cap);             // the window holds at most res_cap tokens
    const int ntile = r1 > r0 ? (r1 - r0 + 15) / 16 : 0;
    const int step = P.n_split_q * NW;
    int j = split + P.n_split_q * (NW - 1 - warp);
    if (j >= ntile) return true;
    uint32_t qb[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int c = 16 * ks + 2 * tig + 8 * rr;
            float a = 0.f, bb = 0.f;
            if (gid < P.grp) {
                a = ROT ? rq[gid * D + c] : load_q<TQ, D>(qg, gid * D + c);
                bb = ROT ? rq[gid * D + c + 1] : load_q<TQ, D>(qg, gid * D + c + 1);
            }
            qb[ks][rr] = pack_bf162(a, bb);
        }
    const uint8_t *kr = reinterpret_cast<const uint8_t *>(P.kres) + (size_t)unit * P.res_cap * ROW;
    const uint8_t *vr = reinterpret_cast<const uint8_t *>(P.vres) + (size_t)unit * P.res_cap * ROW;
    const int a_row = lane & 15, a_col = (lane >> 4) * 8;
    const int v_tok = (lane & 7) + ((lane >> 4) << 3), v_col = ((lane >> 3) & 1) * 8;
    for (; j < ntile; j += step) {
        const int t0 = r0 + 16 * j;
        const int rows = min(16, r1 - t0);
        if (lane >= rows && lane < 16) {
            uint4 *zk = reinterpret_cast<uint4 *>(stage + lane * PITCH);
            uint4 *zv = reinterpret_cast<uint4 *>(stage + TILE + lane * PITCH);
#pragma unroll
            for (int i = 0; i < ROW / 16; ++i) zk[i] = zv[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (lane == 0) mbar_arrive_expect_tx(bar, 2u * rows * ROW);
        __syncwarp();
        if (lane < rows) {
            const int slot = (t0 + lane) % P.res_cap;
            bulk_g2s(stage + lane * PITCH, kr + (size_t)slot * ROW, ROW, bar);
            bulk_g2s(stage + TILE + lane * PITCH, vr + (size_t)slot * ROW, ROW, bar);
        }
        if (!mbar_wait(bar, phase)) return false;
        phase ^= 1;
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, stage + a_row * PITCH + (16 * ks + a_col) * 2);
            mma16816_bf16(sc, a, qb[ks][0], qb[ks][1]);
        }
        float gmax[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool col_ok = 2 * tig + e < P.grp;
            sc[e] = (col_ok && gid < rows) ? sc[e] * P.qscale : kNegBig;
            sc[e + 2] = (col_ok && gid + 8 < rows) ? sc[e + 2] * P.qscale : kNegBig;
            if (P.raw && col_ok) {
                float *rw = P.raw + ((size_t)unit * P.raw_stride + t0 + gid) * 4 + 2 * tig + e;
                if (gid < rows) rw[0] = sc[e];
                if (gid + 8 < rows) rw[8 * 4] = sc[e + 2];
            }
            float mx = fmaxf(sc[e], sc[e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            gmax[e] = mx;
        }
        float alpha[2] = {1.f, 1.f};
#pragma unroll
        for (int e = 0; e < 2; ++e)
            if (gmax[e] > m_run[e] + kLazy) {
                alpha[e] = ex2(m_run[e] - gmax[e]);
                m_run[e] = gmax[e];
            }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= alpha[0];
                o[mt][1] *= alpha[1];
                o[mt][2] *= alpha[0];
                o[mt][3] *= alpha[1];
            }
            l_run[0] *= alpha[0];
            l_run[1] *= alpha[1];
        }
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = ex2(sc[i] - m_run[i & 1]);
        const uint32_t b0 = movmatrix_trans(pack_bf162(p[0], p[1]));
        const uint32_t b1 = movmatrix_trans(pack_bf162(p[2], p[3]));
        // the sum uses the bf16-rounded probabilities the MMA multiplies
        l_run[0] += __bfloat162float(__float2bfloat16_rn(p[0])) + __bfloat162float(__float2bfloat16_rn(p[2]));
        l_run[1] += __bfloat162float(__float2bfloat16_rn(p[1])) + __bfloat162float(__float2bfloat16_rn(p[3]));
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, stage + TILE + v_tok * PITCH + (16 * mt + v_col) * 2);
            mma16816_bf16(o[mt], a, b0, b1);
        }
        fence_async_smem();                      // this tile's reads before the next tile's bulk copies
        __syncwarp();
    }
    return true;
}

template <int BITS, int D, typename TQ, typename TR, bool ROT>
__global__ void __launch_bounds__(kThreads, 4)
draft_kivi_kernel(KiviParams P)
{
    if (!P.early_records) {
        pdl_wait();
        pdl_trigger();
    }
    using Gm = KiviGeom<BITS, D>;
    constexpr int KS = Gm::KS, NG = Gm::NG, REC = Gm::REC, NST = Gm::NST;
    constexpr int STAGE = 2 * REC;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);               // [NW][NST]
    uint8_t *ones = smem + 128;                                         // 4D bytes of fp16 1.0 (a K meta section)
    uint8_t *zeros = ones + 4 * D;                                      // 2D bytes of 0
    float *rq = reinterpret_cast<float *>(zeros + 2 * D);               // [4][D] rotated queries (ROT)
    uint8_t *ring = zeros + 2 * D + (ROT ? 16 * D : 0);                 // [NW][NST][2 records]
    float *wbuf = reinterpret_cast<float *>(ring);                      // reused after the loop

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int unit = blockIdx.x, split = blockIdx.y;   // long splits first, residual split last
    const int b = unit / P.Hkv, kvh = unit % P.Hkv;
    const int grp = P.grp;
    const int n_split = P.n_split_q + P.n_split_r;
    float *dst = P.part + ((size_t)unit * n_split + split) * part_floats(D);
    const TQ *qg = reinterpret_cast<const TQ *>(P.q) + ((size_t)b * P.Hq + kvh * grp) * D;

    for (int i = threadIdx.x; i < D; i += kThreads) reinterpret_cast<uint32_t *>(ones)[i] = kOnes;
    for (int i = threadIdx.x; i < D / 2; i += kThreads) reinterpret_cast<uint32_t *>(zeros)[i] = 0u;

    if (split < P.n_split_q) {
        // ---------------------------------------------- quantized groups --
        const int ng = min(P.n_groups[b], P.max_groups);
        // the unit's filled groups (often fewer than the capacity the split
        // count was planned for) are divided evenly over the splits, in pairs
        const int npairs = (ng + 1) / 2;
        const int g_lo = min(ng, 2 * (int)((long)npairs * split / P.n_split_q));
        const int g_hi = min(ng, 2 * (int)((long)npairs * (split + 1) / P.n_split_q));
        const uint8_t *rec_base = P.records + (size_t)unit * P.max_groups * REC;
        uint64_t *mybar = bars + warp * NST;
        uint8_t *myring = ring + (size_t)warp * NST * STAGE;
        const int n_pairs = (g_hi - g_lo + 1) / 2;
        const int n_mine = n_pairs > warp ? (n_pairs - warp + NW - 1) / NW : 0;
        // the records are read once per launch: evict-first, so they do not push
        // the partials, the window rows and this kernel's code out of L2
        const uint64_t rec_policy = l2_evict_first();
        auto issue = [&](int s, int it) {
            const int g = g_lo + 2 * (warp + it * NW);
            const uint32_t bytes = (g + 1 < g_hi ? 2 : 1) * REC;
            mbar_arrive_expect_tx(&mybar[s], bytes);
            bulk_g2s_hint(myring + s * STAGE, rec_base + (size_t)g * REC, bytes, &mybar[s], rec_policy);
        };
        // q first, as (c, c + 1) pairs (one 32-bit bf16 or 64-bit fp32 load
        // each when the unit's q rows are aligned for it): every warp's first
        // record copies, requested next, fill the memory system for a few
        // microseconds, and loads issued after them wait behind that traffic
        const int hq = gid & 3;
        const bool qvalid = hq < grp;
        const bool q_pairs = (reinterpret_cast<uintptr_t>(qg) & (2 * sizeof(TQ) - 1)) == 0;
        float2 qq[KS][2];
        auto load_qq = [&] {
            if constexpr (!ROT) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr)
                        qq[ks][rr] = qvalid ? load_q2<TQ, D>(qg, hq * D + 16 * ks + 2 * tig + 8 * rr, q_pairs)
                                            : make_float2(0.f, 0.f);
            }
        };
        auto first_copies = [&] {
            if (lane == 0) {
                for (int s = 0; s < NST; ++s) mbar_init(&mybar[s], 1);
                fence_mbar_init();
                for (int s = 0; s < NST && s < n_mine; ++s) issue(s, s);
            }
        };
        if (P.early_records) {
            // stable records: their first copies overlap the previous kernel's
            // end; q (written by it) after the wait
            first_copies();
            pdl_wait();
            pdl_trigger();
            load_qq();
        } else {
            load_qq();
            first_copies();
        }
        if constexpr (ROT) {
            rotate_queries<TQ, D>(qg, grp, rq);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int c = hq * D + 16 * ks + 2 * tig + 8 * rr;
                    qq[ks][rr] = qvalid ? make_float2(rq[c], rq[c + 1]) : make_float2(0.f, 0.f);
                }
        }
        // B fragments of q (column n = gid): heads 0..3 scaled by 2^(-b e) for
        // the channel's code exponent, copies 4..7 unscaled (zero-point sums)
        uint32_t qf[KS][2];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const float f = gid < 4 ? exp2f(-(float)(BITS * Pairs<BITS, D>::exp_of(2 * ks + rr))) : 1.f;
                const float a = qvalid ? qq[ks][rr].x * P.qscale * f : 0.f;
                const float bb = qvalid ? qq[ks][rr].y * P.qscale * f : 0.f;
                qf[ks][rr] = pack_half2(a, bb);
            }
        __syncthreads();                                  // ones / zeros written

        float m_run[2] = {kNegBig, kNegBig}, l_run[2] = {0.f, 0.f};
        float o_acc[KS][4];
#pragma unroll
        for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
        float vb_acc[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        for (int it = 0; it < n_mine; ++it) {
            const int st = it % NST;
            if (!mbar_wait(&mybar[st], (it / NST) & 1)) {
                if (lane == 0) report_timeout(P.status, 1);
                ok = false;
                break;
            }
            const int g = g_lo + 2 * (warp + it * NW);
            const bool two = g + 1 < g_hi;
            const uint8_t *recA = myring + st * STAGE;
            // a lone last group pairs with itself; its second copy is masked
            // out below (scores -inf, so it adds nothing to the values)
            const uint8_t *recB = two ? recA + REC : recA;
            // ---- scores of both groups (no branch between them, so their
            // instructions can interleave)
            float sc[2][2][4];
            group_scores<BITS, D>(recA, gid < 4 ? recA + Gm::KM : ones, qf, lane, tig, sc[0]);
            group_scores<BITS, D>(recB, gid < 4 ? recB + Gm::KM : ones, qf, lane, tig, sc[1]);
            if (!two) {
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) sc[1][mt][0] = sc[1][mt][1] = sc[1][mt][2] = sc[1][mt][3] = kNegBig;
            }
            if (P.raw && tig < 2) {
                // H2O: every visible score is kept for the mass pass after the merge
                float *rw = P.raw + ((size_t)unit * P.raw_stride + (size_t)g * G + gid) * 4;
#pragma unroll
                for (int G2 = 0; G2 < 2; ++G2)
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int h = 2 * tig + (i & 1);
                            if ((G2 == 0 || two) && h < grp)
                                rw[(G2 * G + 16 * mt + 8 * (i >> 1)) * 4 + h] = sc[G2][mt][i];
                        }
            }
            // ---- online softmax over the 64 tokens (exp2 domain, lazy rescale).
            // Each lane first takes the maximum of its own scores; the running
            // maximum of a column moves only when some score exceeds it by more
            // than kLazy (a factor 2^kLazy), and only then is the column maximum
            // reduced across the lanes (after the first groups of a split that
            // is rare).
            float lmax[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = kNegBig;
                if (2 * tig + e < grp) {
#pragma unroll
                    for (int G2 = 0; G2 < 2; ++G2)
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) mx = fmaxf(mx, fmaxf(sc[G2][mt][e], sc[G2][mt][e + 2]));
                } else {
                    // padding columns (head >= grp, or 4..7) stay at a finite floor
#pragma unroll
                    for (int G2 = 0; G2 < 2; ++G2)
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) sc[G2][mt][e] = sc[G2][mt][e + 2] = kNegBig;
                }
                lmax[e] = mx;
            }
            if (__any_sync(0xffffffffu, lmax[0] > m_run[0] + kLazy || lmax[1] > m_run[1] + kLazy)) {
                float alpha[2] = {1.f, 1.f};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float mx = lmax[e];
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    if (mx > m_run[e] + kLazy) {
                        alpha[e] = ex2(m_run[e] - mx);
                        m_run[e] = mx;
                    }
                }
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    o_acc[mt][0] *= alpha[0];
                    o_acc[mt][1] *= alpha[1];
                    o_acc[mt][2] *= alpha[0];
                    o_acc[mt][3] *= alpha[1];
                }
                vb_acc[0] *= alpha[0];
                vb_acc[1] *= alpha[1];
                vb_acc[2] *= alpha[0];
                vb_acc[3] *= alpha[1];
            }
            uint32_t pb[2][2][2];      // [group][token half][k half]
#pragma unroll
            for (int G2 = 0; G2 < 2; ++G2)
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const float2 m2 = make_float2(m_run[0], m_run[1]);
                    const float2 d01 = sub2(make_float2(sc[G2][mt][0], sc[G2][mt][1]), m2);
                    const float2 d23 = sub2(make_float2(sc[G2][mt][2], sc[G2][mt][3]), m2);
                    pb[G2][mt][0] = movmatrix_trans(pack_half2(ex2(d01.x), ex2(d01.y)));
                    pb[G2][mt][1] = movmatrix_trans(pack_half2(ex2(d23.x), ex2(d23.y)));
                }
            // ---- values of both groups (a masked copy has p = 0)
            {
                const uint8_t *zv_src = gid < NG ? recA + Gm::VM + 2 * D : zeros;
                group_values<BITS, D>(recA, zv_src, pb[0], lane, tig, o_acc, vb_acc);
            }
            {
                const uint8_t *zv_src = gid < NG ? recB + Gm::VM + 2 * D : zeros;
                group_values<BITS, D>(recB, zv_src, pb[1], lane, tig, o_acc, vb_acc);
            }
            fence_async_smem();                  // this stage's reads before its bulk refill
            __syncwarp();
            if (lane == 0 && it + NST < n_mine) issue(st, it + NST);
        }
        if (!ok) {
            // a bounded wait gave up: drop this warp's contribution
            m_run[0] = m_run[1] = kNegBig;
            l_run[0] = l_run[1] = 0.f;
#pragma unroll
            for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
            vb_acc[0] = vb_acc[1] = vb_acc[2] = vb_acc[3] = 0.f;
        }
        // the probability sums are rows 8..15 of the zero-point accumulator,
        // equal on every lane of a column: one lane per column keeps them, so
        // the lane reduction below counts them once
        l_run[0] = gid == 0 ? vb_acc[2] : 0.f;
        l_run[1] = gid == 0 ? vb_acc[3] : 0.f;
        // zero-point contribution of channel group gc for heads 2 tig + e
        // (row gc of the zero-point accumulator lives on lanes 4 gc + tig)
        float vbias[NG][2];
#pragma unroll
        for (int gc = 0; gc < NG; ++gc)
#pragma unroll
            for (int e = 0; e < 2; ++e) vbias[gc][e] = __shfl_sync(0xffffffffu, vb_acc[e], gc * 4 + tig);
        // o in plain units: rows 16 mt + gid (+8) lose 2^-24 and the code
        // factor 2^(b e) of their class and gain the zero-point sums
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const float f0 = kTwo24 * exp2f(-(float)(BITS * Pairs<BITS, D>::exp_of(2 * mt)));
            const float f1 = kTwo24 * exp2f(-(float)(BITS * Pairs<BITS, D>::exp_of(2 * mt + 1)));
            o_acc[mt][0] = fmaf(o_acc[mt][0], f0, vbias[mt / 2][0]);
            o_acc[mt][1] = fmaf(o_acc[mt][1], f0, vbias[mt / 2][1]);
            o_acc[mt][2] = fmaf(o_acc[mt][2], f1, vbias[mt / 2][0]);
            o_acc[mt][3] = fmaf(o_acc[mt][3], f1, vbias[mt / 2][1]);
        }
        if constexpr (std::is_same<TR, __nv_bfloat16>::value) {
            // the bf16 window's tiles of this split continue the same state
            // (stage 0 of the warp's stream ring has had (n_mine + 1) / 2 phases)
            if (ok && !ring_tiles_mma<D, TQ, ROT>(P, unit, b, split, warp, lane, qg, rq, myring, &mybar[0],
                                                  (uint32_t)((n_mine + 1) / 2) & 1u, m_run, l_run, o_acc)) {
                if (lane == 0) report_timeout(P.status, 2);
                m_run[0] = m_run[1] = kNegBig;
                l_run[0] = l_run[1] = 0.f;
#pragma unroll
                for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
            }
        }
        // lanes sharing a column hold partial row sums: reduce
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
            l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
            l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
        }
        __syncthreads();   // every warp done with its ring before wbuf reuse
        float *wm = wbuf, *wl = wbuf + NW * 4, *wo = wbuf + NW * 8;
        if (tig < 2) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * tig + e;
                if (gid == 0) {
                    wm[warp * 4 + h] = m_run[e];
                    wl[warp * 4 + h] = l_run[e];
                }
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    wo[(warp * 4 + h) * D + 16 * mt + gid] = o_acc[mt][e];
                    wo[(warp * 4 + h) * D + 16 * mt + gid + 8] = o_acc[mt][e + 2];
                }
            }
        }
        cta_merge_store<D>(wbuf, dst, grp);
        last_cta_combine<TQ, D>(P.part + (size_t)unit * n_split * part_floats(D), n_split,
                                P.counters + unit, grp,
                                reinterpret_cast<TQ *>(P.out) + ((size_t)b * P.Hq + kvh * grp) * D,
                                P.ml ? P.ml + (size_t)unit * 8 : nullptr);
    } else {
        // ------------------------------------- residual ring (fp32 SIMT) --
        if (P.early_records) {
            pdl_wait();
            pdl_trigger();
        }
        // Split r of the ring takes positions p0 + r * res_per_split onwards;
        // its rows are staged in shared memory (the idle stream ring) by bulk
        // copies, a chunk at a time, so the per-token math never waits on a
        // global load.
        const int len = P.seq_len[b];
        const int ng = min(P.n_groups[b], P.max_groups);
        const int r = split - P.n_split_q;
        const int t_lo = ng * G + r * P.res_per_split;
        const int t_hi = min(len, t_lo + P.res_per_split);
        constexpr int ROW = D * (int)sizeof(TR);
        constexpr int CHUNK = (NW * Gm::NST * 2 * Gm::REC) / (2 * ROW);
        static_assert(CHUNK >= NW, "the stream ring stages at least one token per warp");
        const uint8_t *kr = reinterpret_cast<const uint8_t *>(P.kres) + (size_t)unit * P.res_cap * ROW;
        const uint8_t *vr = reinterpret_cast<const uint8_t *>(P.vres) + (size_t)unit * P.res_cap * ROW;
        const TR *ksm = reinterpret_cast<const TR *>(ring);
        const TR *vsm = reinterpret_cast<const TR *>(ring + CHUNK * ROW);
        uint64_t *resbar = bars;
        if (threadIdx.x == 0) {
            mbar_init(resbar, 1);
            fence_mbar_init();
        }
        constexpr int CPL = D / 32;          // channels per lane
        if constexpr (ROT) rotate_queries<TQ, D>(qg, grp, rq);
        float qv[4][CPL];
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int i = 0; i < CPL; ++i)
                qv[h][i] = h < grp ? (ROT ? rq[h * D + lane * CPL + i] : load_q<TQ, D>(qg, h * D + lane * CPL + i)) *
                                         P.qscale
                                   : 0.f;
        float m[4], l[4], o[4][CPL];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            m[h] = kNegBig;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[h][i] = 0.f;
        }
        int phase = 0;
        for (int t0 = t_lo; t0 < t_hi; t0 += CHUNK) {
            const int nt = min(CHUNK, t_hi - t0);
            fence_async_smem();                  // the previous chunk's reads before the refill
            __syncthreads();                     // the staging bytes are free (and the barrier is set up)
            if (threadIdx.x == 0) {
                mbar_arrive_expect_tx(resbar, 2u * nt * ROW);
                // positions t0 .. t0 + nt - 1 sit at ring slots pos % res_cap:
                // at most two contiguous runs
                int done = 0, pos = t0;
                while (done < nt) {
                    const int slot = pos % P.res_cap;
                    const int run = min(nt - done, P.res_cap - slot);
                    bulk_g2s(ring + done * ROW, kr + (size_t)slot * ROW, run * ROW, resbar);
                    bulk_g2s(ring + (CHUNK + done) * ROW, vr + (size_t)slot * ROW, run * ROW, resbar);
                    done += run;
                    pos += run;
                }
            }
            const bool got = mbar_wait(resbar, phase);
            phase ^= 1;
            if (!got) report_timeout(P.status, 2);
            if (!__syncthreads_and(got)) {      // uniform exit; the split contributes nothing
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    m[h] = kNegBig;
                    l[h] = 0.f;
#pragma unroll
                    for (int i = 0; i < CPL; ++i) o[h][i] = 0.f;
                }
                break;
            }
            for (int t = warp; t < nt; t += NW) {
                float kx[CPL], vx[CPL];
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    kx[i] = Elem<TR>::to_f(ksm[t * D + lane * CPL + i]);
                    vx[i] = Elem<TR>::to_f(vsm[t * D + lane * CPL + i]);
                }
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float sdot = 0.f;
#pragma unroll
                    for (int i = 0; i < CPL; ++i) sdot = fmaf(qv[h][i], kx[i], sdot);
                    sdot = warp_sum(sdot);
                    if (P.raw && lane == 0 && h < grp)
                        P.raw[((size_t)unit * P.raw_stride + t0 + t) * 4 + h] = sdot;
                    const float mn = fmaxf(m[h], sdot);
                    const float a = exp2f(m[h] - mn), pp = exp2f(sdot - mn);
                    m[h] = mn;
                    l[h] = l[h] * a + pp;
#pragma unroll
                    for (int i = 0; i < CPL; ++i) o[h][i] = o[h][i] * a + pp * vx[i];
                }
            }
        }
        __syncthreads();
        float *wm = wbuf, *wl = wbuf + NW * 4, *wo = wbuf + NW * 8;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if (lane == 0) {
                wm[warp * 4 + h] = m[h];
                wl[warp * 4 + h] = l[h];
            }
#pragma unroll
            for (int i = 0; i < CPL; ++i) wo[(warp * 4 + h) * D + lane * CPL + i] = o[h][i];
        }
        cta_merge_store<D>(wbuf, dst, grp);
        last_cta_combine<TQ, D>(P.part + (size_t)unit * n_split * part_floats(D), n_split,
                                P.counters + unit, grp,
                                reinterpret_cast<TQ *>(P.out) + ((size_t)b * P.Hq + kvh * grp) * D,
                                P.ml ? P.ml + (size_t)unit * 8 : nullptr);
    }
}

// ----------------------------------------------------------- dense kernel --
// 32-token tiles of K and V staged by two bulk copies (rows of a (b, h) are
// contiguous); lane = token for scores, lane = channel slice for values.
constexpr int DENSE_NST = 2;

struct DenseParams {
    const void *q, *k, *v;
    const int32_t *seq_len;
    float *part;
    unsigned int *counters;                            // [units], zero between calls
    void *out;
    int32_t *status;
    int Hkv, Hq, grp, L_stride, n_split, tiles_per_split;
    float qscale;
    float *raw;                                        // optional [units][max_len][4] log2-domain scores
    float *ml;                                         // optional [units][8]: final max, sum per head
    int max_len;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
draft_dense_kernel(DenseParams P)
{
    pdl_wait();
    pdl_trigger();
    constexpr int TILE = G * D * sizeof(T);
    constexpr int CPL = D / 32;
    constexpr int PER = 16 / sizeof(T);
    constexpr int NCH = D / PER;
    constexpr int QSTR = 4 * PER + 4;        // padded stride of a channel chunk
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    float *qs = reinterpret_cast<float *>(smem + 128);                  // [NCH][4][PER] (+pad)
    uint8_t *ring = smem + 128 + NCH * QSTR * 4;                         // [NW][NST][2][TILE]
    float *wbuf = reinterpret_cast<float *>(ring);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.y, split = blockIdx.x;
    const int b = unit / P.Hkv, kvh = unit % P.Hkv;
    const int grp = P.grp;
    float *dst = P.part + ((size_t)unit * P.n_split + split) * part_floats(D);
    const T *qg = reinterpret_cast<const T *>(P.q) + ((size_t)b * P.Hq + kvh * grp) * D;
    for (int i = threadIdx.x; i < 4 * D; i += kThreads) {
        const int h = i / D, c = i % D;
        qs[(c / PER) * QSTR + h * PER + c % PER] = h < grp ? Elem<T>::to_f(qg[i]) * P.qscale : 0.f;
    }
    const int len = P.seq_len[b];
    const int ntile = (len + G - 1) / G;
    const int t_lo = split * P.tiles_per_split, t_hi = min(ntile, t_lo + P.tiles_per_split);
    const T *kb = reinterpret_cast<const T *>(P.k) + (size_t)unit * P.L_stride * D;
    const T *vb = reinterpret_cast<const T *>(P.v) + (size_t)unit * P.L_stride * D;
    uint64_t *mybar = bars + warp * DENSE_NST;
    uint8_t *myring = ring + (size_t)warp * DENSE_NST * 2 * TILE;
    if (lane == 0)
        for (int s = 0; s < DENSE_NST; ++s) mbar_init(&mybar[s], 1);
    fence_mbar_init();
    __syncthreads();

    const int n_mine = t_hi > t_lo + warp ? (t_hi - t_lo - warp + NW - 1) / NW : 0;
    auto issue = [&](int s, int tile) {
        const int rows = min(G, len - tile * G);
        const uint32_t bytes = rows * D * sizeof(T);
        mbar_arrive_expect_tx(&mybar[s], 2 * bytes);
        bulk_g2s(myring + (2 * s) * TILE, kb + (size_t)tile * G * D, bytes, &mybar[s]);
        bulk_g2s(myring + (2 * s + 1) * TILE, vb + (size_t)tile * G * D, bytes, &mybar[s]);
    };
    if (lane == 0)
        for (int s = 0; s < DENSE_NST && s < n_mine; ++s) issue(s, t_lo + warp + s * NW);

    float m[4], l[4], o[4][CPL];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        m[h] = kNegBig;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) o[h][i] = 0.f;
    }
    bool ok = true;
    for (int it = 0; it < n_mine; ++it) {
        const int st = it % DENSE_NST;
        const int tile = t_lo + warp + it * NW;
        if (!mbar_wait(&mybar[st], (it / DENSE_NST) & 1)) {
            if (lane == 0) report_timeout(P.status, 2);
            ok = false;
            break;
        }
        const T *kt = reinterpret_cast<const T *>(myring + (2 * st) * TILE);
        const T *vt = reinterpret_cast<const T *>(myring + (2 * st + 1) * TILE);
        const int rows = min(G, len - tile * G);
        // scores: lane = token; rotate the channel order by lane to spread banks
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        if (lane < rows) {
            for (int jj = 0; jj < NCH; ++jj) {
                const int j = (jj + lane) % NCH;
                uint4 u = *reinterpret_cast<const uint4 *>(kt + lane * D + j * PER);
                float x[PER];
                if constexpr (sizeof(T) == 2) {
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) { x[2 * e] = bf16_lo(w[e]); x[2 * e + 1] = bf16_hi(w[e]); }
                } else {
                    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
                    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
                }
                const float *qj = qs + j * QSTR;
#pragma unroll
                for (int h = 0; h < 4; ++h)
#pragma unroll
                    for (int e = 0; e < PER; ++e) s[h] = fmaf(qj[h * PER + e], x[e], s[h]);
            }
        }
        float p[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float sv = lane < rows ? s[h] : kNegBig;
            const float mx = warp_max(sv);
            const float mn = fmaxf(m[h], mx);
            const float a = exp2f(m[h] - mn);
            p[h] = lane < rows ? exp2f(sv - mn) : 0.f;
            m[h] = mn;
            l[h] = l[h] * a + warp_sum(p[h]);
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[h][i] *= a;
        }
        // values: lane = channel slice, loop over the tile's tokens
        for (int t = 0; t < rows; ++t) {
            float vx[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) vx[i] = Elem<T>::to_f(vt[t * D + lane * CPL + i]);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float ph = __shfl_sync(0xffffffffu, p[h], t);
#pragma unroll
                for (int i = 0; i < CPL; ++i) o[h][i] = fmaf(ph, vx[i], o[h][i]);
            }
        }
        fence_async_smem();                      // this stage's reads before its bulk refill
        __syncwarp();
        if (lane == 0 && it + DENSE_NST < n_mine) issue(st, t_lo + warp + (it + DENSE_NST) * NW);
    }
    if (!ok) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            m[h] = kNegBig;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[h][i] = 0.f;
        }
    }
    __syncthreads();
    float *wm = wbuf, *wl = wbuf + NW * 4, *wo = wbuf + NW * 8;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        if (lane == 0) {
            wm[warp * 4 + h] = m[h];
            wl[warp * 4 + h] = l[h];
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) wo[(warp * 4 + h) * D + lane * CPL + i] = o[h][i];
    }
    cta_merge_store<D>(wbuf, dst, grp);
    last_cta_combine<T, D>(P.part + (size_t)unit * P.n_split * part_floats(D), P.n_split, P.counters + unit, grp,
                           reinterpret_cast<T *>(P.out) + ((size_t)b * P.Hq + kvh * grp) * D);
}

// ------------------------------------------------- dense kernel, bf16 MMA --
// bf16 caches: the same per-warp ring and online softmax as the KIVI kernel,
// with the K and V tiles themselves as MMA operands.  A warp takes 16-token
// tiles; each row arrives by its own bulk copy into a padded shared-memory
// row (pitch D*2 + 16 bytes), so the ldmatrix reads below are free of bank
// conflicts.  S = K q (A = K rows via ldmatrix, B = q), P moves to the B
// layout with movmatrix, O^T += V^T P (A = V^T via ldmatrix.trans).
constexpr int DM_TOK = 16;                    // tokens per tile
constexpr int DM_NST = 2;                     // ring stages per warp

template <int D>
struct DmGeom {
    static constexpr int PITCH = D * 2 + 16;
    static constexpr int TILE = DM_TOK * PITCH;              // one K or V tile
    static constexpr int STAGE = 2 * TILE;
    static constexpr int RING = NW * DM_NST * STAGE;
    static constexpr int SMEM = 128 + RING;                  // barriers + rings (merge buffer reuses the rings)
};

template <int D>
__global__ void __launch_bounds__(kThreads)
draft_dense_mma_kernel(DenseParams P)
{
    pdl_wait();
    pdl_trigger();
    using Gm = DmGeom<D>;
    constexpr int KS = D / 16;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *ring = smem + 128;
    float *wbuf = reinterpret_cast<float *>(ring);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int unit = blockIdx.y, split = blockIdx.x;
    const int b = unit / P.Hkv, kvh = unit % P.Hkv;
    const int grp = P.grp;
    float *dst = P.part + ((size_t)unit * P.n_split + split) * part_floats(D);
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(P.q) + ((size_t)b * P.Hq + kvh * grp) * D;
    // stale rows of a partial last tile must hold finite values (their p is 0)
    for (int i = threadIdx.x; i < Gm::RING / 16; i += kThreads) reinterpret_cast<uint4 *>(ring)[i] = make_uint4(0, 0, 0, 0);
    // B fragments of q: column n = gid is head gid (zero for gid >= grp)
    uint32_t qf[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int c = 16 * ks + 2 * tig + 8 * rr;
            if (gid < grp)
                qf[ks][rr] = *reinterpret_cast<const uint32_t *>(qg + gid * D + c);
            else
                qf[ks][rr] = 0u;
        }
    const int len = P.seq_len[b];
    const int ntile = (len + DM_TOK - 1) / DM_TOK;
    const int t_lo = split * P.tiles_per_split, t_hi = min(ntile, t_lo + P.tiles_per_split);
    const __nv_bfloat16 *kb = reinterpret_cast<const __nv_bfloat16 *>(P.k) + (size_t)unit * P.L_stride * D;
    const __nv_bfloat16 *vb = reinterpret_cast<const __nv_bfloat16 *>(P.v) + (size_t)unit * P.L_stride * D;
    uint64_t *mybar = bars + warp * DM_NST;
    uint8_t *myring = ring + (size_t)warp * DM_NST * Gm::STAGE;
    if (lane == 0)
        for (int s = 0; s < DM_NST; ++s) mbar_init(&mybar[s], 1);
    fence_mbar_init();
    __syncthreads();

    const int n_mine = t_hi > t_lo + warp ? (t_hi - t_lo - warp + NW - 1) / NW : 0;
    auto issue = [&](int s, int tile) {          // all lanes: lane t copies token row t (t < 16)
        const int rows = min(DM_TOK, len - tile * DM_TOK);
        if (lane == 0) mbar_arrive_expect_tx(&mybar[s], 2 * rows * D * 2);
        __syncwarp();
        if (lane < rows) {
            uint8_t *d0 = myring + s * Gm::STAGE + lane * Gm::PITCH;
            const size_t row = (size_t)tile * DM_TOK + lane;
            bulk_g2s(d0, kb + row * D, D * 2, &mybar[s]);
            bulk_g2s(d0 + Gm::TILE, vb + row * D, D * 2, &mybar[s]);
        }
    };
    for (int s = 0; s < DM_NST && s < n_mine; ++s) issue(s, t_lo + warp + s * NW);

    float m_run[2] = {kNegBig, kNegBig}, l_run[2] = {0.f, 0.f};
    float o_acc[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    bool ok = true;
    // ldmatrix lane addressing
    const int a_row = lane & 15, a_col = (lane >> 4) * 8;                       // K tile (non-transposed)
    const int v_tok = (lane & 7) + ((lane >> 4) << 3), v_col = ((lane >> 3) & 1) * 8;   // V tile (transposed)
    for (int it = 0; it < n_mine; ++it) {
        const int st = it % DM_NST;
        const int tile = t_lo + warp + it * NW;
        if (!mbar_wait(&mybar[st], (it / DM_NST) & 1)) {
            if (lane == 0) report_timeout(P.status, 4);
            ok = false;
            break;
        }
        const uint8_t *kt = myring + st * Gm::STAGE;
        const uint8_t *vt = kt + Gm::TILE;
        const int rows = min(DM_TOK, len - tile * DM_TOK);
        // ---- scores: rows = tokens gid, gid + 8; columns = heads 2 tig, 2 tig + 1
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, kt + a_row * Gm::PITCH + (16 * ks + a_col) * 2);
            mma16816_bf16(sc, a, qf[ks][0], qf[ks][1]);
        }
        float gmax[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool col_ok = 2 * tig + e < grp;
            sc[e] = (col_ok && gid < rows) ? sc[e] * P.qscale : kNegBig;
            sc[e + 2] = (col_ok && gid + 8 < rows) ? sc[e + 2] * P.qscale : kNegBig;
            if (P.raw && col_ok) {
                // H2O: keep every visible score for the mass pass after the combine
                float *rw = P.raw + ((size_t)unit * P.max_len + (size_t)tile * DM_TOK + gid) * 4 + 2 * tig + e;
                if (gid < rows) rw[0] = sc[e];
                if (gid + 8 < rows) rw[8 * 4] = sc[e + 2];
            }
            float mx = fmaxf(sc[e], sc[e + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            gmax[e] = mx;
        }
        float alpha[2] = {1.f, 1.f};
#pragma unroll
        for (int e = 0; e < 2; ++e)
            if (gmax[e] > m_run[e] + kLazy) {
                alpha[e] = ex2(m_run[e] - gmax[e]);
                m_run[e] = gmax[e];
            }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o_acc[mt][0] *= alpha[0];
                o_acc[mt][1] *= alpha[1];
                o_acc[mt][2] *= alpha[0];
                o_acc[mt][3] *= alpha[1];
            }
            l_run[0] *= alpha[0];
            l_run[1] *= alpha[1];
        }
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = ex2(sc[i] - m_run[i & 1]);
        const uint32_t b0 = movmatrix_trans(pack_bf162(p[0], p[1]));
        const uint32_t b1 = movmatrix_trans(pack_bf162(p[2], p[3]));
        // the sum uses the bf16-rounded probabilities the MMA multiplies
        l_run[0] += __bfloat162float(__float2bfloat16_rn(p[0])) + __bfloat162float(__float2bfloat16_rn(p[2]));
        l_run[1] += __bfloat162float(__float2bfloat16_rn(p[1])) + __bfloat162float(__float2bfloat16_rn(p[3]));
        // ---- values: O^T[channel][head] += V^T P
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, vt + v_tok * Gm::PITCH + (16 * mt + v_col) * 2);
            mma16816_bf16(o_acc[mt], a, b0, b1);
        }
        fence_async_smem();                      // this stage's reads before its bulk refill
        __syncwarp();
        if (it + DM_NST < n_mine) issue(st, t_lo + warp + (it + DM_NST) * NW);
    }
    if (!ok) {
        m_run[0] = m_run[1] = kNegBig;
        l_run[0] = l_run[1] = 0.f;
#pragma unroll
        for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
        l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
        l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
    }
    __syncthreads();   // every warp done with its ring before wbuf reuse
    float *wm = wbuf, *wl = wbuf + NW * 4, *wo = wbuf + NW * 8;
    if (tig < 2) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * tig + e;
            if (gid == 0) {
                wm[warp * 4 + h] = m_run[e];
                wl[warp * 4 + h] = l_run[e];
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                wo[(warp * 4 + h) * D + 16 * mt + gid] = o_acc[mt][e];
                wo[(warp * 4 + h) * D + 16 * mt + gid + 8] = o_acc[mt][e + 2];
            }
        }
    }
    cta_merge_store<D>(wbuf, dst, grp);
    last_cta_combine<__nv_bfloat16, D>(P.part + (size_t)unit * P.n_split * part_floats(D), P.n_split,
                                       P.counters + unit, grp,
                                       reinterpret_cast<__nv_bfloat16 *>(P.out) + ((size_t)b * P.Hq + kvh * grp) * D,
                                       P.ml ? P.ml + (size_t)unit * 8 : nullptr);
}

// H2O mass pass: scores[unit][pos] += sum over the unit's query heads of
// softmax probability of cached token j (pos = kept_idx[unit][j], or j), from
// the stored log2-domain scores and each head's final max and sum.
__global__ void h2o_accumulate_kernel(const float *__restrict__ raw, const float *__restrict__ ml,
                                      const int32_t *__restrict__ seq_len, int max_len, int Hkv, int grp,
                                      const int32_t *__restrict__ kept_idx, int kept_stride, float *scores,
                                      int scores_stride)
{
    const int unit = blockIdx.y, b = unit / Hkv;
    const int len = min(seq_len[b], max_len);
    float M[4], invL[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        M[h] = ml[unit * 8 + h];
        const float L = ml[unit * 8 + 4 + h];
        invL[h] = (h < grp && L > 0.f) ? 1.f / L : 0.f;
    }
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < len; j += gridDim.x * blockDim.x) {
        const float4 r = *reinterpret_cast<const float4 *>(raw + ((size_t)unit * max_len + j) * 4);
        const float rv[4] = {r.x, r.y, r.z, r.w};
        float mass = 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h)
            if (h < grp) mass += exp2f(rv[h] - M[h]) * invL[h];
        const int pos = kept_idx ? kept_idx[(size_t)unit * kept_stride + j] : j;
        scores[(size_t)unit * scores_stride + pos] += mass;
    }
}

// ----------------------------------------------------------------- host ----
int num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

struct KiviPlan {
    int n_split_q, groups_per_split, n_split_r, res_per_split;
};

constexpr int kResTokensPerSplit = 256;

KiviPlan kivi_plan(const vc_qcache *c)
{
    const int units = c->B * c->Hkv;
    const int ng = c->max_groups;
    const int sms = num_sms();
    KiviPlan p;
    if (c->res_dtype == VC_BF16) {
        // The bf16 window is handled inside the quantized splits (tensor-core
        // tiles), so every CTA is a quantized split.  Split count minimising
        // waves x (group pairs per warp + ~3 pairs of fixed cost per CTA) /
        // the last wave's fill: full waves of equal CTAs keep every SM busy
        // to the end (measured at 32k: 9 splits for 64 kv units, 576 CTAs in
        // one wave of 608 slots; 9 for 128 units).
        p.n_split_r = 0;
        p.res_per_split = 0;
        const int slots = sms * 4;                     // 4 resident CTAs per SM
        int best = 1;
        double best_t = -1.0;
        const int max_s = ng > 0 ? std::min(kMaxSplit, (ng + 3) / 4) : 1;   // at least two group pairs per split
        for (int s = 1; s <= max_s; ++s) {
            int gps = (ng + s - 1) / s;
            gps += gps & 1;
            const int se = ng > 0 ? (ng + gps - 1) / gps : 1;
            const int pairs_per_warp = (gps / 2 + NW - 1) / NW;
            const long n_cta = (long)units * se;
            const long waves = (n_cta + slots - 1) / slots;
            const double fill = (double)n_cta / ((double)waves * slots);
            const double t = (double)waves * (pairs_per_warp + 3) / fill;
            if (best_t < 0.0 || t < best_t) {
                best_t = t;
                best = s;
            }
        }
        p.groups_per_split = ng > 0 ? (ng + best - 1) / best : 2;
        p.groups_per_split += p.groups_per_split & 1;
        p.n_split_q = ng > 0 ? (ng + p.groups_per_split - 1) / p.groups_per_split : 1;
        return p;
    }
    const int slots = sms * 4;                         // 4 resident CTAs per SM
    // the fp32 ring: one split per 256 of its capacity's tokens
    p.n_split_r = std::max(1, std::min(kMaxSplit / 2, (c->res_cap + kResTokensPerSplit - 1) / kResTokensPerSplit));
    p.res_per_split = (c->res_cap + p.n_split_r - 1) / p.n_split_r;
    // Split count minimising waves x (group pairs per warp + ~3 pairs of
    // fixed cost per CTA) for CTAs of equal length; the ring splits are more
    // CTAs per kv unit.
    int best = 1;
    long best_t = -1;
    const int max_s = ng > 0 ? (ng + 3) / 4 : 1;       // at least two group pairs per split
    for (int s = 1; s <= max_s && s + p.n_split_r <= kMaxSplit; ++s) {
        int gps = (ng + s - 1) / s;
        gps += gps & 1;
        const int se = ng > 0 ? (ng + gps - 1) / gps : 0;
        const int pairs_per_warp = (gps / 2 + NW - 1) / NW;
        const long waves = ((long)units * (se + p.n_split_r) + slots - 1) / slots;
        const long t = waves * (pairs_per_warp + 3);
        if (best_t < 0 || t < best_t) {
            best_t = t;
            best = s;
        }
    }
    p.groups_per_split = ng > 0 ? (ng + best - 1) / best : 2;
    p.groups_per_split += p.groups_per_split & 1;       // whole pairs
    p.n_split_q = ng > 0 ? (ng + p.groups_per_split - 1) / p.groups_per_split : 0;
    return p;
}

struct DensePlan {
    int n_split, tiles_per_split;
};

DensePlan dense_plan(const vc_cache_view *v)
{
    const int units = v->B * v->Hkv;
    DensePlan p;
    if (v->dt == VC_BF16) {
        // bf16 MMA kernel: split count minimising waves x (tiles per warp + ~4
        // tiles of fixed cost) for CTAs of equal length, 3 CTAs per SM
        const int nt = (v->max_len + DM_TOK - 1) / DM_TOK;
        const int slots = num_sms() * 3;
        int best = 1;
        long best_t = -1;
        for (int s = 1; s <= kMaxSplit && s <= (nt + NW - 1) / NW; ++s) {
            const int per = (nt + s - 1) / s;
            const int se = (nt + per - 1) / per;
            const long waves = ((long)units * se + slots - 1) / slots;
            const long t = waves * ((per + NW - 1) / NW + 4);
            if (best_t < 0 || t < best_t) {
                best_t = t;
                best = se;
            }
        }
        p.tiles_per_split = nt > 0 ? (nt + best - 1) / best : 1;
        p.n_split = nt > 0 ? (nt + p.tiles_per_split - 1) / p.tiles_per_split : 1;
        return p;
    }
    const int nt = (v->max_len + G - 1) / G;
    const int target_ctas = num_sms() * 4 * 2;
    int s = (target_ctas + units - 1) / units;
    const int max_s = (nt + NW - 1) / NW;
    if (s > max_s) s = max_s;
    if (s > kMaxSplit) s = kMaxSplit;
    if (s < 1) s = 1;
    p.tiles_per_split = nt > 0 ? (nt + s - 1) / s : 1;
    p.n_split = nt > 0 ? (nt + p.tiles_per_split - 1) / p.tiles_per_split : 1;
    return p;
}

// Tokens a KIVI cache can hold per kv unit (the H2O score rows).
inline int kivi_token_cap(const vc_qcache *c) { return c->max_groups * G + c->res_cap; }

template <int BITS, int D, typename TQ, typename TR, bool ROT>
cudaError_t launch_kivi(const void *q, const vc_qcache *c, int Hq, float scale, void *out, void *ws,
                        cudaStream_t st, float *raw = nullptr, float *ml = nullptr, bool early = false)
{
    using Gm = KiviGeom<BITS, D>;
    const KiviPlan pl = kivi_plan(c);
    KiviParams P;
    P.raw = raw;
    P.ml = ml;
    P.raw_stride = kivi_token_cap(c);
    P.q = q;
    P.records = (const uint8_t *)c->records;
    P.kres = c->k_res;
    P.vres = c->v_res;
    P.n_groups = c->n_groups;
    P.seq_len = c->seq_len;
    P.status = (int32_t *)ws;
    P.counters = (unsigned int *)((uint8_t *)ws + kStatusBytes);
    P.part = (float *)((uint8_t *)ws + kStatusBytes + align256((size_t)c->B * c->Hkv * 4));
    P.out = out;
    P.Hkv = c->Hkv;
    P.Hq = Hq;
    P.grp = Hq / c->Hkv;
    P.max_groups = c->max_groups;
    P.res_cap = c->res_cap;
    P.n_split_q = pl.n_split_q;
    P.n_split_r = pl.n_split_r;
    P.res_per_split = pl.res_per_split;
    P.qscale = scale * kLog2e;
    P.early_records = early ? 1 : 0;
    const size_t rot_bytes = ROT ? 16 * D : 0;
    size_t smem = 128 + 6 * D + rot_bytes + (size_t)NW * Gm::NST * 2 * Gm::REC;
    const size_t merge = 128 + 6 * D + rot_bytes + (size_t)merge_floats(D) * 4;
    if (smem < merge) smem = merge;
    auto kern = draft_kivi_kernel<BITS, D, TQ, TR, ROT>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(c->B * c->Hkv, pl.n_split_q + pl.n_split_r);
    return launch_pdl(kern, grid, dim3(kThreads), smem, st, P);
}

template <typename T, int D>
cudaError_t launch_dense(const void *q, const vc_cache_view *v, int Hq, float scale, void *out,
                         void *ws, cudaStream_t st, float *raw = nullptr, float *ml = nullptr)
{
    const DensePlan pl = dense_plan(v);
    DenseParams P;
    P.raw = raw;
    P.ml = ml;
    P.max_len = v->max_len;
    P.q = q;
    P.k = v->k;
    P.v = v->v;
    P.seq_len = v->seq_len;
    P.status = (int32_t *)ws;
    P.counters = (unsigned int *)((uint8_t *)ws + kStatusBytes);
    P.part = (float *)((uint8_t *)ws + kStatusBytes + align256((size_t)v->B * v->Hkv * 4));
    P.out = out;
    P.Hkv = v->Hkv;
    P.Hq = Hq;
    P.grp = Hq / v->Hkv;
    P.L_stride = v->L_stride;
    P.n_split = pl.n_split;
    P.tiles_per_split = pl.tiles_per_split;
    P.qscale = scale * kLog2e;
    if constexpr (sizeof(T) == 2) {
        using Gm = DmGeom<D>;
        size_t smem = Gm::SMEM;
        const size_t merge = 128 + (size_t)merge_floats(D) * 4;
        if (smem < merge) smem = merge;
        auto kern = draft_dense_mma_kernel<D>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        dim3 grid(pl.n_split, v->B * v->Hkv);
        return launch_pdl(kern, grid, dim3(kThreads), smem, st, P);
    }
    constexpr int PER = 16 / sizeof(T);
    const size_t qbytes = (size_t)(D / PER) * (4 * PER + 4) * 4;
    size_t smem = 128 + qbytes + (size_t)NW * DENSE_NST * 2 * G * D * sizeof(T);
    const size_t merge = 128 + qbytes + (size_t)merge_floats(D) * 4;
    if (smem < merge) smem = merge;
    auto kern = draft_dense_kernel<T, D>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(pl.n_split, v->B * v->Hkv);
    return launch_pdl(kern, grid, dim3(kThreads), smem, st, P);
}

template <int BITS, int D, typename TQ>
cudaError_t kivi_by_res(const void *q, const vc_qcache *c, int Hq, float s, void *o, void *ws,
                        cudaStream_t st, float *raw = nullptr, float *ml = nullptr, bool early = false)
{
    if (c->cfg.rotate)
        return c->res_dtype == VC_BF16
                   ? launch_kivi<BITS, D, TQ, __nv_bfloat16, true>(q, c, Hq, s, o, ws, st, raw, ml, early)
                   : launch_kivi<BITS, D, TQ, float, true>(q, c, Hq, s, o, ws, st, raw, ml, early);
    return c->res_dtype == VC_BF16
               ? launch_kivi<BITS, D, TQ, __nv_bfloat16, false>(q, c, Hq, s, o, ws, st, raw, ml, early)
               : launch_kivi<BITS, D, TQ, float, false>(q, c, Hq, s, o, ws, st, raw, ml, early);
}

template <int D, typename TQ>
cudaError_t kivi_by_bits(const void *q, const vc_qcache *c, int Hq, float s, void *o, void *ws,
                         cudaStream_t st, float *raw = nullptr, float *ml = nullptr, bool early = false)
{
    return c->cfg.bits == 2 ? kivi_by_res<2, D, TQ>(q, c, Hq, s, o, ws, st, raw, ml, early)
                            : kivi_by_res<4, D, TQ>(q, c, Hq, s, o, ws, st, raw, ml, early);
}

}  // namespace

size_t draft_h2o_ws_bytes(const vc_cache_view *view, int Hq)
{
    if (view->kind == VC_CACHE_KIVI) {
        const vc_qcache *c = view->kivi;
        return draft_ws_bytes(view, Hq) + align256((size_t)c->B * c->Hkv * 8 * 4) +
               align256((size_t)c->B * c->Hkv * kivi_token_cap(c) * 4 * 4);
    }
    return draft_ws_bytes(view, Hq) + align256((size_t)view->B * view->Hkv * 8 * 4) +
           align256((size_t)view->B * view->Hkv * view->max_len * 4 * 4);
}

size_t draft_ws_bytes(const vc_cache_view *view, int Hq)
{
    (void)Hq;
    if (view->kind == VC_CACHE_KIVI) {
        const vc_qcache *c = view->kivi;
        const KiviPlan p = kivi_plan(c);
        return kStatusBytes + align256((size_t)c->B * c->Hkv * 4) +
               align256((size_t)c->B * c->Hkv * (p.n_split_q + p.n_split_r) * part_floats(c->d) * 4);
    }
    const DensePlan p = dense_plan(view);
    return kStatusBytes + align256((size_t)view->B * view->Hkv * 4) +
           align256((size_t)view->B * view->Hkv * p.n_split * part_floats(view->d) * 4);
}

cudaError_t draft_attn(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq,
                       float sm_scale, void *out, void *ws, cudaStream_t st)
{
    if (view->kind == VC_CACHE_KIVI) {
        const vc_qcache *c = view->kivi;
        const bool early = (view->flags & VC_VIEW_RECORDS_STABLE) != 0;
        if (c->d == 128)
            return q_dt == VC_BF16 ? kivi_by_bits<128, __nv_bfloat16>(q, c, Hq, sm_scale, out, ws, st, nullptr, nullptr, early)
                                   : kivi_by_bits<128, float>(q, c, Hq, sm_scale, out, ws, st, nullptr, nullptr, early);
        return q_dt == VC_BF16 ? kivi_by_bits<64, __nv_bfloat16>(q, c, Hq, sm_scale, out, ws, st, nullptr, nullptr, early)
                               : kivi_by_bits<64, float>(q, c, Hq, sm_scale, out, ws, st, nullptr, nullptr, early);
    }
    if (view->d == 128)
        return view->dt == VC_BF16 ? launch_dense<__nv_bfloat16, 128>(q, view, Hq, sm_scale, out, ws, st)
                                   : launch_dense<float, 128>(q, view, Hq, sm_scale, out, ws, st);
    return view->dt == VC_BF16 ? launch_dense<__nv_bfloat16, 64>(q, view, Hq, sm_scale, out, ws, st)
                               : launch_dense<float, 64>(q, view, Hq, sm_scale, out, ws, st);
}

}  // namespace vc

namespace vc {

cudaError_t draft_attn_h2o(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq, float sm_scale,
                           void *out, float *scores, int scores_stride, const int32_t *kept_idx, int kept_stride,
                           void *ws, cudaStream_t st)
{
    uint8_t *base = (uint8_t *)ws;
    if (view->kind == VC_CACHE_KIVI) {
        // quantized records and ring: scores stored by the draft kernel itself
        const vc_qcache *c = view->kivi;
        const size_t main_ws = draft_ws_bytes(view, Hq);
        float *ml = (float *)(base + main_ws);
        float *raw = (float *)(base + main_ws + align256((size_t)c->B * c->Hkv * 8 * 4));
        cudaError_t e;
        if (c->d == 128)
            e = q_dt == VC_BF16 ? kivi_by_bits<128, __nv_bfloat16>(q, c, Hq, sm_scale, out, ws, st, raw, ml)
                                : kivi_by_bits<128, float>(q, c, Hq, sm_scale, out, ws, st, raw, ml);
        else
            e = q_dt == VC_BF16 ? kivi_by_bits<64, __nv_bfloat16>(q, c, Hq, sm_scale, out, ws, st, raw, ml)
                                : kivi_by_bits<64, float>(q, c, Hq, sm_scale, out, ws, st, raw, ml);
        if (e != cudaSuccess) return e;
        const int units = c->B * c->Hkv;
        const int cap = kivi_token_cap(c);
        const int blocks = std::max(1, std::min(64, (cap + 255) / 256));
        h2o_accumulate_kernel<<<dim3(blocks, units), 256, 0, st>>>(raw, ml, c->seq_len, cap, c->Hkv, Hq / c->Hkv,
                                                                   kept_idx, kept_stride, scores, scores_stride);
        return cudaGetLastError();
    }
    const size_t main_ws = draft_ws_bytes(view, Hq);
    float *ml = (float *)(base + main_ws);
    float *raw = (float *)(base + main_ws + align256((size_t)view->B * view->Hkv * 8 * 4));
    const cudaError_t e = view->d == 128
                              ? launch_dense<__nv_bfloat16, 128>(q, view, Hq, sm_scale, out, ws, st, raw, ml)
                              : launch_dense<__nv_bfloat16, 64>(q, view, Hq, sm_scale, out, ws, st, raw, ml);
    if (e != cudaSuccess) return e;
    const int units = view->B * view->Hkv;
    const int blocks = std::max(1, std::min(64, (view->max_len + 255) / 256));
    h2o_accumulate_kernel<<<dim3(blocks, units), 256, 0, st>>>(raw, ml, view->seq_len, view->max_len, view->Hkv,
                                                               Hq / view->Hkv, kept_idx, kept_stride, scores,
                                                               scores_stride);
    return cudaGetLastError();
}

}  // namespace vc
