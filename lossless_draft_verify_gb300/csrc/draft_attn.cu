// draft_attn.cu -- single-query decode attention over the compressed draft
// cache (VeriCache drafts on the compressed cache; drafting is
// HBM-bandwidth-bound, paper page "What the paper found").
//
// KIVI cache kernel.  Grid = (split, kv unit); each CTA streams a contiguous
// range of 32-token group records through per-warp shared-memory rings filled
// by cp.async.bulk (one bulk copy per record, mbarrier completion).  A warp
// owns whole groups and computes, for the Hq/Hkv <= 4 query heads of its kv
// head, the scores and the weighted values with m16n8k16 tensor-core MMAs on
// the integer codes themselves: the per-channel K scale is folded into the
// query (q' = q * s), the per-token V scale into the probabilities
// (p' = p * s), and the zero-points enter through two small MMAs whose
// operands are the padding columns 4..7 of the head dimension (n = 8).  Codes
// are turned into exact fp16 integers with one shift + one LOP3 per pair
// (1024 + code), the 1024 offset being cancelled exactly for K through the
// same MMA (sum of q') and subtracted with HSUB2 for V.  Online softmax in the
// exp2 domain with lazy rescaling.  The residual (full-precision ring) is one
// extra split handled with fp32 CUDA-core math.  A combine kernel merges the
// split partials.
//
// Dense cache kernel (compacted dropped cache, or an uncompressed cache):
// fp32 CUDA-core math over 32-token tiles staged by cp.async.bulk.
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

// ---------------------------------------------------------------- PTX ----
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

constexpr uint32_t kMagic = 0x64006400u;   // half2(1024, 1024)
constexpr uint32_t kOnes = 0x3C003C00u;    // half2(1, 1)

template <int BITS>
__device__ __forceinline__ uint32_t unpack_pair(const uint32_t *words, int p)
{
    constexpr int P = 16 / BITS;
    constexpr uint32_t mask = BITS == 2 ? 0x00030003u : 0x000F000Fu;
    return lop3_and_or(words[p / P] >> (BITS * (p % P)), mask, kMagic);
}

// ------------------------------------------------------------ KIVI kernel --
template <int BITS, int D>
struct KiviGeom {
    static constexpr int KS = D / 16;                  // QK k-steps, PV m-tiles
    static constexpr int NG = D / 32;                  // V channel groups
    static constexpr int CODE_BYTES = G * D * BITS / 8;
    static constexpr int WPL = G * D / 32 * BITS / 32; // code words per lane per section
    static constexpr int KM = 2 * CODE_BYTES;          // K meta offset
    static constexpr int VM = KM + 4 * D;              // V meta offset
    static constexpr int REC = VM + 4 * D;             // record bytes
    static constexpr int NSTAGE = REC <= 3072 ? 4 : 3;
};

struct KiviParams {
    const void *q;
    const uint8_t *records;
    const void *kres, *vres;
    const int32_t *n_groups, *seq_len;
    float *part;
    int32_t *status;
    int Hkv, Hq, grp, max_groups, res_cap, n_split_q, groups_per_split;
    float qscale;                                      // sm_scale * log2(e)
};

template <typename TQ, int D>
__device__ __forceinline__ float load_q(const TQ *q, int idx) { return Elem<TQ>::to_f(q[idx]); }

// Merge the NW warps' (m, l, o) of this CTA in shared memory and store the
// CTA partial.  Every warp has written wm[w][h], wl[w][h], wo[w][h][c].
template <int D>
__device__ void cta_merge_store(float *wbuf, float *dst, int grp)
{
    __syncthreads();
    float *wm = wbuf;                       // [NW][4]
    float *wl = wbuf + NW * 4;              // [NW][4]
    float *wo = wbuf + NW * 8;              // [NW][4][D]
    for (int i = threadIdx.x; i < 4 * D; i += kThreads) {
        const int h = i / D;
        float M = kNegBig;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * 4 + h]);
        float o = 0.f;
        for (int w = 0; w < NW; ++w) o += wo[(w * 4 + h) * D + (i % D)] * exp2f(wm[w * 4 + h] - M);
        dst[8 + i] = h < grp ? o : 0.f;
    }
    if (threadIdx.x < 4) {
        const int h = threadIdx.x;
        float M = kNegBig, L = 0.f;
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * 4 + h]);
        for (int w = 0; w < NW; ++w) L += wl[w * 4 + h] * exp2f(wm[w * 4 + h] - M);
        dst[h] = M;
        dst[4 + h] = h < grp ? L : 0.f;
    }
}

template <int BITS, int D, typename TQ, typename TR>
__global__ void __launch_bounds__(kThreads, 3)
draft_kivi_kernel(KiviParams P)
{
    using Gm = KiviGeom<BITS, D>;
    constexpr int KS = Gm::KS, NG = Gm::NG, REC = Gm::REC, NST = Gm::NSTAGE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);               // [NW][NST]
    uint8_t *ring = smem + 128;                                         // [NW][NST][REC]
    float *wbuf = reinterpret_cast<float *>(smem + 128);                // reused after the loop

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int unit = blockIdx.y, split = blockIdx.x;
    const int b = unit / P.Hkv, kvh = unit % P.Hkv;
    const int grp = P.grp;
    float *dst = P.part + ((size_t)unit * (P.n_split_q + 1) + split) * part_floats(D);

    // per-lane online-softmax state for columns 2*tig, 2*tig+1
    float m_run[2] = {kNegBig, kNegBig}, l_run[2] = {0.f, 0.f};
    float o_acc[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    float vb_acc[4] = {0.f, 0.f, 0.f, 0.f};

    const TQ *qg = reinterpret_cast<const TQ *>(P.q) + ((size_t)b * P.Hq + kvh * grp) * D;

    if (split < P.n_split_q) {
        // ---------------------------------------------- quantized groups --
        const int ng = min(P.n_groups[b], P.max_groups);
        const int g_lo = split * P.groups_per_split;
        const int g_hi = min(ng, g_lo + P.groups_per_split);
        const uint8_t *rec_base = P.records + (size_t)unit * P.max_groups * REC;
        uint64_t *mybar = bars + warp * NST;
        uint8_t *myring = ring + (size_t)warp * NST * REC;
        // B fragments of q (columns n = gid; 0..3 real heads, 4..7 copies)
        uint32_t qf[KS][2];
        {
            const int h = gid & 3;
            const bool valid = h < grp;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int c = 16 * ks + 2 * tig + 8 * rr;
                    float a = valid ? load_q<TQ, D>(qg, h * D + c) * P.qscale : 0.f;
                    float bb = valid ? load_q<TQ, D>(qg, h * D + c + 1) * P.qscale : 0.f;
                    qf[ks][rr] = pack_half2(a, bb);
                }
        }
        if (lane == 0)
            for (int s = 0; s < NST; ++s) mbar_init(&mybar[s], 1);
        fence_mbar_init();
        __syncwarp();
        const int n_mine = g_hi > g_lo + warp ? (g_hi - g_lo - warp + NW - 1) / NW : 0;
        if (lane == 0)
            for (int s = 0; s < NST && s < n_mine; ++s) {
                const int g = g_lo + warp + s * NW;
                mbar_arrive_expect_tx(&mybar[s], REC);
                bulk_g2s(myring + s * REC, rec_base + (size_t)g * REC, REC, &mybar[s]);
            }
        bool ok = true;
        for (int it = 0; it < n_mine; ++it) {
            const int st = it % NST;
            if (!mbar_wait(&mybar[st], (it / NST) & 1)) {
                if (lane == 0) report_timeout(P.status, 1);
                ok = false;
                break;
            }
            const uint8_t *rec = myring + st * REC;
            const uint32_t *kmeta = reinterpret_cast<const uint32_t *>(rec + Gm::KM + tig * D);
            const uint32_t *vmeta = reinterpret_cast<const uint32_t *>(rec + Gm::VM + tig * D);

            // ---- scores: S = codes * q' (+ zero/offset bias) ----------------
            float cb[4] = {0.f, 0.f, 0.f, 0.f};
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                uint32_t kw[Gm::WPL];
                const uint4 *src = reinterpret_cast<const uint4 *>(rec) + lane * (Gm::WPL / 4);
#pragma unroll
                for (int i = 0; i < Gm::WPL / 4; ++i) {
                    uint4 u = src[i];
                    kw[4 * i] = u.x; kw[4 * i + 1] = u.y; kw[4 * i + 2] = u.z; kw[4 * i + 3] = u.w;
                }
                uint32_t ks_pair[2 * KS], kz_pair[2 * KS];
#pragma unroll
                for (int i = 0; i < 2 * KS; i += 4) {
                    uint4 u = *reinterpret_cast<const uint4 *>(kmeta + i);
                    ks_pair[i] = u.x; ks_pair[i + 1] = u.y; ks_pair[i + 2] = u.z; ks_pair[i + 3] = u.w;
                    uint4 z = *reinterpret_cast<const uint4 *>(kmeta + D / 8 + i);
                    kz_pair[i] = z.x; kz_pair[i + 1] = z.y; kz_pair[i + 2] = z.z; kz_pair[i + 3] = z.w;
                }
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t bq[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr)
                        bq[rr] = gid < 4 ? hmul2(qf[ks][rr], ks_pair[2 * ks + rr]) : qf[ks][rr];
                    // bias rows: row 0 = ones (sum of q'), row 1 = z (sum of z*q)
                    uint32_t ab[4];
                    ab[0] = gid == 0 ? kOnes : (gid == 1 ? kz_pair[2 * ks] : 0u);
                    ab[1] = 0u;
                    ab[2] = gid == 0 ? kOnes : (gid == 1 ? kz_pair[2 * ks + 1] : 0u);
                    ab[3] = 0u;
                    mma16816(cb, ab, bq[0], bq[1]);
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        uint32_t a[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) a[r] = unpack_pair<BITS>(kw, (mt * KS + ks) * 4 + r);
                        mma16816(sc[mt], a, bq[0], bq[1]);
                    }
                }
            }
            // bias for columns 2*tig + e (valid for tig < 2)
            float bias[2];
            {
                const int t1 = tig & 1;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float sq = __shfl_sync(0xffffffffu, cb[e], t1);
                    const float zq = __shfl_sync(0xffffffffu, cb[e], 6 + t1);
                    bias[e] = zq - 1024.f * sq;
                }
            }
            // ---- online softmax (exp2 domain) ---------------------------------
            float gmax[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                // padding columns (head >= grp, or 4..7) are pinned to a finite
                // floor so they never trigger a rescale and stay finite
                if (2 * tig + e >= grp) {
                    sc[0][e] = sc[0][e + 2] = sc[1][e] = sc[1][e + 2] = kNegBig;
                    bias[e] = 0.f;
                }
                float x = sc[0][e] + bias[e];
                sc[0][e] = x;
                float y = sc[0][e + 2] + bias[e];
                sc[0][e + 2] = y;
                float z = sc[1][e] + bias[e];
                sc[1][e] = z;
                float w = sc[1][e + 2] + bias[e];
                sc[1][e + 2] = w;
                float mx = fmaxf(fmaxf(x, y), fmaxf(z, w));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                gmax[e] = mx;
            }
            float alpha[2] = {1.f, 1.f};
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (gmax[e] > m_run[e] + kLazy) {
                    alpha[e] = exp2f(m_run[e] - gmax[e]);
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
                // zero-point accumulator columns 4+h live on lanes tig = 2 + h/2
                const float a0 = __shfl_sync(0xffffffffu, alpha[0], lane ^ 2);
                const float a1 = __shfl_sync(0xffffffffu, alpha[1], lane ^ 2);
                vb_acc[0] *= a0;
                vb_acc[1] *= a1;
                vb_acc[2] *= a0;
                vb_acc[3] *= a1;
            }
            uint32_t pb[2][2];          // B fragments of P^T per token half (ks) and k half
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                float p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = exp2f(sc[mt][i] - m_run[i & 1]);
                l_run[0] += p[0] + p[2];
                l_run[1] += p[1] + p[3];
                pb[mt][0] = movmatrix_trans(pack_half2(p[0], p[1]));
                pb[mt][1] = movmatrix_trans(pack_half2(p[2], p[3]));
                // columns 4..7 carry the unscaled p of heads 0..3
                pb[mt][0] = __shfl_sync(0xffffffffu, pb[mt][0], lane & 15);
                pb[mt][1] = __shfl_sync(0xffffffffu, pb[mt][1], lane & 15);
            }
            // ---- values: O += codes^T * p' (+ zero-point bias) ---------------
            {
                uint32_t vw[Gm::WPL];
                const uint4 *src = reinterpret_cast<const uint4 *>(rec + Gm::CODE_BYTES) + lane * (Gm::WPL / 4);
#pragma unroll
                for (int i = 0; i < Gm::WPL / 4; ++i) {
                    uint4 u = src[i];
                    vw[4 * i] = u.x; vw[4 * i + 1] = u.y; vw[4 * i + 2] = u.z; vw[4 * i + 3] = u.w;
                }
                uint32_t sv[2][2][NG];
#pragma unroll
                for (int i = 0; i < 4 * NG; i += 4) {
                    uint4 u = *reinterpret_cast<const uint4 *>(vmeta + i);
                    uint32_t *f = &sv[0][0][0];
                    f[i] = u.x; f[i + 1] = u.y; f[i + 2] = u.z; f[i + 3] = u.w;
                }
                // zero-point rows gc = gid (< NG): pairs (ks, rr) of channel group gid
                uint32_t zv[2][2];
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr)
                        zv[ks][rr] = gid < NG ? vmeta[D / 8 + (2 * ks + rr) * NG + gid] : 0u;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t az[4] = {zv[ks][0], 0u, zv[ks][1], 0u};
                    mma16816(vb_acc, az, pb[ks][0], pb[ks][1]);
#pragma unroll
                    for (int gc = 0; gc < NG; ++gc) {
                        const uint32_t b0 = gid < 4 ? hmul2(pb[ks][0], sv[ks][0][gc]) : pb[ks][0];
                        const uint32_t b1 = gid < 4 ? hmul2(pb[ks][1], sv[ks][1][gc]) : pb[ks][1];
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int mt = 2 * gc + half;
                            uint32_t a[4];
#pragma unroll
                            for (int r = 0; r < 4; ++r)
                                a[r] = hsub2(unpack_pair<BITS>(vw, (mt * 2 + ks) * 4 + r), kMagic);
                            mma16816(o_acc[mt], a, b0, b1);
                        }
                    }
                }
            }
            __syncwarp();
            // refill this stage with the group NST iterations ahead
            if (lane == 0 && it + NST < n_mine) {
                const int g = g_lo + warp + (it + NST) * NW;
                mbar_arrive_expect_tx(&mybar[st], REC);
                bulk_g2s(myring + st * REC, rec_base + (size_t)g * REC, REC, &mybar[st]);
            }
        }
        if (!ok) {
            // a bounded wait gave up: drop this warp's contribution
            m_run[0] = m_run[1] = kNegBig;
            l_run[0] = l_run[1] = 0.f;
#pragma unroll
            for (int i = 0; i < KS; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
            vb_acc[0] = vb_acc[1] = vb_acc[2] = vb_acc[3] = 0.f;
        }
        // finish per-warp state: reduce l over lanes sharing a column
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
            l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
            l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
        }
        // zero-point contribution of channel group gc for heads 2*tig+e
        float vbias[NG][2];
#pragma unroll
        for (int gc = 0; gc < NG; ++gc)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                vbias[gc][e] = __shfl_sync(0xffffffffu, vb_acc[e], gc * 4 + (tig & 1) + 2);
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
                    const int c0 = 16 * mt + gid;
                    wo[(warp * 4 + h) * D + c0] = o_acc[mt][e] + vbias[mt / 2][e];
                    wo[(warp * 4 + h) * D + c0 + 8] = o_acc[mt][e + 2] + vbias[mt / 2][e];
                }
            }
        }
        cta_merge_store<D>(wbuf, dst, grp);
    } else {
        // ------------------------------------- residual ring (fp32 SIMT) --
        const int len = P.seq_len[b];
        const int ng = min(P.n_groups[b], P.max_groups);
        const int p0 = ng * G;
        const TR *kr = reinterpret_cast<const TR *>(P.kres) + (size_t)unit * P.res_cap * D;
        const TR *vr = reinterpret_cast<const TR *>(P.vres) + (size_t)unit * P.res_cap * D;
        constexpr int CPL = D / 32;          // channels per lane
        float qv[4][CPL];
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int i = 0; i < CPL; ++i)
                qv[h][i] = h < grp ? load_q<TQ, D>(qg, h * D + lane * CPL + i) * P.qscale : 0.f;
        float m[4], l[4], o[4][CPL];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            m[h] = kNegBig;
            l[h] = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[h][i] = 0.f;
        }
        for (int pos = p0 + warp; pos < len; pos += NW) {
            const size_t slot = (size_t)(pos % P.res_cap) * D + lane * CPL;
            float kx[CPL], vx[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                kx[i] = Elem<TR>::to_f(kr[slot + i]);
                vx[i] = Elem<TR>::to_f(vr[slot + i]);
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) s = fmaf(qv[h][i], kx[i], s);
                s = warp_sum(s);
                const float mn = fmaxf(m[h], s);
                const float a = exp2f(m[h] - mn), p = exp2f(s - mn);
                m[h] = mn;
                l[h] = l[h] * a + p;
#pragma unroll
                for (int i = 0; i < CPL; ++i) o[h][i] = o[h][i] * a + p * vx[i];
            }
        }
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
    int32_t *status;
    int Hkv, Hq, grp, L_stride, n_split, tiles_per_split;
    float qscale;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
draft_dense_kernel(DenseParams P)
{
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
}

// --------------------------------------------------------------- combine --
template <typename TQ, int D>
__global__ void combine_kernel(const float *__restrict__ part, int n_split, int Hkv, int Hq,
                               int grp, TQ *__restrict__ out)
{
    const int unit = blockIdx.x;
    const int b = unit / Hkv, kvh = unit % Hkv;
    const float *pp = part + (size_t)unit * n_split * part_floats(D);
    for (int i = threadIdx.x; i < grp * D; i += blockDim.x) {
        const int h = i / D, c = i % D;
        float M = kNegBig;
        for (int s = 0; s < n_split; ++s) M = fmaxf(M, pp[(size_t)s * part_floats(D) + h]);
        float L = 0.f, O = 0.f;
        for (int s = 0; s < n_split; ++s) {
            const float *q = pp + (size_t)s * part_floats(D);
            const float w = exp2f(q[h] - M);
            L += q[4 + h] * w;
            O += q[8 + h * D + c] * w;
        }
        out[((size_t)b * Hq + kvh * grp + h) * D + c] = Elem<TQ>::from_f(L > 0.f ? O / L : 0.f);
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
    int n_split_q, groups_per_split;
};

KiviPlan kivi_plan(const vc_qcache *c)
{
    const int units = c->B * c->Hkv;
    const int ng = c->max_groups;
    const int target_ctas = num_sms() * 3 * 2;
    int s = (target_ctas + units - 1) / units;
    s = s < 1 ? 1 : s;
    const int max_s = (ng + NW * 2 - 1) / (NW * 2);    // keep >= 2 groups per warp
    if (s > max_s) s = max_s > 0 ? max_s : 1;
    KiviPlan p;
    p.groups_per_split = ng > 0 ? (ng + s - 1) / s : 1;
    p.n_split_q = ng > 0 ? (ng + p.groups_per_split - 1) / p.groups_per_split : 0;
    return p;
}

struct DensePlan {
    int n_split, tiles_per_split;
};

DensePlan dense_plan(const vc_cache_view *v)
{
    const int units = v->B * v->Hkv;
    const int nt = (v->max_len + G - 1) / G;
    const int target_ctas = num_sms() * 4 * 2;
    int s = (target_ctas + units - 1) / units;
    const int max_s = (nt + NW - 1) / NW;
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    DensePlan p;
    p.tiles_per_split = nt > 0 ? (nt + s - 1) / s : 1;
    p.n_split = nt > 0 ? (nt + p.tiles_per_split - 1) / p.tiles_per_split : 1;
    return p;
}

template <int BITS, int D, typename TQ, typename TR>
cudaError_t launch_kivi(const void *q, const vc_qcache *c, int Hq, float scale, void *out, void *ws,
                        cudaStream_t st)
{
    using Gm = KiviGeom<BITS, D>;
    const KiviPlan pl = kivi_plan(c);
    KiviParams P;
    P.q = q;
    P.records = (const uint8_t *)c->records;
    P.kres = c->k_res;
    P.vres = c->v_res;
    P.n_groups = c->n_groups;
    P.seq_len = c->seq_len;
    P.status = (int32_t *)ws;
    P.part = (float *)((uint8_t *)ws + kStatusBytes);
    P.Hkv = c->Hkv;
    P.Hq = Hq;
    P.grp = Hq / c->Hkv;
    P.max_groups = c->max_groups;
    P.res_cap = c->res_cap;
    P.n_split_q = pl.n_split_q;
    P.groups_per_split = pl.groups_per_split;
    P.qscale = scale * kLog2e;
    size_t smem = 128 + (size_t)NW * Gm::NSTAGE * Gm::REC;
    const size_t merge = (size_t)NW * part_floats(D) * 4;
    if (smem < 128 + merge) smem = 128 + merge;
    auto kern = draft_kivi_kernel<BITS, D, TQ, TR>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(pl.n_split_q + 1, c->B * c->Hkv);
    kern<<<grid, kThreads, smem, st>>>(P);
    combine_kernel<TQ, D><<<c->B * c->Hkv, 256, 0, st>>>(P.part, pl.n_split_q + 1, c->Hkv, Hq,
                                                         P.grp, (TQ *)out);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_dense(const void *q, const vc_cache_view *v, int Hq, float scale, void *out,
                         void *ws, cudaStream_t st)
{
    const DensePlan pl = dense_plan(v);
    DenseParams P;
    P.q = q;
    P.k = v->k;
    P.v = v->v;
    P.seq_len = v->seq_len;
    P.status = (int32_t *)ws;
    P.part = (float *)((uint8_t *)ws + kStatusBytes);
    P.Hkv = v->Hkv;
    P.Hq = Hq;
    P.grp = Hq / v->Hkv;
    P.L_stride = v->L_stride;
    P.n_split = pl.n_split;
    P.tiles_per_split = pl.tiles_per_split;
    P.qscale = scale * kLog2e;
    constexpr int PER = 16 / sizeof(T);
    const size_t qbytes = (size_t)(D / PER) * (4 * PER + 4) * 4;
    size_t smem = 128 + qbytes + (size_t)NW * DENSE_NST * 2 * G * D * sizeof(T);
    const size_t merge = 128 + qbytes + (size_t)NW * part_floats(D) * 4;
    if (smem < merge) smem = merge;
    auto kern = draft_dense_kernel<T, D>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(pl.n_split, v->B * v->Hkv);
    kern<<<grid, kThreads, smem, st>>>(P);
    combine_kernel<T, D><<<v->B * v->Hkv, 256, 0, st>>>(P.part, pl.n_split, v->Hkv, Hq, P.grp,
                                                       (T *)out);
    return cudaGetLastError();
}

template <int BITS, int D, typename TQ>
cudaError_t kivi_by_res(const void *q, const vc_qcache *c, int Hq, float s, void *o, void *ws,
                        cudaStream_t st)
{
    return c->res_dtype == VC_BF16 ? launch_kivi<BITS, D, TQ, __nv_bfloat16>(q, c, Hq, s, o, ws, st)
                                   : launch_kivi<BITS, D, TQ, float>(q, c, Hq, s, o, ws, st);
}

template <int D, typename TQ>
cudaError_t kivi_by_bits(const void *q, const vc_qcache *c, int Hq, float s, void *o, void *ws,
                         cudaStream_t st)
{
    return c->cfg.bits == 2 ? kivi_by_res<2, D, TQ>(q, c, Hq, s, o, ws, st)
                            : kivi_by_res<4, D, TQ>(q, c, Hq, s, o, ws, st);
}

}  // namespace

size_t draft_ws_bytes(const vc_cache_view *view, int Hq)
{
    (void)Hq;
    if (view->kind == VC_CACHE_KIVI) {
        const vc_qcache *c = view->kivi;
        const KiviPlan p = kivi_plan(c);
        return kStatusBytes +
               align256((size_t)c->B * c->Hkv * (p.n_split_q + 1) * part_floats(c->d) * 4);
    }
    const DensePlan p = dense_plan(view);
    return kStatusBytes + align256((size_t)view->B * view->Hkv * p.n_split * part_floats(view->d) * 4);
}

cudaError_t draft_attn(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq,
                       float sm_scale, void *out, void *ws, cudaStream_t st)
{
    if (view->kind == VC_CACHE_KIVI) {
        const vc_qcache *c = view->kivi;
        if (c->d == 128)
            return q_dt == VC_BF16 ? kivi_by_bits<128, __nv_bfloat16>(q, c, Hq, sm_scale, out, ws, st)
                                   : kivi_by_bits<128, float>(q, c, Hq, sm_scale, out, ws, st);
        return q_dt == VC_BF16 ? kivi_by_bits<64, __nv_bfloat16>(q, c, Hq, sm_scale, out, ws, st)
                               : kivi_by_bits<64, float>(q, c, Hq, sm_scale, out, ws, st);
    }
    if (view->d == 128)
        return view->dt == VC_BF16 ? launch_dense<__nv_bfloat16, 128>(q, view, Hq, sm_scale, out, ws, st)
                                   : launch_dense<float, 128>(q, view, Hq, sm_scale, out, ws, st);
    return view->dt == VC_BF16 ? launch_dense<__nv_bfloat16, 64>(q, view, Hq, sm_scale, out, ws, st)
                               : launch_dense<float, 64>(q, view, Hq, sm_scale, out, ws, st);
}

}  // namespace vc
