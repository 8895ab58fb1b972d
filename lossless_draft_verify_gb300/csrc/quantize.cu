// quantize.cu -- KIVI-style asymmetric group quantization of the draft cache
// (KIVI: a compressor named on the VeriCache paper page, "What the paper
// found"; ref [42] on pith.science).  K per channel over groups of 32 tokens,
// V per token over groups of 32 channels, fp16 scale and zero-point per group,
// packed into the record layout the draft kernel consumes (include/vc.h).
//
// One CTA of 2*d threads quantizes one (sequence, kv head, token group):
// the group's 32 K rows and 32 V rows are staged in shared memory with
// 16-byte loads; d/2 threads reduce the min/max of K channel pairs and d
// threads those of the V (token, 32-channel group) rows, each deriving the
// directed-rounded fp16 meta and the reciprocal of its scale once; then
// every thread assembles whole 32-bit code words of the record (the words one
// draft-kernel lane reads, in fragment order) in registers, with no atomics,
// and the record leaves with 128-bit stores.  The quotient (x - z)/s is
// evaluated with the reciprocal and recomputed with an exact IEEE division
// whenever it lies within rounding distance of a half-integer, so the codes
// are those of the correctly rounded quotient.  HBM-bound: reads 2*32*d*2
// bytes, writes one record per group.
#include <algorithm>

#include <cooperative_groups.h>

#include "vc_common.cuh"
#include "vc_internal.h"

namespace cg = cooperative_groups;

namespace vc {
namespace {

constexpr int G = 32;

// RU(a / m) for finite a >= 0 and a small integer m: the smallest float y
// with y * m >= a (the definition of rounding upward).  The estimate a * (1/m)
// is within two ulps (three steps allow for a binade edge); each FMA computes
// y * m - a with one rounding, so its
// sign is that of the exact difference and the steps land on the answer.
__device__ __forceinline__ float div_ru_small(float a, float m, float inv_m)
{
    float y = a * inv_m;
#pragma unroll
    for (int k = 0; k < 3; ++k)
        if (fmaf(y, m, -a) < 0.0f) y = __uint_as_float(__float_as_uint(y) + 1u);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const float p = __uint_as_float(__float_as_uint(y) - 1u);
        if (y > 0.0f && fmaf(p, m, -a) >= 0.0f) y = p;
    }
    return y;
}

// Directed-rounding quantization parameters of one group (see include/vc.h).
__device__ __forceinline__ void group_params(float mn, float mx, int qmax, uint16_t &sb,
                                             uint16_t &zb, float &sf, float &zf)
{
    __half z = __float2half_rd(mn);
    zf = __half2float(z);
    float range = __fadd_ru(mx, -zf);
    float step = div_ru_small(range, (float)qmax, 1.0f / (float)qmax);
    __half s = __float2half_ru(step);
    sf = __half2float(s);
    sb = __half_as_ushort(s);
    zb = __half_as_ushort(z);
}

// Approximate reciprocal of a scale (at most 1 ulp off); the code logic
// below tolerates it.
__device__ __forceinline__ float rcp_scale(float s)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
    return s != 0.0f ? r : 0.0f;
}

// all ones when |e| lies above the near-half threshold, else zero
__device__ __forceinline__ uint32_t near_mask(float e, float thr)
{
    uint32_t m;
    asm("set.gt.u32.f32 %0, %1, %2;" : "=r"(m) : "f"(fabsf(e)), "f"(thr));
    return m;
}

// code = clamp(rint(RN(RN(x - z) / s)), 0, qmax).  The codes are first taken
// from q = RN(x - z) * rcp(s), rounded to an integer by adding 1.5 * 2^23
// (round to nearest, ties to even).  q lies within 2^-17 of RN(d / s) for
// q <= 15, so whenever q is farther than kNearHalf from a half-integer both
// round to the same integer; the codes nearer than that are recomputed from
// the exact quotient.  d >= 0 and d / s <= qmax by the choice of z and s, so
// no clamp is needed on either path.
constexpr float kRoundMagic = 12582912.0f;
constexpr float kNearHalf = 0.5f - 0x1p-15f;

__device__ __noinline__ uint32_t exact_code(float x, float zf, float sf)
{
    return (uint32_t)rintf(__fdiv_rn(__fadd_rn(x, -zf), sf));
}

// Position of code pair (kappa, mu) inside a lane's words (see include/vc.h).
template <int BITS, int D>
__device__ __forceinline__ void pair_pos(int kappa, int mu, int &word, int &slot)
{
    constexpr int W = D * BITS / 32;
    if (BITS == 2) {
        constexpr int h = W / 2, q = W / 4;
        if (kappa < 3 * h) {
            word = 2 * (kappa % h) + mu / 2;
            slot = kappa / h + 5 * (mu % 2);
        } else {
            const int k2 = kappa - 3 * h;
            word = 4 * (k2 % q) + mu;
            slot = 3 + k2 / q;
        }
    } else {
        constexpr int h = W / 2;
        word = 2 * (kappa % h) + mu / 2;
        slot = kappa / h + 2 * (mu % 2);
    }
}

// byte offset of word w of lane l in a code section
__device__ __forceinline__ int word_byte(int lane, int w) { return 16 * (32 * (w >> 2) + lane) + 4 * (w & 3); }

template <int BITS, int D>
struct RecGeom {
    static constexpr int CODE = G * D * BITS / 8;   // bytes per code section
    static constexpr int KM = 2 * CODE;
    static constexpr int VM = KM + 4 * D;
    static constexpr int REC = VM + 4 * D;
};

// ------------------------------------------------------------------------
// Staged quantizer.  The group's 32 K rows and 32 V rows are copied
// into shared memory with 16-byte loads; the scale, zero-point and reciprocal
// of every K channel and every V (token, channel group) are computed once;
// then each thread assembles whole 32-bit code words of the record (the words
// a draft-kernel lane reads) in registers, with no shared-memory atomics, and
// the finished record leaves with 128-bit stores.
// ------------------------------------------------------------------------

template <typename T, int BITS, int D>
struct QStage {
    static constexpr int NG = D / G;
    static constexpr int PITCH = D + 16 / (int)sizeof(T);      // staged row, 16-byte pad (no bank conflicts)
    static constexpr int ROW_BYTES = PITCH * (int)sizeof(T);
    static constexpr int X_BYTES = G * ROW_BYTES;                // one staged K or V group
    static constexpr int WORK_BYTES = 3 * D * 4 + 3 * NG * G * 4 + RecGeom<BITS, D>::REC;
    static constexpr int BYTES = 2 * X_BYTES + WORK_BYTES;      // one stage + work
};

// Copy n rows of D elements (16-byte aligned) into staged rows of PITCH.
template <typename T, int D, typename RowFn>
__device__ __forceinline__ void stage_rows(RowFn row, T *dst, int n, int tid, int nthr)
{
    constexpr int CH = D * (int)sizeof(T) / 16;
    constexpr int PITCH = D + 16 / (int)sizeof(T);
    for (int i = tid; i < n * CH; i += nthr) {
        const int t = i / CH, ch = i % CH;
        const uint4 u = *reinterpret_cast<const uint4 *>(row(t) + ch * (16 / (int)sizeof(T)));
        *reinterpret_cast<uint4 *>(dst + t * PITCH + ch * (16 / (int)sizeof(T))) = u;
    }
}

template <typename T>
__device__ __forceinline__ float2 load_pair(const T *p);
template <>
__device__ __forceinline__ float2 load_pair<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
    return make_float2(bf16_lo(w), bf16_hi(w));
}
template <>
__device__ __forceinline__ float2 load_pair<float>(const float *p)
{
    return *reinterpret_cast<const float2 *>(p);
}

// Pair (kappa, mu) in slot sl of code word w, for a word index known only at
// run time (inverse of pair_pos).
template <int BITS, int D>
__device__ __forceinline__ void slot_pair(int w, int sl, int &kappa, int &mu)
{
    constexpr int W = D * BITS / 32;
    if (BITS == 2) {
        constexpr int h = W / 2, q = W / 4;
        if (sl < 3) {
            kappa = h * sl + (w >> 1);
            mu = 2 * (w & 1);
        } else if (sl >= 5) {
            kappa = h * (sl - 5) + (w >> 1);
            mu = 2 * (w & 1) + 1;
        } else {
            kappa = 3 * h + q * (sl - 3) + (w >> 2);
            mu = w & 3;
        }
    } else {
        constexpr int h = W / 2;
        kappa = h * (sl & 1) + (w >> 1);
        mu = 2 * (w & 1) + (sl >> 1);
    }
}

// The two values of code pair (kappa, mu) of lane (gid, tig) and the index of
// their statistics: K pairs are channels c, c + 1 of one token (statistics
// per channel), V pairs tokens t, t + 1 of one channel (statistics per token
// of the channel's group, stored [group][token]).
template <typename T, int D, int SEC>
__device__ __forceinline__ float2 pair_values(const T *x, int kappa, int mu, int gid, int tig, int &st)
{
    constexpr int PITCH = D + 16 / (int)sizeof(T);
    if (SEC == 0) {
        const int t = 16 * (mu >> 1) + 8 * (mu & 1) + gid;
        const int c = 16 * (kappa >> 1) + 8 * (kappa & 1) + 2 * tig;
        st = c;
        return load_pair<T>(x + t * PITCH + c);
    } else {
        const int c = 16 * (kappa >> 1) + 8 * (kappa & 1) + gid;
        const int t = 16 * (mu >> 1) + 8 * (mu & 1) + 2 * tig;
        st = (c / G) * G + t;
        return make_float2(Elem<T>::to_f(x[t * PITCH + c]), Elem<T>::to_f(x[(t + 1) * PITCH + c]));
    }
}

// Where the code pair of slot sl in word i of a thread sits: (kappa, mu) =
// (kc + kp, mc + mp), with (kc, mc) fixed by (i, sl) and (kp, mp) one of two
// per-thread pairs (sel) that depend only on the thread's warp p of the
// section (the inverse of pair_pos split into its constant and per-thread
// parts; with the loops over i and sl unrolled, kc and mc are constants).
struct SlotSplit {
    int kc, mc, sel;
};
template <int BITS, int D>
__device__ __forceinline__ SlotSplit slot_split(int i, int sl)
{
    constexpr int W = D * BITS / 32;
    if (BITS == 2) {
        constexpr int h = W / 2, q = W / 4;
        if (sl < 3) return {h * sl, 2 * i, 0};
        if (sl >= 5) return {h * (sl - 5), 2 * i + 1, 0};
        return {3 * h + q * (sl - 3), i, 1};
    } else {
        constexpr int h = W / 2;
        return {h * (sl & 1) + (i >> 1), 2 * (i & 1) + (sl >> 1), 0};
    }
}

// Code words of one section for this thread: words WPT*p .. WPT*p + WPT - 1
// of lane (gid, tig), stored into the section image.  A pair (kappa, mu) holds
// channels 8 kappa + 2 tig, +1 of token 8 mu + gid (K) or tokens 8 mu + 2 tig,
// +1 of channel 8 kappa + gid (V), so every staged value and statistic is at a
// per-thread base plus a constant offset.
template <typename T, int BITS, int D, int SEC>
__device__ __forceinline__ void code_words(const T *x, const float *stz, const float *strs, const float *sts,
                                           uint8_t *secimg, int lane, int p)
{
    constexpr int WPT = BITS;                      // W * 32 / D words per thread
    constexpr int SLOTS = 16 / BITS;
    constexpr int PITCH = D + 16 / (int)sizeof(T);
    constexpr uint32_t qmax = (1u << BITS) - 1u;
    const int gid = lane >> 2, tig = lane & 3;
    // per-thread parts: sel 0 (kp, mp) = (p or 2p, 0), sel 1 (p / 2, 2 (p % 2))
    const int kp[2] = {BITS == 2 ? p : 2 * p, p >> 1};
    const int mp[2] = {0, 2 * (p & 1)};
    int cb[2], tb[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        cb[s] = 8 * kp[s] + (SEC == 0 ? 2 * tig : gid);
        tb[s] = 8 * mp[s] + (SEC == 0 ? gid : 2 * tig);
    }
    const T *xb[2] = {x + tb[0] * PITCH + cb[0], x + tb[1] * PITCH + cb[1]};
    uint32_t words[WPT];
    uint32_t near = 0;                             // bit (i, sl, hh): needs the exact quotient
#pragma unroll
    for (int i = 0; i < WPT; ++i) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int sl = 0; sl < SLOTS; ++sl) {
            const SlotSplit ss = slot_split<BITS, D>(i, sl);
            const T *px = xb[ss.sel] + 8 * ss.mc * PITCH + 8 * ss.kc;
            float2 xv;
            int st;
            if constexpr (SEC == 0) {
                xv = load_pair<T>(px);
                st = cb[ss.sel] + 8 * ss.kc;
            } else {
                xv = make_float2(Elem<T>::to_f(px[0]), Elem<T>::to_f(px[PITCH]));
                st = ((cb[ss.sel] + 8 * ss.kc) & ~(G - 1)) + tb[ss.sel] + 8 * ss.mc;
            }
            const float2 z = *reinterpret_cast<const float2 *>(stz + st);
            const float2 rs = *reinterpret_cast<const float2 *>(strs + st);
            // d = RN(x - z), q = RN(d * rcp(s)), m = RN(q + 1.5 * 2^23) (integer
            // part = rint(q)), e = q - rint(q), both lanes at once
            const float2 magic = make_float2(kRoundMagic, kRoundMagic);
            const float2 q = mul2(sub2(xv, z), rs);
            const float2 r = sub2(add2(q, magic), magic);
            const float2 e = sub2(q, r);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int bit = (i * SLOTS + sl) * 2 + hh;
                near |= near_mask(hh ? e.y : e.x, kNearHalf) & (1u << bit);
            }
            const float wsl = (float)(1u << (BITS * sl));
            acc = fma2(r, make_float2(wsl, wsl), acc);
        }
        words[i] = (uint32_t)acc.x | ((uint32_t)acc.y << 16);
    }
    // codes within rounding distance of a half-integer: the exact quotient
    while (near) {
        const int bit = __ffs(near) - 1;
        near &= near - 1;
        const int i = bit / (2 * SLOTS), sl = (bit / 2) % SLOTS, hh = bit & 1;
        int kappa, mu, st;
        slot_pair<BITS, D>(WPT * p + i, sl, kappa, mu);
        const float2 xv = pair_values<T, D, SEC>(x, kappa, mu, gid, tig, st);
        const uint32_t c = exact_code(hh ? xv.y : xv.x, stz[st + hh], sts[st + hh]);
        const int sh = BITS * sl + 16 * hh;
        words[i] = (words[i] & ~(qmax << sh)) | (c << sh);
    }
    uint8_t *dst = secimg + word_byte(lane, WPT * p);
    if constexpr (WPT == 2)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(words[0], words[1]);
    else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

// min / max of n bf16 (or fp32) pairs at stride `step` elements
template <typename T>
__device__ __forceinline__ void pair_minmax(const T *x, int n, int step, float2 &mn, float2 &mx);
template <>
__device__ __forceinline__ void pair_minmax<__nv_bfloat16>(const __nv_bfloat16 *x, int n, int step, float2 &mn,
                                                           float2 &mx)
{
    __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(x), hi = lo;
#pragma unroll 8
    for (int t = 1; t < n; ++t) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(x + t * step);
        lo = __hmin2(lo, v);
        hi = __hmax2(hi, v);
    }
    mn = __bfloat1622float2(lo);
    mx = __bfloat1622float2(hi);
}
template <>
__device__ __forceinline__ void pair_minmax<float>(const float *x, int n, int step, float2 &mn, float2 &mx)
{
    mn = mx = *reinterpret_cast<const float2 *>(x);
#pragma unroll 8
    for (int t = 1; t < n; ++t) {
        const float2 v = *reinterpret_cast<const float2 *>(x + t * step);
        mn.x = fminf(mn.x, v.x);
        mn.y = fminf(mn.y, v.y);
        mx.x = fmaxf(mx.x, v.x);
        mx.y = fmaxf(mx.y, v.y);
    }
}

// Quantize one staged group (K rows kx, V rows vx at the staged pitch) into
// the record `rec`, by a block of 2 D threads; `work` holds the statistics and
// the record image (QStage::WORK_BYTES).  The staged rows must be visible to
// every thread on entry; they are no longer read once the second barrier
// inside has passed.
template <typename T, int BITS, int D>
__device__ void quantize_staged(const T *kx, const T *vx, uint8_t *work, uint8_t *__restrict__ rec)
{
    using Gm = RecGeom<BITS, D>;
    using St = QStage<T, BITS, D>;
    constexpr int qmax = (1 << BITS) - 1;
    constexpr int NG = D / G;
    constexpr int PITCH = St::PITCH;
    const int tid = threadIdx.x;
    float *kst = reinterpret_cast<float *>(work);
    float *vst = kst + 3 * D;
    uint8_t *img = work + 3 * D * 4 + 3 * NG * G * 4;
    // ---- statistics, one group parameter per thread: threads [0, D) take K
    // channel c (the two lanes of a pair each reduce 16 tokens of channels
    // c & ~1, c | 1 and exchange), threads [D, 2D) a V (token, channel group)
    if (tid < D) {
        const int cp = tid >> 1, half = tid & 1;
        float2 mn, mx;
        pair_minmax<T>(kx + half * (G / 2) * PITCH + 2 * cp, G / 2, PITCH, mn, mx);
        mn.x = fminf(mn.x, __shfl_xor_sync(0xffffffffu, mn.x, 1));
        mn.y = fminf(mn.y, __shfl_xor_sync(0xffffffffu, mn.y, 1));
        mx.x = fmaxf(mx.x, __shfl_xor_sync(0xffffffffu, mx.x, 1));
        mx.y = fmaxf(mx.y, __shfl_xor_sync(0xffffffffu, mx.y, 1));
        const int ch = 2 * cp + half;
        uint16_t sb, zb;
        float sf, zf;
        group_params(half ? mn.y : mn.x, half ? mx.y : mx.x, qmax, sb, zb, sf, zf);
        kst[ch] = zf;
        kst[D + ch] = rcp_scale(sf);
        kst[2 * D + ch] = sf;
        // quad j, k-step ks: zero pair then scale pair for rr = 0, then rr = 1
        const int ks = ch >> 4, col = ch & 15;
        const int j = (col & 7) >> 1, rr = col >> 3;
        const int off = Gm::KM + 16 * (4 * ks + j) + 8 * rr + 2 * (ch & 1);
        *reinterpret_cast<uint16_t *>(img + off) = zb;
        *reinterpret_cast<uint16_t *>(img + off + 4) = sb;
    } else {
        const int i = tid - D;
        const int t = i % G, gc = i / G;
        float2 a, b;
        pair_minmax<T>(vx + t * PITCH + gc * G, G / 2, 2, a, b);
        uint16_t sb, zb;
        float sf, zf;
        group_params(fminf(a.x, a.y), fmaxf(b.x, b.y), qmax, sb, zb, sf, zf);
        vst[gc * G + t] = zf;
        vst[NG * G + gc * G + t] = rcp_scale(sf);
        vst[2 * NG * G + gc * G + t] = sf;
        const int ks = t >> 4, colt = t & 15;
        const int j = (colt & 7) >> 1, n = (2 * ks + (colt >> 3)) * NG + gc;
        const int off = Gm::VM + 16 * (4 * (n >> 2) + j) + 4 * (n & 3) + 2 * (t & 1);
        *reinterpret_cast<uint16_t *>(img + off) = sb;
        *reinterpret_cast<uint16_t *>(img + off + 2 * D) = zb;
    }
    __syncthreads();                                       // statistics and meta written
    // ---- code words: threads [0, D) the K section, [D, 2D) the V section
    {
        const int j = tid % D;
        const int lane = j & 31, p = j >> 5;
        if (tid < D)
            code_words<T, BITS, D, 0>(kx, kst, kst + D, kst + 2 * D, img, lane, p);
        else
            code_words<T, BITS, D, 1>(vx, vst, vst + NG * G, vst + 2 * NG * G, img + Gm::CODE, lane, p);
    }
    __syncthreads();                                       // record image complete
    uint4 *dst = reinterpret_cast<uint4 *>(rec);
    const uint4 *srcv = reinterpret_cast<const uint4 *>(img);
    for (int i = tid; i < Gm::REC / 16; i += 2 * D) dst[i] = srcv[i];
}

// Key rotation (rotated caches, vc_quant_cfg.rotate): each key row x becomes
// T(W(x) * 2^-ceil(log2(D)/2)), W the binary32 Walsh-Hadamard butterfly
// network with stages h = 1, 2, ..., D/2 mapping the pair (i, i + h),
// i mod 2h < h, to (a + b, a - b).  The query side uses 2^-floor(log2(D)/2),
// so that rotated dot products equal the plain ones (H H^T = D I).
template <int D>
struct RotScale {
    static constexpr int LG = D == 128 ? 7 : 6;
    static constexpr float K = LG == 7 ? 0.0625f : 0.125f;
};

// n rows from src(r) to dst(r) (D elements of T each), ROWS at a time through
// buf, by all threads of the block (block-uniform call).
template <typename T, int D, int ROWS, typename SrcFn, typename DstFn>
__device__ void rotate_rows(int n, SrcFn src, DstFn dst, float (*buf)[D])
{
    for (int r0 = 0; r0 < n; r0 += ROWS) {
        const int nr = min(ROWS, n - r0);
        for (int i = threadIdx.x; i < nr * D; i += blockDim.x) buf[i / D][i % D] = Elem<T>::to_f(src(r0 + i / D)[i % D]);
        __syncthreads();
        for (int h = 1; h < D; h <<= 1) {
            for (int p = threadIdx.x; p < nr * (D / 2); p += blockDim.x) {
                const int r = p / (D / 2), kk = p % (D / 2);
                const int i = (kk / h) * 2 * h + (kk % h);
                const float a = buf[r][i], b = buf[r][i + h];
                buf[r][i] = a + b;
                buf[r][i + h] = a - b;
            }
            __syncthreads();
        }
        for (int i = threadIdx.x; i < nr * D; i += blockDim.x)
            dst(r0 + i / D)[i % D] = Elem<T>::from_f(buf[i / D][i % D] * RotScale<D>::K);
        __syncthreads();
    }
}

// Prefill: one CTA per (group, kv head, sequence); its 32 K and 32 V rows
// arrive by one bulk copy each (all 64 in flight at once, one mbarrier with a
// bounded wait; a wait that gives up sets bit 2 of the cache's status word
// and leaves the group's record unwritten), are rotated in place for a
// rotated cache, then quantized.
template <typename T, int BITS, int D, bool ROT>
__global__ void __launch_bounds__(2 * D, 5)
quantize_prefill_kernel(const T *__restrict__ k, const T *__restrict__ v, int Hkv, int L_stride,
                        int max_groups, uint8_t *__restrict__ records, int32_t *status)
{
    using Gm = RecGeom<BITS, D>;
    using St = QStage<T, BITS, D>;
    constexpr int ROW = D * (int)sizeof(T);
    __shared__ __align__(16) uint8_t sm[St::BYTES];
    __shared__ __align__(8) uint64_t bar;
    const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * Hkv + h;
    const size_t row0 = bh * L_stride + (size_t)g * G;
    T *kx = reinterpret_cast<T *>(sm);
    T *vx = reinterpret_cast<T *>(sm + St::X_BYTES);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x < 2 * G) {
        const int t = threadIdx.x & (G - 1);
        const bool is_v = threadIdx.x >= G;
        bulk_g2s((is_v ? vx : kx) + t * St::PITCH, (is_v ? v : k) + (row0 + t) * D, ROW, &bar);
    }
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&bar, 2 * G * ROW);
    const bool got = mbar_wait(&bar, 0);
    if (!__syncthreads_and(got)) {
        if (threadIdx.x == 0 && status) atomicOr(status, 4);
        return;
    }
    if constexpr (ROT) {
        // the key rows, rotated in place
        __shared__ __align__(16) float buf[8][D];
        rotate_rows<T, D, 8>(
            G, [&](int t) { return kx + t * St::PITCH; }, [&](int t) { return kx + t * St::PITCH; }, buf);
    }
    quantize_staged<T, BITS, D>(kx, vx, sm + 2 * St::X_BYTES, records + (bh * max_groups + g) * Gm::REC);
}

// Copy positions n_q*G .. L-1 into the ring (keys rotated for a rotated
// cache) and publish the lengths.
template <typename T, int D, bool ROT>
__global__ void residual_copy_kernel(const T *__restrict__ k, const T *__restrict__ v, int B,
                                     int Hkv, int L, int L_stride, int nq_tokens, T *kres,
                                     T *vres, int res_cap, int32_t *n_groups, int32_t *seq_len)
{
    const size_t bh = blockIdx.x;
    const int ntok = L - nq_tokens;
    for (int i = threadIdx.x; i < ntok * D; i += blockDim.x) {
        const int t = i / D, c = i % D;
        const long pos = nq_tokens + t;
        const size_t src = (bh * L_stride + pos) * D + c;
        const size_t dst = (bh * res_cap + pos % res_cap) * D + c;
        if (!ROT) kres[dst] = k[src];
        vres[dst] = v[src];
    }
    if constexpr (ROT) {
        __shared__ __align__(16) float buf[8][D];
        rotate_rows<T, D, 8>(
            ntok, [&](int t) { return k + (bh * L_stride + nq_tokens + t) * D; },
            [&](int t) { return kres + (bh * res_cap + (size_t)((nq_tokens + t) % res_cap)) * D; }, buf);
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < B; i += blockDim.x) {
            n_groups[i] = nq_tokens / G;
            seq_len[i] = L;
        }
}

// Append new tokens into the ring, then quantize every complete group that
// left the residual window.  Grid (Hc, B) in clusters of Hc = min(Hkv, 8)
// CTAs: CTA r of sequence b handles kv heads r, r + Hc, ...; every CTA reads
// the old lengths, and after a cluster barrier (all reads done) rank 0
// publishes the new ones.
// Commit mode (len_base, n_acc non-null): roll back to len_base[b] and take
// n_acc[b] + 1 rows.  With n_new null every sequence takes max_new rows.
template <typename T, int BITS, int D, bool ROT>
__global__ void __launch_bounds__(2 * D)
append_kernel(const T *__restrict__ k_new, const T *__restrict__ v_new,
              const int32_t *__restrict__ n_new, const int32_t *__restrict__ len_base,
              const int32_t *__restrict__ n_acc, int max_new, int Hkv, T *kres, T *vres,
              int res_cap, int residual, int requantize, int max_groups,
              uint8_t *__restrict__ records, int32_t *n_groups, int32_t *seq_len, int32_t *status)
{
    pdl_wait();
    pdl_trigger();
    using Gm = RecGeom<BITS, D>;
    using St = QStage<T, BITS, D>;
    __shared__ __align__(16) uint8_t sm[St::BYTES];
    const int rank = blockIdx.x, Hc = gridDim.x;
    const int b = blockIdx.y;
    const bool leader = rank == 0 && threadIdx.x == 0;
    const int ng0 = n_groups[b];
    int len0 = len_base ? len_base[b] : seq_len[b];
    if (len0 < ng0 * G) {
        if (leader && status) atomicOr(status, 2);
        len0 = ng0 * G;
    }
    int nn = n_acc ? n_acc[b] + 1 : (n_new ? n_new[b] : max_new);
    nn = nn < 0 ? 0 : (nn > max_new ? max_new : nn);
    // unquantized tokens after the append must fit the ring
    const int room = res_cap - (len0 - ng0 * G);
    if (nn > room) {
        if (leader && status) atomicOr(status, 1);
        nn = room > 0 ? room : 0;
    }
    const int len1 = len0 + nn;
    int ng1 = ng0;
    if (requantize) {
        while ((ng1 + 1) * G <= len1 - residual && ng1 < max_groups) ++ng1;
    }
    for (int h = rank; h < Hkv; h += Hc) {
        const size_t bh = (size_t)b * Hkv + h;
        for (int i = threadIdx.x; i < nn * D; i += 2 * D) {
            const int t = i / D, c = i % D;
            const size_t src = ((bh * max_new) + t) * D + c;
            const size_t dst = (bh * res_cap + (size_t)((len0 + t) % res_cap)) * D + c;
            if (!ROT) kres[dst] = k_new[src];
            vres[dst] = v_new[src];
        }
        if constexpr (ROT) {
            __shared__ __align__(16) float buf[8][D];
            rotate_rows<T, D, 8>(
                nn, [&](int t) { return k_new + (bh * max_new + t) * D; },
                [&](int t) { return kres + (bh * res_cap + (size_t)((len0 + t) % res_cap)) * D; }, buf);
        }
        __syncthreads();
        for (int g = ng0; g < ng1; ++g) {
            auto ring_row = [&](const T *ring, int t) {
                return ring + (bh * res_cap + (size_t)(((long)g * G + t) % res_cap)) * D;
            };
            T *kx = reinterpret_cast<T *>(sm);
            T *vx = reinterpret_cast<T *>(sm + St::X_BYTES);
            stage_rows<T, D>([&](int t) { return ring_row(kres, t); }, kx, G, threadIdx.x, 2 * D);
            stage_rows<T, D>([&](int t) { return ring_row(vres, t); }, vx, G, threadIdx.x, 2 * D);
            __syncthreads();
            quantize_staged<T, BITS, D>(kx, vx, sm + 2 * St::X_BYTES, records + (bh * max_groups + g) * Gm::REC);
            __syncthreads();
        }
    }
    cg::this_cluster().sync();
    if (leader) {
        seq_len[b] = len1;
        n_groups[b] = ng1;
    }
}

template <typename T, int BITS, int D>
cudaError_t launch_prefill(const void *k, const void *v, int B, int Hkv, int L, int L_stride,
                           const vc_qcache *c, cudaStream_t st)
{
    const int R = c->cfg.residual;
    const int nq = (L - R > 0) ? ((L - R) / G) * G : 0;
    const bool rot = c->cfg.rotate != 0;
    if (nq > 0) {
        dim3 grid(nq / G, Hkv, B);
        auto kern = rot ? quantize_prefill_kernel<T, BITS, D, true> : quantize_prefill_kernel<T, BITS, D, false>;
        kern<<<grid, 2 * D, 0, st>>>((const T *)k, (const T *)v, Hkv, L_stride, c->max_groups,
                                     (uint8_t *)c->records, c->status);
    }
    auto rc = rot ? residual_copy_kernel<T, D, true> : residual_copy_kernel<T, D, false>;
    rc<<<B * Hkv, 256, 0, st>>>((const T *)k, (const T *)v, B, Hkv, L, L_stride, nq, (T *)c->k_res,
                                (T *)c->v_res, c->res_cap, c->n_groups, c->seq_len);
    return cudaGetLastError();
}

template <typename T, int BITS, int D>
cudaError_t launch_append(const vc_qcache *c, const void *kn, const void *vn, const int32_t *n_new,
                          const int32_t *len_base, const int32_t *n_acc, int max_new, int requantize,
                          cudaStream_t st)
{
    const int hc = c->Hkv < 8 ? c->Hkv : 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(hc, c->B, 1);
    cfg.blockDim = dim3(2 * D, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = hc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // the kernel waits on the device
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    auto kern = c->cfg.rotate ? append_kernel<T, BITS, D, true> : append_kernel<T, BITS, D, false>;
    return cudaLaunchKernelEx(&cfg, kern, (const T *)kn, (const T *)vn, n_new, len_base,
                              n_acc, max_new, c->Hkv, (T *)c->k_res, (T *)c->v_res, c->res_cap,
                              c->cfg.residual, requantize, c->max_groups, (uint8_t *)c->records, c->n_groups,
                              c->seq_len, c->status);
}

template <typename T>
cudaError_t dispatch_prefill(const void *k, const void *v, int B, int Hkv, int L, int L_stride,
                             int d, const vc_qcache *c, cudaStream_t st)
{
    const int bits = c->cfg.bits;
    if (d == 128) return bits == 2 ? launch_prefill<T, 2, 128>(k, v, B, Hkv, L, L_stride, c, st)
                                   : launch_prefill<T, 4, 128>(k, v, B, Hkv, L, L_stride, c, st);
    return bits == 2 ? launch_prefill<T, 2, 64>(k, v, B, Hkv, L, L_stride, c, st)
                     : launch_prefill<T, 4, 64>(k, v, B, Hkv, L, L_stride, c, st);
}

template <typename T>
cudaError_t dispatch_append(const vc_qcache *c, const void *kn, const void *vn, const int32_t *nn,
                            const int32_t *lb, const int32_t *na, int max_new, int rq, cudaStream_t st)
{
    const int bits = c->cfg.bits;
    if (c->d == 128) return bits == 2 ? launch_append<T, 2, 128>(c, kn, vn, nn, lb, na, max_new, rq, st)
                                      : launch_append<T, 4, 128>(c, kn, vn, nn, lb, na, max_new, rq, st);
    return bits == 2 ? launch_append<T, 2, 64>(c, kn, vn, nn, lb, na, max_new, rq, st)
                     : launch_append<T, 4, 64>(c, kn, vn, nn, lb, na, max_new, rq, st);
}

}  // namespace

cudaError_t quantize_prefill(const void *k, const void *v, vc_dtype dt, int B, int Hkv, int L,
                             int L_stride, int d, const vc_qcache *c, cudaStream_t st)
{
    return dt == VC_BF16 ? dispatch_prefill<__nv_bfloat16>(k, v, B, Hkv, L, L_stride, d, c, st)
                         : dispatch_prefill<float>(k, v, B, Hkv, L, L_stride, d, c, st);
}

cudaError_t qcache_append(const vc_qcache *c, const void *kn, const void *vn, const int32_t *nn,
                          const int32_t *len_base, const int32_t *n_acc, int max_new, int requantize,
                          cudaStream_t st)
{
    return c->res_dtype == VC_BF16
               ? dispatch_append<__nv_bfloat16>(c, kn, vn, nn, len_base, n_acc, max_new, requantize, st)
               : dispatch_append<float>(c, kn, vn, nn, len_base, n_acc, max_new, requantize, st);
}

}  // namespace vc
