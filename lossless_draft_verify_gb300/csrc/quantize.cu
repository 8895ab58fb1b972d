// quantize.cu -- KIVI-style asymmetric group quantization of the draft cache
// (KIVI: a compressor named on the VeriCache paper page, "What the paper
// found"; ref [42] on pith.science).  K per channel over groups of 32 tokens,
// V per token over groups of 32 channels, fp16 scale and zero-point per group,
// packed into the record layout the draft kernel consumes (see include/vc.h).
//
// One 128-thread CTA quantizes one (sequence, kv head, token group): the two
// 32 x d tiles are staged in shared memory as fp32, each K channel / V
// (token, channel-group) is reduced by one thread, and the record is written
// with coalesced 32-bit stores.  The operation is HBM-bound (it reads the
// bf16 tiles once and writes ~3/16 of that), with no tensor-core work.
#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int G = 32;            // group size (tokens for K, channels for V)
constexpr int kThreads = 128;

// Directed-rounding quantization parameters of one group (see include/vc.h).
__device__ __forceinline__ void group_params(float mn, float mx, int qmax, uint16_t &sb,
                                             uint16_t &zb, float &sf, float &zf)
{
    __half z = __float2half_rd(mn);
    zf = __half2float(z);
    float range = __fadd_ru(mx, -zf);
    float step = __fdiv_ru(range, (float)qmax);
    __half s = __float2half_ru(step);
    sf = __half2float(s);
    sb = __half_as_ushort(s);
    zb = __half_as_ushort(z);
}

__device__ __forceinline__ uint32_t group_code(float x, float sf, float zf, int qmax)
{
    if (sf == 0.0f) return 0u;
    float r = rintf(__fdiv_rn(__fadd_rn(x, -zf), sf));
    r = fminf(fmaxf(r, 0.0f), (float)qmax);
    return (uint32_t)r;
}

template <int D>
struct QSmem {
    float k[G][D + 1];
    float v[G][D + 1];
    uint8_t kc[G][D];
    uint8_t vc[G][D];
    uint16_t ks[D], kz[D];
    uint16_t vs[G][D / G], vz[G][D / G];
};

// Quantize the staged tiles and write one record.  All threads participate.
template <int BITS, int D>
__device__ void quantize_staged_group(QSmem<D> &sm, uint8_t *__restrict__ rec)
{
    constexpr int qmax = (1 << BITS) - 1;
    constexpr int NG = D / G;
    const int tid = threadIdx.x;
    // K: one thread per channel, over the 32 tokens of the group.
    if (tid < D) {
        const int c = tid;
        float mn = sm.k[0][c], mx = mn;
#pragma unroll 8
        for (int t = 1; t < G; ++t) {
            float x = sm.k[t][c];
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        uint16_t sb, zb;
        float sf, zf;
        group_params(mn, mx, qmax, sb, zb, sf, zf);
        sm.ks[c] = sb;
        sm.kz[c] = zb;
#pragma unroll 8
        for (int t = 0; t < G; ++t) sm.kc[t][c] = (uint8_t)group_code(sm.k[t][c], sf, zf, qmax);
    }
    // V: one thread per (token, channel group); warp = channel group, lane = token.
    if (tid < G * NG) {
        const int t = tid % G, gc = tid / G;
        float mn = sm.v[t][gc * G], mx = mn;
#pragma unroll 8
        for (int i = 1; i < G; ++i) {
            float x = sm.v[t][gc * G + i];
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        uint16_t sb, zb;
        float sf, zf;
        group_params(mn, mx, qmax, sb, zb, sf, zf);
        sm.vs[t][gc] = sb;
        sm.vz[t][gc] = zb;
#pragma unroll 8
        for (int i = 0; i < G; ++i)
            sm.vc[t][gc * G + i] = (uint8_t)group_code(sm.v[t][gc * G + i], sf, zf, qmax);
    }
    __syncthreads();

    // Pack codes in fragment order.
    constexpr int E = G * D / 32;                 // codes per lane
    constexpr int WPL = E * BITS / 32;            // 32-bit words per lane
    constexpr int P = 16 / BITS;                  // code pairs per word
    constexpr int KS = D / 16;
    constexpr int WORDS = 32 * WPL;               // words per code section
    uint32_t *kcw = reinterpret_cast<uint32_t *>(rec);
    uint32_t *vcw = kcw + WORDS;
    for (int wi = tid; wi < WORDS; wi += kThreads) {
        const int lane = wi / WPL, w = wi % WPL;
        const int gid = lane >> 2, tig = lane & 3;
        uint32_t kword = 0, vword = 0;
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const int p = w * P + j;
            const int r = p & 3, blk = p >> 2;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int shift = BITS * j + 16 * hh;
                {   // K: blk = mt * KS + ks
                    const int mt = blk / KS, ks = blk % KS;
                    const int t = 16 * mt + gid + 8 * (r & 1);
                    const int c = 16 * ks + 2 * tig + hh + 8 * (r >> 1);
                    kword |= (uint32_t)sm.kc[t][c] << shift;
                }
                {   // V: blk = mt * 2 + ks
                    const int mt = blk >> 1, ks = blk & 1;
                    const int c = 16 * mt + gid + 8 * (r & 1);
                    const int t = 16 * ks + 2 * tig + hh + 8 * (r >> 1);
                    vword |= (uint32_t)sm.vc[t][c] << shift;
                }
            }
        }
        kcw[wi] = kword;
        vcw[wi] = vword;
    }
    // Meta sections: 4 blocks of D bytes each = D words per section.
    uint32_t *kmw = vcw + WORDS;
    uint32_t *vmw = kmw + D;
    for (int wi = tid; wi < D; wi += kThreads) {
        const int j = (4 * wi) / D, o = 4 * wi - j * D;
        const bool zero = o >= D / 2;
        const int q = (zero ? o - D / 2 : o) / 4;
        {   // K meta: q = 2 ks + rr
            const int ks = q >> 1, rr = q & 1;
            const int c0 = 16 * ks + 2 * j + 8 * rr;
            const uint16_t *src = zero ? sm.kz : sm.ks;
            kmw[wi] = (uint32_t)src[c0] | ((uint32_t)src[c0 + 1] << 16);
        }
        {   // V meta: q = (2 ks + rr) * NG + gc
            const int gc = q % NG, kr = q / NG;
            const int ks = kr >> 1, rr = kr & 1;
            const int t0 = 16 * ks + 2 * j + 8 * rr;
            const uint16_t(*src)[NG] = zero ? sm.vz : sm.vs;
            vmw[wi] = (uint32_t)src[t0][gc] | ((uint32_t)src[t0 + 1][gc] << 16);
        }
    }
}

// Stage rows row0..row0+31 of a [rows][D] tensor (element type T) as fp32.
template <typename T, int D>
__device__ __forceinline__ void stage_tile(float (*dst)[D + 1], const T *__restrict__ src)
{
    constexpr int PER16 = 16 / sizeof(T);
    constexpr int CHUNKS = G * D / PER16;
    for (int i = threadIdx.x; i < CHUNKS; i += kThreads) {
        const int t = i / (D / PER16), c0 = (i % (D / PER16)) * PER16;
        uint4 u = ldg_stream(src + (size_t)t * D + c0);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dst[t][c0 + 2 * e] = bf16_lo(w[e]);
                dst[t][c0 + 2 * e + 1] = bf16_hi(w[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[t][c0 + e] = __uint_as_float(w[e]);
        }
    }
}

// Stage ring positions pos0..pos0+31 of (b, h) as fp32.
template <typename T, int D>
__device__ __forceinline__ void stage_ring_tile(float (*dst)[D + 1], const T *__restrict__ ring,
                                                long pos0, int res_cap)
{
    for (int i = threadIdx.x; i < G * D; i += kThreads) {
        const int t = i / D, c = i % D;
        dst[t][c] = Elem<T>::to_f(ring[(size_t)((pos0 + t) % res_cap) * D + c]);
    }
}

template <typename T, int BITS, int D>
__global__ void __launch_bounds__(kThreads)
quantize_prefill_kernel(const T *__restrict__ k, const T *__restrict__ v, int Hkv, int L_stride,
                        int max_groups, uint8_t *__restrict__ records, size_t rec_bytes)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    QSmem<D> &sm = *reinterpret_cast<QSmem<D> *>(smem_raw);
    const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * Hkv + h;
    const size_t row0 = bh * L_stride + (size_t)g * G;
    stage_tile<T, D>(sm.k, k + row0 * D);
    stage_tile<T, D>(sm.v, v + row0 * D);
    __syncthreads();
    quantize_staged_group<BITS, D>(sm, records + (bh * max_groups + g) * rec_bytes);
}

// Copy positions n_q*G .. L-1 into the ring and publish the lengths.
template <typename T, int D>
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
        kres[dst] = k[src];
        vres[dst] = v[src];
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < B; i += blockDim.x) {
            n_groups[i] = nq_tokens / G;
            seq_len[i] = L;
        }
}

// Append new tokens into the ring, then quantize every complete group that
// left the residual window.  One CTA per sequence handles all its kv heads, so
// the lengths of sequence b are read and written by exactly one CTA.
template <typename T, int BITS, int D>
__global__ void __launch_bounds__(kThreads)
append_kernel(const T *__restrict__ k_new, const T *__restrict__ v_new,
              const int32_t *__restrict__ n_new, const int32_t *__restrict__ len_base,
              const int32_t *__restrict__ n_acc, int max_new, int Hkv, T *kres, T *vres,
              int res_cap, int residual, int requantize, int max_groups,
              uint8_t *__restrict__ records, size_t rec_bytes, int32_t *n_groups,
              int32_t *seq_len, int32_t *status)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    QSmem<D> &sm = *reinterpret_cast<QSmem<D> *>(smem_raw);
    const int b = blockIdx.x;
    const int ng0 = n_groups[b];
    // commit mode: roll back to the round-start length, then take the n_acc + 1
    // verified tokens; never below the quantized prefix
    int len0 = len_base ? len_base[b] : seq_len[b];
    if (len0 < ng0 * G) {
        if (threadIdx.x == 0 && status) atomicOr(status, 2);
        len0 = ng0 * G;
    }
    int nn = n_acc ? n_acc[b] + 1 : n_new[b];
    nn = nn < 0 ? 0 : (nn > max_new ? max_new : nn);
    // Unquantized tokens after the append must fit the ring.
    const int room = res_cap - (len0 - ng0 * G);
    if (nn > room) {
        if (threadIdx.x == 0 && status) atomicOr(status, 1);
        nn = room > 0 ? room : 0;
    }
    const int len1 = len0 + nn;
    int ng1 = ng0;
    if (requantize) {
        while ((ng1 + 1) * G <= len1 - residual && ng1 < max_groups) ++ng1;
    }
    for (int h = 0; h < Hkv; ++h) {
        const size_t bh = (size_t)b * Hkv + h;
        for (int i = threadIdx.x; i < nn * D; i += kThreads) {
            const int t = i / D, c = i % D;
            const size_t src = ((bh * max_new) + t) * D + c;
            const size_t dst = (bh * res_cap + (size_t)((len0 + t) % res_cap)) * D + c;
            kres[dst] = k_new[src];
            vres[dst] = v_new[src];
        }
        __syncthreads();
        for (int g = ng0; g < ng1; ++g) {
            stage_ring_tile<T, D>(sm.k, kres + bh * res_cap * D, (long)g * G, res_cap);
            stage_ring_tile<T, D>(sm.v, vres + bh * res_cap * D, (long)g * G, res_cap);
            __syncthreads();
            quantize_staged_group<BITS, D>(sm, records + (bh * max_groups + g) * rec_bytes);
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) {
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
    const size_t rb = vc_record_bytes(BITS, D);
    const size_t smem = sizeof(QSmem<D>);
    auto kern = quantize_prefill_kernel<T, BITS, D>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (nq > 0) {
        dim3 grid(nq / G, Hkv, B);
        kern<<<grid, kThreads, smem, st>>>((const T *)k, (const T *)v, Hkv, L_stride,
                                           c->max_groups, (uint8_t *)c->records, rb);
    }
    residual_copy_kernel<T, D><<<B * Hkv, 256, 0, st>>>(
        (const T *)k, (const T *)v, B, Hkv, L, L_stride, nq, (T *)c->k_res, (T *)c->v_res,
        c->res_cap, c->n_groups, c->seq_len);
    return cudaGetLastError();
}

template <typename T, int BITS, int D>
cudaError_t launch_append(const vc_qcache *c, const void *kn, const void *vn, const int32_t *n_new,
                          const int32_t *len_base, const int32_t *n_acc, int max_new, int requantize,
                          cudaStream_t st)
{
    const size_t smem = sizeof(QSmem<D>);
    auto kern = append_kernel<T, BITS, D>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    kern<<<c->B, kThreads, smem, st>>>((const T *)kn, (const T *)vn, n_new, len_base, n_acc, max_new, c->Hkv,
                                       (T *)c->k_res, (T *)c->v_res, c->res_cap, c->cfg.residual,
                                       requantize, c->max_groups, (uint8_t *)c->records,
                                       vc_record_bytes(BITS, D), c->n_groups, c->seq_len,
                                       c->status);
    return cudaGetLastError();
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
