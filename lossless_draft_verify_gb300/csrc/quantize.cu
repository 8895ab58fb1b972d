// quantize.cu -- KIVI-style asymmetric group quantization of the draft cache
// (KIVI: a compressor named on the VeriCache paper page, "What the paper
// found"; ref [42] on pith.science).  K per channel over groups of 32 tokens,
// V per token over groups of 32 channels, fp16 scale and zero-point per group,
// packed into the record layout the draft kernel consumes (include/vc.h).
//
// One CTA of 2*d threads quantizes one (sequence, kv head, token group):
// threads [0, d) own one K channel each (32 tokens), threads [d, 2d) own one
// V (token, channel group) each.  Every thread reads its 32 inputs straight
// from global memory, reduces min/max, derives the directed-rounded fp16
// meta, computes the codes and ORs them into the record image in shared
// memory at their fragment-order position; the image is then written with
// 128-bit stores.  The quotient (x - z)/s is evaluated with the group's
// reciprocal and recomputed with an exact IEEE division whenever it lies
// within rounding distance of a half-integer, so the codes are those of the
// correctly rounded quotient.  HBM-bound: reads 2*32*d*2 bytes, writes one
// record per group.
#include <cooperative_groups.h>

#include "vc_common.cuh"
#include "vc_internal.h"

namespace cg = cooperative_groups;

namespace vc {
namespace {

constexpr int G = 32;

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

// code = clamp(rint(RN(RN(x - z) / s)), 0, qmax); rs = RN(1/s).  d * rs is
// within a few ulp of RN(d / s) (q <= 15), so away from a half-integer both
// round to the same integer; near one the exact quotient decides.
__device__ __noinline__ float exact_quotient(float d, float s) { return __fdiv_rn(d, s); }

__device__ __forceinline__ uint32_t group_code(float x, float sf, float zf, float rs, int qmax)
{
    if (sf == 0.0f) return 0u;
    const float d = __fadd_rn(x, -zf);
    const float q = d * rs;
    float r = rintf(q);
    if (fabsf(q - r) > 0.49999f) r = rintf(exact_quotient(d, sf));   // rare: near a half-integer
    r = fminf(fmaxf(r, 0.0f), (float)qmax);
    return (uint32_t)r;
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

// Quantize one group whose token rows are row(t) (t in [0, 32)); threads
// [0, D) must be given K rows and threads [D, 2D) V rows.  Writes `rec`.
// blockDim.x == 2 * D; img is a shared record image.
template <typename T, int BITS, int D, typename RowFn>
__device__ void quantize_group(RowFn row, uint8_t *__restrict__ rec, uint32_t *img)
{
    using Gm = RecGeom<BITS, D>;
    constexpr int qmax = (1 << BITS) - 1;
    constexpr int NG = D / G;
    const int tid = threadIdx.x;
    uint8_t *bimg = reinterpret_cast<uint8_t *>(img);
    for (int i = tid; i < Gm::REC / 4; i += 2 * D) img[i] = 0u;
    __syncthreads();
    if (tid < D) {
        // ---- K: channel c over the group's 32 tokens
        const int c = tid;
        float x[G];
#pragma unroll
        for (int t = 0; t < G; ++t) x[t] = Elem<T>::to_f(row(t)[c]);
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int t = 1; t < G; ++t) {
            mn = fminf(mn, x[t]);
            mx = fmaxf(mx, x[t]);
        }
        uint16_t sb, zb;
        float sf, zf;
        group_params(mn, mx, qmax, sb, zb, sf, zf);
        const float rs = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
        const int ks = c >> 4, col = c & 15;
        const int tig = (col & 7) >> 1, hh = col & 1, rh = col >> 3;
        const int kappa = 2 * ks + rh;
        // token t = 16 (mu/2) + 8 (mu%2) + gid goes to lane 4 gid + tig, word
        // w(mu), shift sh(mu): the four (word, shift) of this channel, once
        int base[4], sh[4];
#pragma unroll
        for (int mu = 0; mu < 4; ++mu) {
            int w, sl;
            pair_pos<BITS, D>(kappa, mu, w, sl);
            base[mu] = word_byte(tig, w);
            sh[mu] = BITS * sl + 16 * hh;
        }
        const bool pair01 = base[0] == base[1], pair23 = base[2] == base[3];
#pragma unroll
        for (int gid = 0; gid < 8; ++gid) {
            uint32_t cd[4];
#pragma unroll
            for (int mu = 0; mu < 4; ++mu)
                cd[mu] = group_code(x[16 * (mu >> 1) + 8 * (mu & 1) + gid], sf, zf, rs, qmax) << sh[mu];
            uint32_t *w0 = reinterpret_cast<uint32_t *>(bimg + base[0] + 64 * gid);
            uint32_t *w2 = reinterpret_cast<uint32_t *>(bimg + base[2] + 64 * gid);
            if (pair01) {
                if (cd[0] | cd[1]) atomicOr(w0, cd[0] | cd[1]);
            } else {
                if (cd[0]) atomicOr(w0, cd[0]);
                if (cd[1]) atomicOr(reinterpret_cast<uint32_t *>(bimg + base[1] + 64 * gid), cd[1]);
            }
            if (pair23) {
                if (cd[2] | cd[3]) atomicOr(w2, cd[2] | cd[3]);
            } else {
                if (cd[2]) atomicOr(w2, cd[2]);
                if (cd[3]) atomicOr(reinterpret_cast<uint32_t *>(bimg + base[3] + 64 * gid), cd[3]);
            }
        }
        // meta: pair n = 2 ks + rr of quad j, half (c & 1)
        const int j = tig, n = 2 * ks + rh;
        const int off = Gm::KM + 16 * (4 * (n >> 2) + j) + 4 * (n & 3) + 2 * (c & 1);
        *reinterpret_cast<uint16_t *>(bimg + off) = sb;
        *reinterpret_cast<uint16_t *>(bimg + off + 2 * D) = zb;
    } else if (tid < 2 * D) {
        // ---- V: token t over channel group gc
        const int i = tid - D;
        const int t = i % G, gc = i / G;
        float x[G];
        const T *src = row(t) + gc * G;
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int e = 0; e < G; e += 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(src + e);
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    x[e + 2 * k] = bf16_lo(wv[k]);
                    x[e + 2 * k + 1] = bf16_hi(wv[k]);
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < G; e += 4) {
                const float4 u = *reinterpret_cast<const float4 *>(src + e);
                x[e] = u.x; x[e + 1] = u.y; x[e + 2] = u.z; x[e + 3] = u.w;
            }
        }
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int e = 1; e < G; ++e) {
            mn = fminf(mn, x[e]);
            mx = fmaxf(mx, x[e]);
        }
        uint16_t sb, zb;
        float sf, zf;
        group_params(mn, mx, qmax, sb, zb, sf, zf);
        const float rs = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
        const int ks = t >> 4, colt = t & 15;
        const int tig = (colt & 7) >> 1, hh = colt & 1, rh = colt >> 3;
        const int mu = 2 * ks + rh;
        uint8_t *vsec = bimg + Gm::CODE;
        // channel c = 32 gc + 8 m + gid (m = e / 8) has class kappa = 4 gc + m
        // and goes to lane 4 gid + tig: the four (word, shift), once
        int base[4], sh[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            int w, sl;
            pair_pos<BITS, D>(4 * gc + m, mu, w, sl);
            base[m] = word_byte(tig, w);
            sh[m] = BITS * sl + 16 * hh;
        }
#pragma unroll
        for (int e = 0; e < G; ++e) {
            const int m = e >> 3, gid = e & 7;
            const uint32_t code = group_code(x[e], sf, zf, rs, qmax);
            if (code) atomicOr(reinterpret_cast<uint32_t *>(vsec + base[m] + 64 * gid), code << sh[m]);
        }
        const int j = tig, n = (2 * ks + rh) * NG + gc;
        const int off = Gm::VM + 16 * (4 * (n >> 2) + j) + 4 * (n & 3) + 2 * (t & 1);
        *reinterpret_cast<uint16_t *>(bimg + off) = sb;
        *reinterpret_cast<uint16_t *>(bimg + off + 2 * D) = zb;
    }
    __syncthreads();
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

template <typename T, int BITS, int D, bool ROT>
__global__ void __launch_bounds__(2 * D, 5)
quantize_prefill_kernel(const T *__restrict__ k, const T *__restrict__ v, int Hkv, int L_stride,
                        int max_groups, uint8_t *__restrict__ records)
{
    using Gm = RecGeom<BITS, D>;
    __shared__ __align__(16) uint32_t img[Gm::REC / 4];
    const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * Hkv + h;
    const size_t row0 = bh * L_stride + (size_t)g * G;
    if constexpr (ROT) {
        // the group's key rows, rotated, in shared memory
        __shared__ __align__(16) float buf[G][D];
        __shared__ __align__(16) T kr[G][D];
        rotate_rows<T, D, G>(
            G, [&](int t) { return k + (row0 + t) * D; }, [&](int t) { return &kr[t][0]; }, buf);
        auto row = [&](int t) -> const T * { return threadIdx.x < D ? &kr[t][0] : v + (row0 + t) * D; };
        quantize_group<T, BITS, D>(row, records + (bh * max_groups + g) * Gm::REC, img);
    } else {
        const T *base = threadIdx.x < D ? k : v;
        auto row = [&](int t) { return base + (row0 + t) * D; };
        quantize_group<T, BITS, D>(row, records + (bh * max_groups + g) * Gm::REC, img);
    }
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
    __shared__ __align__(16) uint32_t img[Gm::REC / 4];
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
            const T *ring = threadIdx.x < D ? kres : vres;
            auto row = [&](int t) {
                return ring + (bh * res_cap + (size_t)(((long)g * G + t) % res_cap)) * D;
            };
            quantize_group<T, BITS, D>(row, records + (bh * max_groups + g) * Gm::REC, img);
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
        if (rot)
            quantize_prefill_kernel<T, BITS, D, true><<<grid, 2 * D, 0, st>>>(
                (const T *)k, (const T *)v, Hkv, L_stride, c->max_groups, (uint8_t *)c->records);
        else
            quantize_prefill_kernel<T, BITS, D, false><<<grid, 2 * D, 0, st>>>(
                (const T *)k, (const T *)v, Hkv, L_stride, c->max_groups, (uint8_t *)c->records);
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
