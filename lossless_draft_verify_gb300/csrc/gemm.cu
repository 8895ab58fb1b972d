// gemm.cu -- the decoder's dense projections, y = x W (+ r), with row results
// that do not depend on how many rows share the launch.
//
// The draft-and-verify loop is lossless only if the verify pass over a block
// of D+1 tokens computes, for every token, exactly what one-token decoding
// computes (paper page, "What the paper found": outputs identical to full-KV
// greedy decoding; the thelatestinai page shows how far batch-dependent
// floating-point order drifts KV-cached decoding).  Both kernels here fix the
// summation order of every output element from the shapes (K, N), the split
// plan and the device alone: the split of K, the order of the splits and the
// order inside a split never depend on M.
//
// bf16 (x [M][K] and W [K][N] row-major, N a multiple of 128, K of 64):
// tcgen05 tensor cores.  One CTA per (128-row tile, 128-column tile, K split):
// warp 0 issues TMA loads of 64-wide K slices (x K-major, W MN-major, 128-byte
// swizzle) into a 3-stage ring (2 CTAs per SM; draft steps with M <= 16 load
// only 16 x rows per stage and keep 6 stages), warp 1 issues tcgen05.mma (M128 N128 K16)
// into a TMEM accumulator, warps 2-5 read TMEM and write either the output
// (one split) or fp32 partials; the last CTA of each output tile to finish
// (a self-resetting counter per tile in the workspace) sums them in split order.
// Argmax epilogue (the LM head of greedy decoding): instead of the bf16 output,
// each (row, 128-column tile) yields the value and column of the first maximum
// of the bf16-rounded row, so the logits are never written.
// fp32 (any shape): CUDA cores, one output element per thread, K in order.
#include <cuda.h>

#include "tcgen05.cuh"
#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int GM = 128, GN = 128, GK = 64;
constexpr int kGemmFusedReduceTiles = 64;
constexpr int G_THREADS = 192;
constexpr uint32_t G_TMEM_COLS = 128;
constexpr int G_MAX_STAGES = 6;

// Shared-memory plan of one CTA: the x slices of every stage first, then the
// W slices.  XR = x rows actually loaded per stage (128, or 16 for draft
// steps with M <= 16: the MMA still reads 128 rows, the rows past 16 fall on
// later x stages or on W data, and their accumulator rows are never stored).
template <int XR, int STAGES>
struct GemmGeom {
    static constexpr int XB = XR * GK * 2;             // x bytes per stage
    static constexpr int WB = GK * GN * 2;             // W bytes per stage (16 KB)
    static constexpr int OFF_W = STAGES * XB;
    static constexpr int OFF_BAR = OFF_W + STAGES * WB;
    static constexpr int SMEM = OFF_BAR + 256;
    static_assert(XR == 128 || OFF_W - XB + GM * GK * 2 <= OFF_BAR, "MMA read window must stay in shared memory");
};

constexpr int kRmsMaxRows = 16;   // rows whose norm the epilogue warps compute

struct GemmBars {
    uint64_t full[G_MAX_STAGES], empty[G_MAX_STAGES], acc_full;
    float rms[kRmsMaxRows];          // 1 / rms of x's rows (row-scale epilogue)
    uint32_t tmem_base;
    int32_t abort_flag;
    int32_t is_last;
};

struct GemmArgs {
    float *part;                 // [S][M][N] fp32, used when S > 1
    unsigned int *counters;      // [m tiles][n tiles], zero between launches (S > 1)
    __nv_bfloat16 *out;          // [M][N]
    const __nv_bfloat16 *resid;  // [M][N] or null (may equal out)
    float *amax_val;             // argmax epilogue: [M][N / GN] tile maxima (out not written), or null
    int32_t *amax_idx;           // [M][N / GN] column of the first maximum in the tile
    int32_t *status;
    int M, N, K, S, kb_per_split;
    int early_w;                 // W may be read before the previous kernel completes
    int swiglu;                  // SwiGLU epilogue (S = 1): out is act [M][N / 2]
    // RMS-normalised input (draft steps, M <= 16, no residual): x is the raw
    // residual stream; every output row m is scaled by 1 / sqrt(mean_k x[m][k]^2
    // + rms_eps), which the epilogue warps compute from x while W streams in,
    // so rmsnorm(x) W needs no separate normalisation pass.  Null: off.
    const __nv_bfloat16 *rms_x;
    int rms_ld;
    float rms_eps;
};

// bf16 rounding of an output element, as the logits store would make it
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// (v, i) beats (bv, bi): larger value, the lower column on equal values
__device__ __forceinline__ bool amax_better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ bool g_wait(uint64_t *bar, uint32_t parity, GemmBars *B, int32_t *status, int where)
{
    if (mbar_wait(bar, parity)) return true;
    report_timeout(status, where);
    atomicExch(&B->abort_flag, 1);
    return false;
}

template <int XR, int GSTAGES>
__global__ void __launch_bounds__(G_THREADS, 2)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, GemmArgs A)
{
    using Gg = GemmGeom<XR, GSTAGES>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    if (smem_u32(sm) & 1023u) {
        pdl_wait();
        if (threadIdx.x == 0) report_timeout(A.status, 98);
        return;
    }
    GemmBars *B = reinterpret_cast<GemmBars *>(sm + Gg::OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * GM;
    const int n0 = blockIdx.y * GN;
    const int split = blockIdx.z;
    const int nkb = A.K / GK;
    const int kb0 = split * A.kb_per_split;
    const int kb1 = min(nkb, kb0 + A.kb_per_split);
    const int n = kb1 - kb0;                       // >= 1 by construction of S

    if (threadIdx.x == 0) {
        for (int s = 0; s < GSTAGES; ++s) {
            mbar_init(&B->full[s], 1);
            mbar_init(&B->empty[s], 1);
        }
        mbar_init(&B->acc_full, 1);
        B->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&B->tmem_base, G_TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = B->tmem_base;

    // The decoder's weights are never written while it runs: its GEMMs request
    // the first stages of W before the wait for the previous kernel, so their
    // loads overlap its tail.  x, the residual and the outputs come after it.
    const int pre = A.early_w ? min(n, GSTAGES) : 0;
    // W is read once per launch: its lines are marked evict-first, so the
    // stream does not push x, the partials and this kernel's code out of L2
    const uint64_t w_policy = l2_evict_first();
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmX);
        tc::prefetch_tmap(&tmW);
        for (int i = 0; i < pre; ++i) {
            uint8_t *sw = sm + Gg::OFF_W + i * Gg::WB;
            const int k = (kb0 + i) * GK;
            mbar_arrive_expect_tx(&B->full[i], Gg::XB + Gg::WB);
            tc::tma_load_3d_hint(sw, &tmW, n0, k, 0, &B->full[i], w_policy);
            tc::tma_load_3d_hint(sw + GK * 128, &tmW, n0 + 64, k, 0, &B->full[i], w_policy);
        }
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < n; ++i) {
                const int s = i % GSTAGES;
                const int k = (kb0 + i) * GK;
                if (i >= pre) {
                    if (!g_wait(&B->empty[s], ((i / GSTAGES) - 1) & 1, B, A.status, 41)) break;
                    if (*reinterpret_cast<volatile int32_t *>(&B->abort_flag)) break;
                    uint8_t *sw = sm + Gg::OFF_W + s * Gg::WB;
                    mbar_arrive_expect_tx(&B->full[s], Gg::XB + Gg::WB);
                    tc::tma_load_3d_hint(sw, &tmW, n0, k, 0, &B->full[s], w_policy);
                    tc::tma_load_3d_hint(sw + GK * 128, &tmW, n0 + 64, k, 0, &B->full[s], w_policy);
                }
                tc::tma_load_3d(sm + s * Gg::XB, &tmX, k, m0, 0, &B->full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(GM, GN, false, true);
            bool ok = true;
            for (int i = 0; i < n; ++i) {
                const int s = i % GSTAGES;
                if (!g_wait(&B->full[s], (i / GSTAGES) & 1, B, A.status, 42)) { ok = false; break; }
                tc::fence_after();
                const uint32_t sx = smem_u32(sm + s * Gg::XB);
                const uint32_t sw = smem_u32(sm + Gg::OFF_W + s * Gg::WB);
#pragma unroll
                for (int kk = 0; kk < GK / 16; ++kk) {
                    // x: K-major rows of 128 B, 8-row atoms 1024 B apart
                    const uint64_t ad = tc::smem_desc(sx + kk * 32, 16, 1024, tc::kSwizzle128B);
                    // W: MN-major; 64-column halves GK*128 B apart, 8 K-rows 1024 B apart
                    const uint64_t bd = tc::smem_desc(sw + kk * 2048, GK * 128, 1024, tc::kSwizzle128B);
                    tc::mma_ss(tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(&B->empty[s]);
            }
            if (ok) tc::commit(&B->acc_full);
        }
    } else {
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int m = m0 + r;
        const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16);
        float rsc = 1.f;
        if (A.rms_x) {
            // 8 epilogue threads per row (consecutive lanes of one warp), 16-byte
            // loads, then a three-step shuffle sum; the four epilogue warps meet
            // at a named barrier before reading the scales
            const int et = threadIdx.x - 64, row = et >> 3, part = et & 7;
            float ss = 0.f;
            if (row < A.M) {
                const __nv_bfloat16 *xr = A.rms_x + (size_t)row * A.rms_ld;
                for (int k = part * 8; k < A.K; k += 64) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(xr + k);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = bf16_lo(w4[e]), b = bf16_hi(w4[e]);
                        ss = fmaf(a, a, ss);
                        ss = fmaf(b, b, ss);
                    }
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            if (part == 0 && row < A.M) B->rms[row] = 1.0f / sqrtf(ss / (float)A.K + A.rms_eps);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            rsc = m < A.M ? B->rms[r] : 1.f;
        }
        const bool ok = g_wait(&B->acc_full, 0, B, A.status, 43);
        if (ok && A.swiglu) {
            // SwiGLU epilogue: columns [0, 64) of the tile are gate columns and
            // [64, 128) the matching up columns (the weight's columns are
            // interleaved per 64); act = silu(g) u from the bf16-rounded g and
            // u, the expression a separate pass over the stored product uses
            tc::fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t ug[32], uu[32];
                tc::ld32(taddr + h * 32, ug);
                tc::ld32(taddr + (h + 2) * 32, uu);
                tc::ld_wait();
                if (m < A.M) {
                    uint32_t packed[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float g0 = bf16_round(__uint_as_float(ug[c]) * rsc);
                        const float g1 = bf16_round(__uint_as_float(ug[c + 1]) * rsc);
                        const float u0 = bf16_round(__uint_as_float(uu[c]) * rsc);
                        const float u1 = bf16_round(__uint_as_float(uu[c + 1]) * rsc);
                        __nv_bfloat162 h2 = __floats2bfloat162_rn((g0 / (1.0f + expf(-g0))) * u0,
                                                                  (g1 / (1.0f + expf(-g1))) * u1);
                        packed[c / 2] = *reinterpret_cast<uint32_t *>(&h2);
                    }
                    uint4 *op = reinterpret_cast<uint4 *>(A.out + (size_t)m * (A.N / 2) + n0 / 2 + h * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        op[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
            }
        } else if (ok) {
            tc::fence_after();
            float best = -INFINITY;
            int bidx = n0;
#pragma unroll 1
            for (int h = 0; h < GN / 32; ++h) {
                uint32_t u[32];
                tc::ld32(taddr + h * 32, u);
                tc::ld_wait();
                if (A.rms_x) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) u[c] = __float_as_uint(__uint_as_float(u[c]) * rsc);
                }
                if (m < A.M) {
                    const int c0 = n0 + h * 32;
                    if (A.S == 1 && A.amax_val) {
                        // argmax epilogue: the first maximum of the bf16-rounded row
                        const __nv_bfloat16 *rp = A.resid ? A.resid + (size_t)m * A.N + c0 : nullptr;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const float v = bf16_round(__uint_as_float(u[c]) + (rp ? __bfloat162float(rp[c]) : 0.f));
                            if (v > best) {
                                best = v;
                                bidx = c0 + c;
                            }
                        }
                    } else if (A.S > 1) {
                        float *dst = A.part + ((size_t)split * A.M + m) * A.N + c0;
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            *reinterpret_cast<float4 *>(dst + c) =
                                make_float4(__uint_as_float(u[c]), __uint_as_float(u[c + 1]),
                                            __uint_as_float(u[c + 2]), __uint_as_float(u[c + 3]));
                    } else {
                        const size_t off = (size_t)m * A.N + c0;
                        uint32_t packed[16];
                        if (A.resid) {
                            const uint4 *rp = reinterpret_cast<const uint4 *>(A.resid + off);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint4 rv = rp[q];
                                const uint32_t w4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int c = q * 8 + e * 2;
                                    const float a = __uint_as_float(u[c]) + bf16_lo(w4[e]);
                                    const float b = __uint_as_float(u[c + 1]) + bf16_hi(w4[e]);
                                    __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
                                    packed[c / 2] = *reinterpret_cast<uint32_t *>(&h2);
                                }
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; c += 2) {
                                __nv_bfloat162 h2 =
                                    __floats2bfloat162_rn(__uint_as_float(u[c]), __uint_as_float(u[c + 1]));
                                packed[c / 2] = *reinterpret_cast<uint32_t *>(&h2);
                            }
                        }
                        uint4 *op = reinterpret_cast<uint4 *>(A.out + off);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            op[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    }
                }
            }
            if (A.S == 1 && A.amax_val && m < A.M) {
                const size_t t = (size_t)m * (A.N / GN) + blockIdx.y;
                A.amax_val[t] = best;
                A.amax_idx[t] = bidx;
            }
            if (A.S > 1 && A.counters) __threadfence();   // partials visible before this CTA's arrival
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tmem, G_TMEM_COLS);
    }
    if (A.S > 1 && A.counters) {
        // the last split CTA of this output tile sums the partials in split
        // order (the same order for every M) and writes the result
        const unsigned int tile = blockIdx.x * gridDim.y + blockIdx.y;
        if (threadIdx.x == 0) {
            __threadfence();
            B->is_last = atomicAdd(&A.counters[tile], 1u) == (unsigned int)(A.S - 1);
        }
        __syncthreads();
        if (B->is_last) {
            __threadfence();
            const int rows = min(GM, A.M - m0);
            const size_t plane = (size_t)A.M * A.N;
            for (int idx = threadIdx.x; idx < rows * (GN / 4); idx += G_THREADS) {
                const int m = m0 + idx / (GN / 4);
                const size_t off = (size_t)m * A.N + n0 + 4 * (idx % (GN / 4));
                // loads of up to 8 splits in flight at once, summed in split order
                float4 acc = __ldcg(reinterpret_cast<const float4 *>(A.part + off));
                for (int s0 = 1; s0 < A.S; s0 += 8) {
                    float4 p[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (s0 + j < A.S)
                            p[j] = __ldcg(reinterpret_cast<const float4 *>(A.part + (s0 + j) * plane + off));
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (s0 + j < A.S) {
                            acc.x += p[j].x;
                            acc.y += p[j].y;
                            acc.z += p[j].z;
                            acc.w += p[j].w;
                        }
                }
                if (A.resid) {
                    const uint2 r = *reinterpret_cast<const uint2 *>(A.resid + off);
                    acc.x += bf16_lo(r.x);
                    acc.y += bf16_hi(r.x);
                    acc.z += bf16_lo(r.y);
                    acc.w += bf16_hi(r.y);
                }
                if (A.amax_val) {
                    // argmax epilogue: the 32 lanes of a warp hold one row's 128
                    // columns, 4 each in column order
                    const int c = n0 + 4 * (idx % (GN / 4));
                    const float v[4] = {bf16_round(acc.x), bf16_round(acc.y), bf16_round(acc.z), bf16_round(acc.w)};
                    float bv = v[0];
                    int bi = c;
#pragma unroll
                    for (int e = 1; e < 4; ++e)
                        if (v[e] > bv) {
                            bv = v[e];
                            bi = c + e;
                        }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                        if (amax_better(ov, oi, bv, bi)) {
                            bv = ov;
                            bi = oi;
                        }
                    }
                    if ((threadIdx.x & 31) == 0) {
                        const size_t t = (size_t)m * (A.N / GN) + blockIdx.y;
                        A.amax_val[t] = bv;
                        A.amax_idx[t] = bi;
                    }
                    continue;
                }
                __nv_bfloat162 a2 = __floats2bfloat162_rn(acc.x, acc.y), b2 = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 o;
                o.x = *reinterpret_cast<uint32_t *>(&a2);
                o.y = *reinterpret_cast<uint32_t *>(&b2);
                *reinterpret_cast<uint2 *>(A.out + off) = o;
            }
            if (threadIdx.x == 0) A.counters[tile] = 0u;
        }
    }
}

// out[m][n] = bf16(sum_s part[s][m][n] (s in order) + resid[m][n]); 4 columns a thread.
__global__ void gemm_splitk_reduce(const float *__restrict__ part, int S, int M, int N,
                                   const __nv_bfloat16 *resid, __nv_bfloat16 *out)
{
    pdl_wait();
    pdl_trigger();
    const size_t i4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)M * N;
    const size_t i = i4 * 4;
    if (i >= total) return;
    float4 acc = *reinterpret_cast<const float4 *>(part + i);
    for (int s = 1; s < S; ++s) {
        const float4 p = *reinterpret_cast<const float4 *>(part + (size_t)s * total + i);
        acc.x += p.x;
        acc.y += p.y;
        acc.z += p.z;
        acc.w += p.w;
    }
    if (resid) {
        const uint2 r = *reinterpret_cast<const uint2 *>(resid + i);
        acc.x += bf16_lo(r.x);
        acc.y += bf16_hi(r.x);
        acc.z += bf16_lo(r.y);
        acc.w += bf16_hi(r.y);
    }
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&a);
    o.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(out + i) = o;
}

// CUDA-core GEMM: one output element per thread, K summed strictly in order
// (16 x 16 tiles staged through shared memory).
template <typename T>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const T *__restrict__ x, const T *__restrict__ w, const T *resid, T *out, int M, int N, int K)
{
    __shared__ float sx[16][17], sw[16][17];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m = blockIdx.y * 16 + ty, n = blockIdx.x * 16 + tx;
    float acc = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
        const int kx = k0 + tx, kw = k0 + ty;
        sx[ty][tx] = (m < M && kx < K) ? Elem<T>::to_f(x[(size_t)m * K + kx]) : 0.f;
        sw[ty][tx] = (kw < K && n < N) ? Elem<T>::to_f(w[(size_t)kw * N + n]) : 0.f;
        __syncthreads();
        const int kn = min(16, K - k0);
        for (int k = 0; k < kn; ++k) acc = fmaf(sx[ty][k], sw[k][tx], acc);
        __syncthreads();
    }
    if (m < M && n < N) {
        const size_t o = (size_t)m * N + n;
        if (resid) acc += Elem<T>::to_f(resid[o]);
        out[o] = Elem<T>::from_f(acc);
    }
}

}  // namespace

bool gemm_uses_tensor_cores(vc_dtype dt, int N, int K)
{
    return dt == VC_BF16 && N % GN == 0 && K % GK == 0 && K > 0;
}

// The K split depends on (N, K), the plan and the device only, never on M.
// kGemmRowInvariant (forward passes): few splits, so that blocks of a few row
// tiles do not pay for large fp32 partials.  kGemmDecode (draft steps, M <= one
// row tile): a product with at least one output tile per SM is not split (that
// many CTAs keep enough weight loads in flight for the HBM rate, and no
// partials are written: at M = 8 the 4096 x 28672 product measured 36.9 us
// unsplit against 42.4 us in 4 splits, the 4096 x 32000 LM head 40.6 against
// 52.2 us in 6); narrower products take the split that fills whole waves of 2
// CTAs per SM best.
int gemm_splits(int N, int K, int plan)
{
    const int ntiles = N / GN, nkb = K / GK;
    const int slots = 2 * device_sm_count();
    if (plan == kGemmRowInvariant) {
        int s = (slots / 2 + ntiles - 1) / ntiles;          // about half a wave per row tile
        s = max(1, min(s, nkb / 8));
        const int per = (nkb + s - 1) / s;
        return (nkb + per - 1) / per;
    }
    if (ntiles >= device_sm_count()) return 1;
    int best_s = 1;
    long best_cost = -1;
    for (int s = 1; s <= 16 && s <= nkb; ++s) {
        const int per = (nkb + s - 1) / s;
        const int se = (nkb + per - 1) / per;
        const long waves = ((long)ntiles * se + slots - 1) / slots;
        // time ~ waves x (K slices + about two slices of fixed CTA cost); fewer splits on ties
        const long cost = waves * (per + 2) * 64 + se;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_s = se;
        }
    }
    return best_s;
}

size_t gemm_ws_bytes(vc_dtype dt, int M, int N, int K, int plan)
{
    if (!gemm_uses_tensor_cores(dt, N, K)) return 0;
    const int S = gemm_splits(N, K, plan);
    return S > 1 ? (size_t)S * M * N * 4 : 0;
}

bool gemm_argmax_ok(vc_dtype dt, int M, int N, int K, int plan, bool have_counters)
{
    if (!gemm_uses_tensor_cores(dt, N, K)) return false;
    const int tiles = ((M + GM - 1) / GM) * (N / GN);
    return gemm_splits(N, K, plan) == 1 || (have_counters && tiles <= kGemmMaxTiles);
}

bool gemm_rms_ok(vc_dtype dt, int M, int N, int K, int ldx, int plan)
{
    return dt == VC_BF16 && (plan & ~kGemmEarlyWeights) == kGemmDecode && M > 0 && M <= kRmsMaxRows &&
           ldx % 8 == 0 && gemm_uses_tensor_cores(dt, N, K);
}

cudaError_t gemm(const void *x, const void *w, const void *resid, void *out, vc_dtype dt, int M, int N, int K,
                 int ldx, void *ws, unsigned int *counters, int32_t *status, cudaStream_t st, int plan,
                 float *amax_val, int32_t *amax_idx, float rms_eps)
{
    const bool early_w = (plan & kGemmEarlyWeights) != 0;
    const bool rms = rms_eps >= 0.f;
    if (rms && (resid || !gemm_rms_ok(dt, M, N, K, ldx, plan))) return cudaErrorNotSupported;
    plan &= ~kGemmEarlyWeights;
    if (M <= 0) return cudaSuccess;
    if (amax_val && !gemm_argmax_ok(dt, M, N, K, plan, counters != nullptr)) return cudaErrorNotSupported;
    if (gemm_uses_tensor_cores(dt, N, K)) {
        const bool small = plan == kGemmDecode && M <= 16;
        CUtensorMap mx, mw;
        if (!tma_map_bf16_3d(&mx, x, K, M, 1, (uint64_t)ldx * 2, (uint64_t)ldx * 2 * M, GK, small ? 16 : GM, 1) ||
            !tma_map_bf16_3d(&mw, w, N, K, 1, (uint64_t)N * 2, (uint64_t)N * 2 * K, 64, GK, 1))
            return cudaErrorInvalidValue;
        GemmArgs A = {};
        A.S = gemm_splits(N, K, plan);
        const int nkb = K / GK;
        A.kb_per_split = (nkb + A.S - 1) / A.S;
        A.part = (float *)ws;
        // Split-K partials are summed by the last CTA of each output tile when
        // the grid has few tiles (measured faster there: one launch less) or
        // when the argmax epilogue needs it; wider products use the
        // all-SM reduction kernel, which measured faster once many tiles
        // finish at the end of the launch (same summation order either way).
        const int tiles = ((M + GM - 1) / GM) * (N / GN);
        const bool fuse = amax_val || tiles <= kGemmFusedReduceTiles;
        A.counters = (A.S > 1 && counters && tiles <= kGemmMaxTiles && fuse) ? counters : nullptr;
        A.out = (__nv_bfloat16 *)out;
        A.resid = (const __nv_bfloat16 *)resid;
        A.amax_val = amax_val;
        A.amax_idx = amax_idx;
        A.status = status;
        A.M = M;
        A.N = N;
        A.K = K;
        A.early_w = early_w ? 1 : 0;
        A.swiglu = 0;
        A.rms_x = rms ? (const __nv_bfloat16 *)x : nullptr;
        A.rms_ld = ldx;
        A.rms_eps = rms ? rms_eps : 0.f;
        dim3 grid((M + GM - 1) / GM, N / GN, A.S);
        cudaError_t e;
        if (small) {
            using Gg = GemmGeom<16, 6>;
            cudaFuncSetAttribute(gemm_tc_kernel<16, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gg::SMEM);
            e = launch_pdl(gemm_tc_kernel<16, 6>, grid, dim3(G_THREADS), Gg::SMEM, st, mx, mw, A);
        } else {
            using Gg = GemmGeom<128, 3>;
            cudaFuncSetAttribute(gemm_tc_kernel<128, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gg::SMEM);
            e = launch_pdl(gemm_tc_kernel<128, 3>, grid, dim3(G_THREADS), Gg::SMEM, st, mx, mw, A);
        }
        if (e != cudaSuccess) return e;
        if (A.S > 1 && !A.counters) {
            const size_t q = (size_t)M * N / 4;
            return launch_pdl(gemm_splitk_reduce, dim3((unsigned)((q + 255) / 256)), dim3(256), 0, st,
                              (const float *)A.part, A.S, M, N, A.resid, A.out);
        }
        return cudaSuccess;
    }
    if (ldx != K) return cudaErrorInvalidValue;
    dim3 grid((N + 15) / 16, (M + 15) / 16);
    if (dt == VC_BF16)
        gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w,
                                                               (const __nv_bfloat16 *)resid, (__nv_bfloat16 *)out,
                                                               M, N, K);
    else
        gemm_simt_kernel<float><<<grid, 256, 0, st>>>((const float *)x, (const float *)w, (const float *)resid,
                                                       (float *)out, M, N, K);
    return cudaGetLastError();
}

bool gemm_swiglu_ok(vc_dtype dt, int F, int K, int plan)
{
    plan &= ~kGemmEarlyWeights;
    return F > 0 && F % 64 == 0 && gemm_uses_tensor_cores(dt, 2 * F, K) && gemm_splits(2 * F, K, plan) == 1;
}

cudaError_t gemm_swiglu(const void *x, const void *w, void *act, vc_dtype dt, int M, int F, int K, int ldx,
                        int32_t *status, cudaStream_t st, int plan, float rms_eps)
{
    if (!gemm_swiglu_ok(dt, F, K, plan)) return cudaErrorNotSupported;
    const bool rms = rms_eps >= 0.f;
    if (rms && !gemm_rms_ok(dt, M, 2 * F, K, ldx, plan)) return cudaErrorNotSupported;
    const bool early_w = (plan & kGemmEarlyWeights) != 0;
    plan &= ~kGemmEarlyWeights;
    if (M <= 0) return cudaSuccess;
    const int N = 2 * F;
    const bool small = plan == kGemmDecode && M <= 16;
    CUtensorMap mx, mw;
    if (!tma_map_bf16_3d(&mx, x, K, M, 1, (uint64_t)ldx * 2, (uint64_t)ldx * 2 * M, GK, small ? 16 : GM, 1) ||
        !tma_map_bf16_3d(&mw, w, N, K, 1, (uint64_t)N * 2, (uint64_t)N * 2 * K, 64, GK, 1))
        return cudaErrorInvalidValue;
    GemmArgs A = {};
    A.S = 1;
    A.kb_per_split = K / GK;
    A.part = nullptr;
    A.counters = nullptr;
    A.out = (__nv_bfloat16 *)act;
    A.resid = nullptr;
    A.amax_val = nullptr;
    A.amax_idx = nullptr;
    A.status = status;
    A.M = M;
    A.N = N;
    A.K = K;
    A.early_w = early_w ? 1 : 0;
    A.swiglu = 1;
    A.rms_x = rms ? (const __nv_bfloat16 *)x : nullptr;
    A.rms_ld = ldx;
    A.rms_eps = rms ? rms_eps : 0.f;
    dim3 grid((M + GM - 1) / GM, N / GN, 1);
    if (small) {
        using Gg = GemmGeom<16, 6>;
        cudaFuncSetAttribute(gemm_tc_kernel<16, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gg::SMEM);
        return launch_pdl(gemm_tc_kernel<16, 6>, grid, dim3(G_THREADS), Gg::SMEM, st, mx, mw, A);
    }
    using Gg = GemmGeom<128, 3>;
    cudaFuncSetAttribute(gemm_tc_kernel<128, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, Gg::SMEM);
    return launch_pdl(gemm_tc_kernel<128, 3>, grid, dim3(G_THREADS), Gg::SMEM, st, mx, mw, A);
}

}  // namespace vc
