// kvpack.cu -- lossless packing of bf16 K/V rows for the host link, and the
// expansion back to bf16 on the GPU.
//
// The full-KV swap-in (VeriCache paper page, "What the paper found": the
// exact KV state is copied in over the interconnect while drafting runs) is
// bound by the link, not by HBM.  Held packed on the host, the cache moves
// 16 + 3d/2 bytes per row instead of 2d (208 instead of 256 at d = 128), and
// an HBM-bound kernel restores every bf16 bit on the GPU.  Row format
// (include/vc.h): base exponent = largest exponent field - 14 (floored at 0),
// a 4-bit code per value (field - base, or 15 when the field lies below the
// window), up to 7 (index, field) escape slots, and each value's sign and
// mantissa byte.  A row with more than 7 escapes is marked (n_esc = 255) and
// counted; it cannot be expanded.
//
// One warp per row: lane l holds values [l * d/32, (l + 1) * d/32), so the
// codes, the sign|mantissa bytes and the escape order (ascending index, by a
// prefix count over the lanes) follow from the lane index.
#include <algorithm>

#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kSlots = 7;
constexpr int kPackThreads = 256;

template <int D>
struct PackGeom {
    static constexpr int VPL = D / 32;              // values per lane
    static constexpr int ROW = 16 + 3 * D / 2;      // packed row bytes
    static constexpr int NIB = 16;                  // codes start here
    static constexpr int SM = 16 + D / 2;           // sign|mantissa bytes start here
};

// VPL bf16 values of a lane as one 32- or 64-bit word
template <int VPL> struct LaneWord;
template <> struct LaneWord<2> { using T = uint32_t; };
template <> struct LaneWord<4> { using T = uint2; };

template <int VPL>
__device__ __forceinline__ void split_word(typename LaneWord<VPL>::T w, uint32_t (&v)[VPL])
{
    if constexpr (VPL == 2) {
        v[0] = w & 0xFFFFu;
        v[1] = w >> 16;
    } else {
        v[0] = w.x & 0xFFFFu;
        v[1] = w.x >> 16;
        v[2] = w.y & 0xFFFFu;
        v[3] = w.y >> 16;
    }
}

// Pack one row by one warp.  h: this warp's 16-byte shared header image.
template <int D>
__device__ __forceinline__ void pack_row(const uint16_t *__restrict__ src_row, uint8_t *row, uint8_t *h, int lane,
                                         int32_t *n_over)
{
    using Gm = PackGeom<D>;
    constexpr int VPL = Gm::VPL;
    using W = typename LaneWord<VPL>::T;
    uint32_t v[VPL];
    split_word<VPL>(reinterpret_cast<const W *>(src_row)[lane], v);
    uint32_t emax = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) emax = max(emax, (v[i] >> 7) & 0xFFu);
    emax = __reduce_max_sync(0xffffffffu, emax);
    const int base = emax >= 14 ? (int)emax - 14 : 0;
    uint32_t code[VPL];
    int nesc = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int c = (int)((v[i] >> 7) & 0xFFu) - base;     // <= 14 by the choice of base
        code[i] = c < 0 ? 15u : (uint32_t)c;
        nesc += c < 0;
    }
    int incl = nesc;                                         // inclusive prefix count over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    // header: zeroed, escape slots filled by their owners, then the counts
    __syncwarp();                                            // h may still be read for the previous row
    if (lane < 4) reinterpret_cast<uint32_t *>(h)[lane] = 0u;
    __syncwarp();
    int slot = incl - nesc;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (code[i] == 15u) {
            if (slot < kSlots) {
                h[2 + 2 * slot] = (uint8_t)(lane * VPL + i);
                h[3 + 2 * slot] = (uint8_t)((v[i] >> 7) & 0xFFu);
            }
            ++slot;
        }
    __syncwarp();
    if (lane == 0) {
        h[0] = (uint8_t)base;
        h[1] = total > kSlots ? 255 : (uint8_t)total;
        if (total > kSlots && n_over) atomicAdd(n_over, 1);
    }
    __syncwarp();
    if (lane < 4) reinterpret_cast<uint32_t *>(row)[lane] = reinterpret_cast<const uint32_t *>(h)[lane];
    uint32_t nib = 0, sm = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        nib |= code[i] << (4 * i);
        sm |= (((v[i] >> 8) & 0x80u) | (v[i] & 0x7Fu)) << (8 * i);
    }
    if constexpr (VPL == 2) {
        row[Gm::NIB + lane] = (uint8_t)nib;
        reinterpret_cast<uint16_t *>(row + Gm::SM)[lane] = (uint16_t)sm;
    } else {
        reinterpret_cast<uint16_t *>(row + Gm::NIB)[lane] = (uint16_t)nib;
        reinterpret_cast<uint32_t *>(row + Gm::SM)[lane] = sm;
    }
}

template <int D>
__global__ void __launch_bounds__(kPackThreads)
kv_pack_kernel(const uint16_t *__restrict__ src, uint8_t *__restrict__ dst, long long rows, int32_t *n_over)
{
    __shared__ __align__(16) uint8_t hdr[kPackThreads / 32][16];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long nw = (long long)gridDim.x * (kPackThreads / 32);
    for (long long r = (long long)blockIdx.x * (kPackThreads / 32) + wib; r < rows; r += nw)
        pack_row<D>(src + r * D, dst + r * PackGeom<D>::ROW, hdr[wib], lane, n_over);
}

// After acceptance: the n_acc[b] + 1 committed rows of the verify block (K
// and V, every layer) packed into the host copy at positions ctx[b] + i.
// One warp per (layer, sequence-head, row).
template <int D>
__global__ void __launch_bounds__(kPackThreads)
kv_writeback_packed_kernel(const uint16_t *__restrict__ kb, const uint16_t *__restrict__ vb, int n_layers, int B,
                           int Hkv, int Dq, const int32_t *__restrict__ n_acc, const int32_t *__restrict__ ctx,
                           uint8_t *kh, uint8_t *vh, int L_stride, int32_t *n_over)
{
    __shared__ __align__(16) uint8_t hdr[kPackThreads / 32][16];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long rows = (long long)n_layers * B * Hkv * Dq;
    const long long nw = (long long)gridDim.x * (kPackThreads / 32);
    for (long long r = (long long)blockIdx.x * (kPackThreads / 32) + wib; r < rows; r += nw) {
        const int i = (int)(r % Dq);
        const long long lbh = r / Dq;                       // (layer * B + b) * Hkv + h
        const int b = (int)((lbh / Hkv) % B);
        const int pos = ctx[b] + i;
        if (i > n_acc[b] || pos >= L_stride) continue;      // uniform over the warp
        const long long dst = lbh * L_stride + pos;
        pack_row<D>(kb + r * D, kh + dst * PackGeom<D>::ROW, hdr[wib], lane, n_over);
        pack_row<D>(vb + r * D, vh + dst * PackGeom<D>::ROW, hdr[wib], lane, n_over);
    }
}

// Expansion: RPI rows per warp and iteration, their loads issued together.
template <int D>
__global__ void __launch_bounds__(kPackThreads)
kv_unpack_kernel(const uint8_t *__restrict__ src, uint16_t *__restrict__ dst, long long rows)
{
    using Gm = PackGeom<D>;
    constexpr int VPL = Gm::VPL;
    constexpr int RPI = 8;
    const int lane = threadIdx.x & 31;
    const long long w0 = (long long)blockIdx.x * (kPackThreads / 32) + (threadIdx.x >> 5);
    const long long nw = (long long)gridDim.x * (kPackThreads / 32);
    for (long long r0 = w0 * RPI; r0 < rows; r0 += nw * RPI) {
        uint4 hd[RPI];
        uint32_t nib[RPI], sm[RPI];
#pragma unroll
        for (int k = 0; k < RPI; ++k) {
            const long long r = min(r0 + k, rows - 1);
            const uint8_t *row = src + r * Gm::ROW;
            hd[k] = *reinterpret_cast<const uint4 *>(row);
            if constexpr (VPL == 2) {
                nib[k] = row[Gm::NIB + lane];
                sm[k] = reinterpret_cast<const uint16_t *>(row + Gm::SM)[lane];
            } else {
                nib[k] = reinterpret_cast<const uint16_t *>(row + Gm::NIB)[lane];
                sm[k] = reinterpret_cast<const uint32_t *>(row + Gm::SM)[lane];
            }
        }
#pragma unroll
        for (int k = 0; k < RPI; ++k) {
            if (r0 + k >= rows) break;
            const uint32_t base = hd[k].x & 0xFFu;
            const int n = min((int)((hd[k].x >> 8) & 0xFFu), kSlots);
            uint32_t e[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) e[i] = base + ((nib[k] >> (4 * i)) & 15u);
            // escape slots: byte 2 + 2j is the index, byte 3 + 2j the field
            const uint32_t hw[4] = {hd[k].x, hd[k].y, hd[k].z, hd[k].w};
#pragma unroll
            for (int j = 0; j < kSlots; ++j) {
                if (j >= n) break;
                const uint32_t pair = (hw[(2 + 2 * j) >> 2] >> (8 * ((2 + 2 * j) & 3))) & 0xFFFFu;
                const int idx = (int)(pair & 0xFFu) - lane * VPL;
#pragma unroll
                for (int i = 0; i < VPL; ++i)
                    if (idx == i) e[i] = pair >> 8;
            }
            uint32_t out[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                const uint32_t b = (sm[k] >> (8 * i)) & 0xFFu;
                out[i] = ((b & 0x80u) << 8) | ((e[i] & 0xFFu) << 7) | (b & 0x7Fu);
            }
            uint16_t *d = dst + (r0 + k) * D;
            if constexpr (VPL == 2) {
                reinterpret_cast<uint32_t *>(d)[lane] = out[0] | (out[1] << 16);
            } else {
                reinterpret_cast<uint2 *>(d)[lane] = make_uint2(out[0] | (out[1] << 16), out[2] | (out[3] << 16));
            }
        }
    }
}

unsigned pack_grid(long long rows, int rows_per_warp)
{
    const long long warps = (rows + rows_per_warp - 1) / rows_per_warp;
    const long long blocks = (warps + kPackThreads / 32 - 1) / (kPackThreads / 32);
    const long long cap = (long long)device_sm_count() * 8;
    return (unsigned)std::max<long long>(1, std::min(blocks, cap));
}

}  // namespace

cudaError_t kv_pack(const void *src, void *dst, long long rows, int d, int32_t *n_over, cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    const unsigned g = pack_grid(rows, 1);
    if (d == 128)
        kv_pack_kernel<128><<<g, kPackThreads, 0, st>>>((const uint16_t *)src, (uint8_t *)dst, rows, n_over);
    else
        kv_pack_kernel<64><<<g, kPackThreads, 0, st>>>((const uint16_t *)src, (uint8_t *)dst, rows, n_over);
    return cudaGetLastError();
}

cudaError_t kv_unpack(const void *src, void *dst, long long rows, int d, cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    const unsigned g = pack_grid(rows, 8);
    if (d == 128)
        kv_unpack_kernel<128><<<g, kPackThreads, 0, st>>>((const uint8_t *)src, (uint16_t *)dst, rows);
    else
        kv_unpack_kernel<64><<<g, kPackThreads, 0, st>>>((const uint8_t *)src, (uint16_t *)dst, rows);
    return cudaGetLastError();
}

cudaError_t kv_writeback_packed(const void *kb, const void *vb, int n_layers, int B, int Hkv, int Dq, int d,
                                const int32_t *n_acc, const int32_t *ctx, void *kh, void *vh, int L_stride,
                                int32_t *n_over, cudaStream_t st)
{
    const long long rows = (long long)n_layers * B * Hkv * Dq;
    if (rows <= 0) return cudaSuccess;
    const unsigned g = pack_grid(rows, 1);
    if (d == 128)
        kv_writeback_packed_kernel<128><<<g, kPackThreads, 0, st>>>((const uint16_t *)kb, (const uint16_t *)vb,
                                                                    n_layers, B, Hkv, Dq, n_acc, ctx, (uint8_t *)kh,
                                                                    (uint8_t *)vh, L_stride, n_over);
    else
        kv_writeback_packed_kernel<64><<<g, kPackThreads, 0, st>>>((const uint16_t *)kb, (const uint16_t *)vb,
                                                                   n_layers, B, Hkv, Dq, n_acc, ctx, (uint8_t *)kh,
                                                                   (uint8_t *)vh, L_stride, n_over);
    return cudaGetLastError();
}

}  // namespace vc

using namespace vc;

extern "C" {

size_t vc_kv_packed_row_bytes(int d)
{
    return (d == 64 || d == 128) ? (size_t)(16 + 3 * d / 2) : 0;
}

vc_status vc_kv_pack(const void *src_bf16, void *dst_packed, int64_t rows, int d, int32_t *n_over,
                     cudaStream_t stream)
{
    if (rows < 0 || (d != 64 && d != 128)) return rows < 0 ? VC_ERR_INVALID : VC_ERR_UNSUPPORTED;
    if (rows == 0) return VC_OK;
    if (!src_bf16 || !dst_packed || ((uintptr_t)src_bf16 & 7u) || ((uintptr_t)dst_packed & 15u) ||
        ((uintptr_t)n_over & 3u))
        return VC_ERR_INVALID;
    return kv_pack(src_bf16, dst_packed, rows, d, n_over, stream) == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

vc_status vc_kv_writeback_packed(const void *k_blk, const void *v_blk, int n_layers, int B, int Hkv, int Dq, int d,
                                 const int32_t *n_acc, const int32_t *ctx_len, void *k_host_packed,
                                 void *v_host_packed, int L_stride, int32_t *n_over, cudaStream_t stream)
{
    if (!k_blk || !v_blk || !n_acc || !ctx_len || !k_host_packed || !v_host_packed) return VC_ERR_INVALID;
    if (n_layers <= 0 || B <= 0 || Hkv <= 0 || Dq <= 0 || L_stride < Dq) return VC_ERR_INVALID;
    if (d != 64 && d != 128) return VC_ERR_UNSUPPORTED;
    if (((uintptr_t)k_blk & 7u) || ((uintptr_t)v_blk & 7u) || ((uintptr_t)k_host_packed & 15u) ||
        ((uintptr_t)v_host_packed & 15u) || ((uintptr_t)n_over & 3u))
        return VC_ERR_INVALID;
    void *kd = nullptr, *vd = nullptr;
    if (cudaHostGetDevicePointer(&kd, k_host_packed, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&vd, v_host_packed, 0) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_INVALID;
    }
    return kv_writeback_packed(k_blk, v_blk, n_layers, B, Hkv, Dq, d, n_acc, ctx_len, kd, vd, L_stride, n_over,
                               stream) == cudaSuccess
               ? VC_OK
               : VC_ERR_CUDA;
}

vc_status vc_kv_unpack(const void *src_packed, void *dst_bf16, int64_t rows, int d, cudaStream_t stream)
{
    if (rows < 0 || (d != 64 && d != 128)) return rows < 0 ? VC_ERR_INVALID : VC_ERR_UNSUPPORTED;
    if (rows == 0) return VC_OK;
    if (!src_packed || !dst_bf16 || ((uintptr_t)src_packed & 15u) || ((uintptr_t)dst_bf16 & 7u))
        return VC_ERR_INVALID;
    return kv_unpack(src_packed, dst_bf16, rows, d, stream) == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // extern "C"
