// accept.cu -- greedy acceptance of a drafted block (the greedy rule of
// speculative decoding, source 2 on the podparley page; output identical to
// full-KV greedy decoding, VeriCache paper page "What the paper found").
//
// One pass over the verify logits [B][D+1][V]: every (row, split) CTA scans a
// contiguous slice with 128-bit streaming loads and reduces (value, index)
// pairs -- larger value wins, equal values keep the lower index, so -0 and +0
// tie -- through warp shuffles and shared memory.  The last CTA to finish a
// sequence (device-scope counter, returned to zero by that CTA) folds the split
// partials of its D+1 rows, finds the first row whose argmax differs from the
// draft, and writes n_acc and next_tok.  HBM-bound: the algorithmic traffic is the logits once.
#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kThreads = 256;

struct ArgMax {
    float v;
    int i;
};

__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b)
{
    // larger value wins; on equal values the lower index wins
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax b;
        b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
        b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
        a = better(a, b);
    }
    return a;
}

struct WsLayout {
    int32_t *status;
    unsigned int *counters;   // [B]
    ArgMax *part;             // [rows][S]
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int splits_for(int V) { return V >= 65536 ? 4 : (V >= 16384 ? 2 : 1); }   // at most 4

__host__ __device__ inline WsLayout ws_layout(void *ws, int B)
{
    uint8_t *p = (uint8_t *)ws;
    WsLayout L;
    L.status = (int32_t *)p;
    L.counters = (unsigned int *)(p + kStatusBytes);
    L.part = (ArgMax *)(p + kStatusBytes + align256((size_t)B * 4));
    return L;
}

template <typename T>
__device__ __forceinline__ void scan_vec(const T *row, int lo, int hi, ArgMax &best)
{
    constexpr int PER = 16 / sizeof(T);
    // lo, hi are multiples of PER; row is 16-byte aligned
    int i = lo + threadIdx.x * PER;
    constexpr int UNROLL = 8;
    for (; i + (UNROLL - 1) * kThreads * PER < hi; i += UNROLL * kThreads * PER) {
        uint4 u[UNROLL];
#pragma unroll
        for (int r = 0; r < UNROLL; ++r) u[r] = ldg_stream(row + i + r * kThreads * PER);
#pragma unroll
        for (int r = 0; r < UNROLL; ++r) {
            const uint32_t w[4] = {u[r].x, u[r].y, u[r].z, u[r].w};
            const int base = i + r * kThreads * PER;
            if constexpr (sizeof(T) == 2) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
                    if (a > best.v) { best.v = a; best.i = base + 2 * e; }
                    if (b > best.v) { best.v = b; best.i = base + 2 * e + 1; }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float a = __uint_as_float(w[e]);
                    if (a > best.v) { best.v = a; best.i = base + e; }
                }
            }
        }
    }
    for (; i < hi; i += kThreads * PER) {
        uint4 u = ldg_stream(row + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
                if (a > best.v) { best.v = a; best.i = i + 2 * e; }
                if (b > best.v) { best.v = b; best.i = i + 2 * e + 1; }
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float a = __uint_as_float(w[e]);
                if (a > best.v) { best.v = a; best.i = i + e; }
            }
        }
    }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads)
accept_kernel(const T *__restrict__ logits, const int32_t *__restrict__ drafts, int B, int D,
              int V, int S, int chunk, int32_t *__restrict__ n_acc, int32_t *__restrict__ next_tok,
              void *ws)
{
    pdl_wait();
    pdl_trigger();
    const WsLayout W = ws_layout(ws, B);
    const int s = blockIdx.x, row = blockIdx.y;
    const int b = row / (D + 1);
    const T *rp = logits + (size_t)row * V;
    const int lo = s * chunk, hi = min(V, lo + chunk);
    // Threads scan increasing indices, so a strict '>' keeps the first
    // occurrence of a tie inside each thread's subsequence.
    ArgMax best{-INFINITY, 0x7fffffff};
    if (VEC) {
        scan_vec<T>(rp, lo, hi, best);
    } else {
        for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
            float a = Elem<T>::to_f(rp[i]);
            if (a > best.v) { best.v = a; best.i = i; }
        }
    }
    __shared__ ArgMax red[kThreads / 32];
    __shared__ bool is_last;
    best = warp_argmax(best);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        ArgMax a = red[0];
        for (int w = 1; w < kThreads / 32; ++w) a = better(a, red[w]);
        W.part[(size_t)row * S + s] = a;
        __threadfence();
        const unsigned int done = atomicAdd(&W.counters[b], 1u);
        is_last = (done == (unsigned int)((D + 1) * S - 1));
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // Last CTA of sequence b: fold the partials of its D+1 rows (a row's S
    // partials requested together, folded in split order), then the accepted
    // length is the first row whose argmax differs from its draft: every row
    // compares its own draft, and the lowest mismatching row wins.
    __shared__ int amax[1024 + 1];
    __shared__ int first_miss;
    if (threadIdx.x == 0) first_miss = D;
    __syncthreads();
    constexpr int kMaxS = 4;                      // splits_for() never exceeds it
    for (int i = threadIdx.x; i <= D; i += kThreads) {
        const ArgMax *pp = W.part + (size_t)(b * (D + 1) + i) * S;
        ArgMax c[kMaxS];
#pragma unroll
        for (int t = 0; t < kMaxS; ++t)
            if (t < S) {
                c[t].v = __ldcg(&pp[t].v);
                c[t].i = __ldcg(&pp[t].i);
            }
        const int dr = i < D ? drafts[(size_t)b * D + i] : -1;
        ArgMax a = c[0];
#pragma unroll
        for (int t = 1; t < kMaxS; ++t)
            if (t < S) a = better(a, c[t]);
        amax[i] = a.i;
        if (i < D && a.i != dr) atomicMin(&first_miss, i);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int n = first_miss;
        n_acc[b] = n;
        next_tok[b] = amax[n];
        W.counters[b] = 0u;                 // every CTA of b has arrived: ready for the next call
    }
}

template <typename T>
cudaError_t launch(const void *logits, const int32_t *drafts, int B, int D, int V, int32_t *n_acc,
                   int32_t *next_tok, void *ws, bool clear_counters, cudaStream_t st)
{
    constexpr int PER = 16 / sizeof(T);
    const WsLayout W = ws_layout(ws, B);
    if (clear_counters) {
        const cudaError_t e = cudaMemsetAsync(W.counters, 0, (size_t)B * 4, st);
        if (e != cudaSuccess) return e;
    }
    const int S = splits_for(V);
    const bool vec = ((uintptr_t)logits % 16 == 0) && (V % PER == 0);
    int chunk = cdiv(V, S);
    if (vec) chunk = cdiv(chunk, PER) * PER;
    dim3 grid(S, B * (D + 1));
    auto kern = vec ? accept_kernel<T, true> : accept_kernel<T, false>;
    if (clear_counters) {
        // after the memset: a plain launch (the kernel's grid-dependency wait is then a no-op)
        kern<<<grid, kThreads, 0, st>>>((const T *)logits, drafts, B, D, V, S, chunk, n_acc, next_tok, ws);
        return cudaGetLastError();
    }
    return launch_pdl(kern, grid, dim3(kThreads), 0, st, (const T *)logits, drafts, B, D, V, S, chunk, n_acc,
                      next_tok, ws);
}

// Acceptance from the LM head's tile maxima ([B][D+1][n_tiles] value and
// column of each 128-column tile's first maximum): a warp per row folds the
// tiles with the same order (larger value, then lower column) and compares
// the row's argmax with its draft; the lowest mismatching row ends the
// accepted prefix (the greedy rule).
__global__ void __launch_bounds__(kThreads)
accept_tiles_kernel(const float *__restrict__ tmax, const int32_t *__restrict__ tidx, int n_tiles,
                    const int32_t *__restrict__ drafts, int D, int32_t *__restrict__ n_acc,
                    int32_t *__restrict__ next_tok)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int amax[1024 + 1];
    __shared__ int first_miss;
    if (threadIdx.x == 0) first_miss = D;
    __syncthreads();
    for (int i = warp; i <= D; i += kThreads / 32) {
        const size_t row = (size_t)b * (D + 1) + i;
        const int dr = (lane == 0 && i < D) ? drafts[(size_t)b * D + i] : -1;
        ArgMax best{-INFINITY, 0x7fffffff};
        for (int t = lane; t < n_tiles; t += 32)
            best = better(best, ArgMax{tmax[row * n_tiles + t], tidx[row * n_tiles + t]});
        best = warp_argmax(best);
        if (lane == 0) {
            amax[i] = best.i;
            if (i < D && best.i != dr) atomicMin(&first_miss, i);   // the lowest mismatching row wins
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int n = first_miss;
        n_acc[b] = n;
        next_tok[b] = amax[n];
    }
}

}  // namespace

cudaError_t accept_tiles(const float *tile_max, const int32_t *tile_idx, int n_tiles, const int32_t *drafts,
                         int B, int D, int32_t *n_acc, int32_t *next_tok, cudaStream_t st)
{
    return launch_pdl(accept_tiles_kernel, dim3(B), dim3(kThreads), 0, st, tile_max, tile_idx, n_tiles, drafts, D,
                      n_acc, next_tok);
}

size_t accept_ws_bytes(int B, int D, int V)
{
    return kStatusBytes + align256((size_t)B * 4) +
           align256((size_t)B * (D + 1) * splits_for(V) * sizeof(ArgMax));
}

cudaError_t accept(const void *logits, vc_dtype dt, const int32_t *drafts, int B, int D, int V,
                   int32_t *n_acc, int32_t *next_tok, void *ws, cudaStream_t st, bool clear_counters)
{
    return dt == VC_BF16 ? launch<__nv_bfloat16>(logits, drafts, B, D, V, n_acc, next_tok, ws, clear_counters, st)
                         : launch<float>(logits, drafts, B, D, V, n_acc, next_tok, ws, clear_counters, st);
}

}  // namespace vc
