// drop.cu -- token-dropping compressor: keep the recent window plus the
// highest accumulated-score older tokens and compact them (H2O, source 3 on
// the podparley page; KVzip 4x on the VeriCache paper page, "What the paper
// found").
//
// Selection is exact and tie-deterministic: candidates are ranked by the key
// (score descending, position ascending).  A three-pass MSB-first radix select
// (11 + 11 + 10 bits) over the order-preserving integer image of the scores
// finds the threshold key T and how many tokens tied at T must be kept (the
// lowest positions).  Compaction is an ordered two-level scan (per-chunk counts,
// a per-unit scan, a block scan inside each chunk), and the same CTAs that
// write the kept indices copy the kept K/V rows with 128-bit loads and stores.
// Everything but the row gather is a small fraction of the bytes moved.
#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr int kChunk = 4096;          // positions per CTA
constexpr int kThreads = 256;
constexpr int kPer = kChunk / kThreads;
constexpr int kBins = 2048;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// larger score -> smaller key (so the kept set is the smallest keys)
__device__ __forceinline__ uint32_t desc_key(float s)
{
    // -0 and +0 are the same score: both map to the key of +0, so a tie
    // between them is broken by position like any other tie
    uint32_t u = (s == 0.f) ? 0u : __float_as_uint(s);
    uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~asc;
}

struct State {
    uint32_t prefix;       // decided high bits of T (right-aligned)
    int32_t remaining;     // how many more keys to take among those matching prefix
    int32_t c_less;        // keys strictly below the decided prefix range
    int32_t pad;
};

struct Ws {
    int32_t *status;
    int32_t *hist;         // [U][kBins]
    State *state;          // [U]
    int32_t *cnt;          // [U][chunks][2]  (lt, eq)
    int32_t *scan;         // [U][chunks][2]  exclusive
};

__host__ __device__ inline Ws ws_layout(void *ws, int U, int chunks)
{
    uint8_t *p = (uint8_t *)ws;
    Ws w;
    w.status = (int32_t *)p;
    p += kStatusBytes;
    w.hist = (int32_t *)p;
    p += align256((size_t)U * kBins * 4);
    w.state = (State *)p;
    p += align256((size_t)U * sizeof(State));
    w.cnt = (int32_t *)p;
    p += align256((size_t)U * chunks * 2 * 4);
    w.scan = (int32_t *)p;
    return w;
}

constexpr int pass_shift(int p) { return p == 0 ? 21 : (p == 1 ? 10 : 0); }
constexpr int pass_width(int p) { return p == 2 ? 10 : 11; }

__global__ void init_state_kernel(State *st, int U, int kk)
{
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u < U) st[u] = State{0u, kk, 0, 0};
}

template <int PASS>
__global__ void __launch_bounds__(kThreads)
hist_kernel(const float *__restrict__ scores, int L, int cand, Ws W)
{
    constexpr int shift = pass_shift(PASS), width = pass_width(PASS);
    __shared__ int h[kBins];
    for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
    __syncthreads();
    const int u = blockIdx.y;
    const State st = W.state[u];
    const float *s = scores + (size_t)u * L;
    const int lo = blockIdx.x * kChunk, hi = min(cand, lo + kChunk);
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
        const uint32_t key = desc_key(s[i]);
        if constexpr (PASS > 0) {
            if ((key >> (shift + width)) != st.prefix) continue;
        }
        atomicAdd(&h[(key >> shift) & ((1u << width) - 1)], 1);
    }
    __syncthreads();
    int *g = W.hist + (size_t)u * kBins;
    for (int i = threadIdx.x; i < (1 << width); i += kThreads)
        if (h[i]) atomicAdd(&g[i], h[i]);
}

// Pick the digit where the running count reaches `remaining`; clear the histogram.
template <int PASS>
__global__ void __launch_bounds__(kThreads)
choose_kernel(Ws W)
{
    constexpr int width = pass_width(PASS);
    constexpr int nb = 1 << width;
    constexpr int per = nb / kThreads;
    const int u = blockIdx.x;
    int *g = W.hist + (size_t)u * kBins;
    __shared__ int tsum[kThreads];
    int local[per];
    int acc = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        local[i] = g[threadIdx.x * per + i];
        acc += local[i];
    }
    tsum[threadIdx.x] = acc;
    __syncthreads();
    // inclusive scan over the 256 thread sums (Hillis-Steele)
    for (int off = 1; off < kThreads; off <<= 1) {
        const int v = threadIdx.x >= off ? tsum[threadIdx.x - off] : 0;
        __syncthreads();
        tsum[threadIdx.x] += v;
        __syncthreads();
    }
    const State st = W.state[u];
    const int before = threadIdx.x ? tsum[threadIdx.x - 1] : 0;
    if (before < st.remaining && st.remaining <= tsum[threadIdx.x]) {
        int run = before;
#pragma unroll
        for (int i = 0; i < per; ++i) {
            if (run + local[i] >= st.remaining) {
                State ns;
                ns.prefix = (st.prefix << width) | (uint32_t)(threadIdx.x * per + i);
                ns.remaining = st.remaining - run;
                ns.c_less = st.c_less + run;
                ns.pad = 0;
                W.state[u] = ns;
                break;
            }
            run += local[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < per; ++i) g[threadIdx.x * per + i] = 0;
}

__device__ __forceinline__ void classify(float s, uint32_t T, bool &lt, bool &eq)
{
    const uint32_t key = desc_key(s);
    lt = key < T;
    eq = key == T;
}

__global__ void __launch_bounds__(kThreads)
count_kernel(const float *__restrict__ scores, int L, int cand, int chunks, uint32_t T_all, int use_state,
             Ws W)
{
    const int u = blockIdx.y, c = blockIdx.x;
    const uint32_t T = use_state ? W.state[u].prefix : T_all;
    const float *s = scores + (size_t)u * L;
    const int lo = c * kChunk, hi = min(cand, lo + kChunk);
    int nl = 0, ne = 0;
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) {
        bool lt, eq;
        classify(s[i], T, lt, eq);
        nl += lt;
        ne += eq;
    }
    nl = __reduce_add_sync(0xffffffffu, nl);
    ne = __reduce_add_sync(0xffffffffu, ne);
    __shared__ int sl[kThreads / 32], se[kThreads / 32];
    if ((threadIdx.x & 31) == 0) {
        sl[threadIdx.x >> 5] = nl;
        se[threadIdx.x >> 5] = ne;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int a = 0, e = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
            a += sl[w];
            e += se[w];
        }
        W.cnt[((size_t)u * chunks + c) * 2] = a;
        W.cnt[((size_t)u * chunks + c) * 2 + 1] = e;
    }
}

__global__ void scan_chunks_kernel(int n_chunks, int chunks, Ws W)
{
    const int u = blockIdx.x;
    if (threadIdx.x == 0) {
        int a = 0, e = 0;
        for (int c = 0; c < n_chunks; ++c) {
            const size_t o = ((size_t)u * chunks + c) * 2;
            W.scan[o] = a;
            W.scan[o + 1] = e;
            a += W.cnt[o];
            e += W.cnt[o + 1];
        }
    }
}

// Write kept indices of one chunk (candidates by rank, recent window by
// position) and copy their K/V rows.
template <typename T>
__global__ void __launch_bounds__(kThreads)
write_kernel(const float *__restrict__ scores, const T *__restrict__ k, const T *__restrict__ v, int L,
             int d, int cand, int kk, int n_keep, int chunks, uint32_t T_all, int need_all, int use_state,
             Ws W, int32_t *__restrict__ kept, T *__restrict__ ko, T *__restrict__ vo)
{
    const int u = blockIdx.y, c = blockIdx.x;
    const int lo = c * kChunk;
    uint32_t Tk = T_all;
    int need = need_all;
    if (use_state) {
        const State st = W.state[u];
        Tk = st.prefix;
        need = st.remaining;
    }
    const float *s = scores + (size_t)u * L;
    int base_l = 0, base_e = 0;
    if (lo < cand) {
        base_l = W.scan[((size_t)u * chunks + c) * 2];
        base_e = W.scan[((size_t)u * chunks + c) * 2 + 1];
    }
    // per-thread flags over kPer consecutive positions
    const int p0 = lo + threadIdx.x * kPer;
    uint32_t fl = 0, fe = 0;
    int nl = 0, ne = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int p = p0 + i;
        if (p < cand) {
            bool lt, eq;
            classify(s[p], Tk, lt, eq);
            fl |= (uint32_t)lt << i;
            fe |= (uint32_t)eq << i;
            nl += lt;
            ne += eq;
        }
    }
    // block exclusive scan of (nl, ne)
    __shared__ int sl[kThreads], se[kThreads];
    sl[threadIdx.x] = nl;
    se[threadIdx.x] = ne;
    __syncthreads();
    for (int off = 1; off < kThreads; off <<= 1) {
        const int a = threadIdx.x >= off ? sl[threadIdx.x - off] : 0;
        const int e = threadIdx.x >= off ? se[threadIdx.x - off] : 0;
        __syncthreads();
        sl[threadIdx.x] += a;
        se[threadIdx.x] += e;
        __syncthreads();
    }
    int rl = base_l + sl[threadIdx.x] - nl;      // lt before this thread's first position
    int re = base_e + se[threadIdx.x] - ne;
    // slots of this CTA's kept positions, gathered in shared memory for the copy
    __shared__ int srcpos[kChunk], dstslot[kChunk];
    __shared__ int nkept;
    if (threadIdx.x == 0) nkept = 0;
    __syncthreads();
    int32_t *ko_idx = kept + (size_t)u * n_keep;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int p = p0 + i;
        int slot = -1;
        if (p < cand) {
            if ((fl >> i) & 1) {
                slot = rl + min(need, re);
                ++rl;
            } else if ((fe >> i) & 1) {
                if (re < need) slot = rl + re;
                ++re;
            }
        } else if (p < L) {
            slot = kk + (p - cand);
        }
        if (slot >= 0) {
            ko_idx[slot] = p;
            const int q = atomicAdd(&nkept, 1);
            srcpos[q] = p;
            dstslot[q] = slot;
        }
    }
    __syncthreads();
    // row copy: 16-byte vectors, a warp moves whole rows; each thread has
    // kUnroll K and kUnroll V loads in flight before it stores them
    constexpr int kUnroll = 4;
    const int vec_per_row = d * (int)sizeof(T) / 16;
    const int vshift = __ffs(vec_per_row) - 1;
    const bool pow2 = (vec_per_row & (vec_per_row - 1)) == 0;
    const int nvec = nkept * vec_per_row;
    const uint4 *__restrict__ ks = reinterpret_cast<const uint4 *>(k + (size_t)u * L * d);
    const uint4 *__restrict__ vs = reinterpret_cast<const uint4 *>(v + (size_t)u * L * d);
    uint4 *__restrict__ kd = reinterpret_cast<uint4 *>(ko + (size_t)u * n_keep * d);
    uint4 *__restrict__ vd = reinterpret_cast<uint4 *>(vo + (size_t)u * n_keep * d);
    for (int i0 = threadIdx.x; i0 < nvec; i0 += kUnroll * kThreads) {
        uint4 bk[kUnroll], bv[kUnroll];
        size_t dst[kUnroll];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
            const int i = i0 + j * kThreads;
            if (i < nvec) {
                const int r = pow2 ? i >> vshift : i / vec_per_row;
                const int e = i - r * vec_per_row;
                const size_t src = (size_t)srcpos[r] * vec_per_row + e;
                dst[j] = (size_t)dstslot[r] * vec_per_row + e;
                bk[j] = ldg_stream(ks + src);
                bv[j] = ldg_stream(vs + src);
            }
        }
#pragma unroll
        for (int j = 0; j < kUnroll; ++j)
            if (i0 + j * kThreads < nvec) {
                kd[dst[j]] = bk[j];
                vd[dst[j]] = bv[j];
            }
    }
}

template <typename T>
cudaError_t run(const float *scores, const void *k, const void *v, int B, int H, int L, int d,
                int64_t keep_top, int64_t keep_recent, int32_t *kept, void *ko, void *vo, void *ws,
                cudaStream_t st)
{
    const int U = B * H;
    const int R = (int)(keep_recent < L ? keep_recent : L);
    const int cand = L - R;
    const int kk = (int)(keep_top < cand ? keep_top : cand);
    const int n_keep = kk + R;
    const int chunks_all = (L + kChunk - 1) / kChunk;
    const int chunks_c = (cand + kChunk - 1) / kChunk;
    if (U == 0 || n_keep == 0) return cudaSuccess;
    const Ws W = ws_layout(ws, U, chunks_all);
    int use_state = 0;
    uint32_t T_all = 0u;     // kk == 0: nothing below T, no tie kept
    int need_all = 0;
    if (kk == cand) T_all = 0xFFFFFFFFu;  // finite scores never map to this key: keep all
    if (kk > 0 && kk < cand) {
        use_state = 1;
        cudaError_t e = cudaMemsetAsync(W.hist, 0, (size_t)U * kBins * 4, st);
        if (e != cudaSuccess) return e;
        init_state_kernel<<<(U + 127) / 128, 128, 0, st>>>(W.state, U, kk);
        dim3 g(chunks_c, U);
        hist_kernel<0><<<g, kThreads, 0, st>>>(scores, L, cand, W);
        choose_kernel<0><<<U, kThreads, 0, st>>>(W);
        hist_kernel<1><<<g, kThreads, 0, st>>>(scores, L, cand, W);
        choose_kernel<1><<<U, kThreads, 0, st>>>(W);
        hist_kernel<2><<<g, kThreads, 0, st>>>(scores, L, cand, W);
        choose_kernel<2><<<U, kThreads, 0, st>>>(W);
    }
    if (chunks_c > 0) {
        count_kernel<<<dim3(chunks_c, U), kThreads, 0, st>>>(scores, L, cand, chunks_all, T_all, use_state, W);
        scan_chunks_kernel<<<U, 32, 0, st>>>(chunks_c, chunks_all, W);
    }
    write_kernel<T><<<dim3(chunks_all, U), kThreads, 0, st>>>(
        scores, (const T *)k, (const T *)v, L, d, cand, kk, n_keep, chunks_all, T_all, need_all, use_state,
        W, kept, (T *)ko, (T *)vo);
    return cudaGetLastError();
}

}  // namespace

size_t drop_ws_bytes(int B, int H, int L)
{
    const int U = B * H;
    const int chunks = (L + kChunk - 1) / kChunk;
    return kStatusBytes + align256((size_t)U * kBins * 4) + align256((size_t)U * sizeof(State)) +
           2 * align256((size_t)U * chunks * 2 * 4);
}

cudaError_t drop_tokens(const float *scores, const void *k, const void *v, vc_dtype dt, int B, int H, int L,
                        int d, int64_t keep_top, int64_t keep_recent, int32_t *kept_idx, void *k_out,
                        void *v_out, void *ws, cudaStream_t st)
{
    return dt == VC_BF16 ? run<__nv_bfloat16>(scores, k, v, B, H, L, d, keep_top, keep_recent, kept_idx,
                                              k_out, v_out, ws, st)
                         : run<float>(scores, k, v, B, H, L, d, keep_top, keep_recent, kept_idx, k_out,
                                      v_out, ws, st);
}

}  // namespace vc
