// verify_attn.cu -- causal block attention of the drafted block against the
// full KV cache (VeriCache verifies drafts against the full cache; the verify
// step is compute-bound, paper page "What the paper found").
//
// Tensor-core path (bf16, d = 128): one CTA per (kv unit, one or two 128-row
// query tiles, key split).  The 128 rows are the (query, head) pairs of the Hq/Hkv query
// heads sharing one kv head, so the GQA heads and the drafted positions
// together form a real dense M = 128 contraction.
//   warp 0      TMA producer: Q once, then 64-key K and V tiles (128-byte
//               swizzle) into a 2-stage ring;
//   warp 1      single-thread tcgen05.mma issuer: S = Q K^T into a double-
//               buffered TMEM tile (128 x 64 fp32), then O += P V into a TMEM
//               accumulator (128 x 128 fp32), S(j+1) overlapping softmax(j);
//   warps 2..5  softmax, one thread per row (warps 6..9 for a second 128-row
//               tile sharing the K/V tiles): tcgen05.ld of its S row, causal
//               mask, exp2 online softmax with lazy rescaling of O (in TMEM),
//               P written to shared memory as bf16 in the canonical K-major
//               layout for the next MMA.
// Tail mode (a second tile of at most 8 rows, e.g. Dq = 33 with 4 heads per
// kv head): kTailWarps further warps compute the tail rows with mma.sync on
// the same K/V stages, read by ldmatrix, each over its own share of every
// tile's keys (its own online-softmax state; the combine merges the shares);
// each fences those generic-proxy reads (fence.proxy.async) before releasing
// a stage to the TMA refill.
// Every mbarrier wait is bounded; a timeout is recorded in the workspace
// status block and the CTA drains out.  Kernels wait on griddepcontrol.wait
// before their first global access (programmatic dependent launch).  Split partials (m, l, o) go to the
// workspace and a combine kernel writes the normalised output.
//
// CUDA-core path (fp32, or shapes outside the tensor-core kernel): one warp per
// (row, key slice), fp32 throughout.
#include <cudaTypedefs.h>

#include <algorithm>

#include "tcgen05.cuh"
#include "vc_common.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1.0e30f;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ======================================================= tensor-core kernel ==
constexpr int TC_D = 128;
constexpr int TC_M = 128;
constexpr int TC_N = 64;                 // keys per tile
constexpr int TC_PART = 4 + TC_D;        // partial row: m, l, pad, pad, o[128]
constexpr float TC_LAZY = 8.0f;

// Geometry of a CTA holding MT row tiles of 128 (query, head) rows that share
// every K/V tile.  MT = 1: 2 CTAs per SM; MT = 2: one CTA per SM, the whole
// TMEM (per tile: S double buffer 2 x 64 columns + O 128 columns).
constexpr int kTailMaxRows = 8;
constexpr int kTailWarps = 2;            // tail warps; each takes TC_N / kTailWarps keys of a tile

template <int MT, bool TAIL = false>
struct TcGeom {
    static constexpr int STAGES = MT == 1 ? 2 : 3;
    static constexpr int THREADS = 64 + 128 * MT + (TAIL ? 32 * kTailWarps : 0);
    static constexpr int SM_Q = 0;                                    // MT x 2 x (128 x 128 B)
    static constexpr int SM_K = SM_Q + MT * TC_M * TC_D * 2;          // stages x (64 x 256 B)
    static constexpr int SM_V = SM_K + STAGES * TC_N * TC_D * 2;
    static constexpr int SM_P = SM_V + STAGES * TC_N * TC_D * 2;      // MT x (128 x 64 bf16), no swizzle
    static constexpr int SM_BAR = SM_P + MT * TC_M * TC_N * 2;
    static constexpr int SMEM = SM_BAR + 512;
    static constexpr uint32_t TMEM_COLS = 256 * MT;
};

struct TcParams {
    const int32_t *ctx_len;
    const __nv_bfloat16 *q;      // [B][Dq][Hq][128] (tail rows)
    float *part;
    int32_t *status;
    int Hkv, Hq, Dq, grp, n_mtiles, n_cta_m, n_split, tiles_per_split;
    int tail_rows;               // rows of the second row tile done by the tail warp (0: none)
    int kv_once;                 // every K/V tile is read by one CTA: load it evict-first
    float scale_log2;
};

__device__ __forceinline__ void mma_bf16_16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans_b16(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// byte address of 16-byte chunk c (0..15, 8 channels each) of key row `key`
// in a 64-key K or V tile loaded by TMA with 128-byte swizzle as two halves of
// 64 channels (the second half TC_N * 128 bytes on)
__device__ __forceinline__ uint32_t swz_chunk(uint32_t tile, int key, int c)
{
    return tile + (uint32_t)((c >> 3) * (TC_N * 128) + key * 128 + (((c & 7) ^ (key & 7)) << 4));
}

template <int MT, int STAGES>
struct Bars {
    uint64_t q_full;
    uint64_t k_full[STAGES], k_empty[STAGES];
    uint64_t v_full[STAGES], v_empty[STAGES];
    uint64_t s_full[MT][2], s_free[MT][2];
    uint64_t p_ready[MT], pv_done[MT];
    uint32_t tmem_base;
    int32_t abort_flag;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename BarsT>
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, BarsT *B, int32_t *status,
                                              int where)
{
    if (mbar_wait(bar, parity)) return true;
    report_timeout(status, where);
    atomicExch(&B->abort_flag, 1);
    return false;
}

template <int MT, bool TAIL>
__global__ void __launch_bounds__(TcGeom<MT, TAIL>::THREADS, MT == 1 ? 2 : 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, TcParams P)
{
    using Gm = TcGeom<MT, TAIL>;
    using BarsT = Bars<MT, Gm::STAGES>;
    constexpr int STAGES = Gm::STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw;
    // the context lengths and the cache may come from the previous kernel
    pdl_wait();
    if (smem_u32(sm) & 1023u) {
        // the swizzled operand tiles need 1024-byte alignment; never expected
        if (threadIdx.x == 0) report_timeout(P.status, 99);
        return;
    }
    BarsT *B = reinterpret_cast<BarsT *>(sm + Gm::SM_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int split = blockIdx.x;
    const int mtc = blockIdx.y % P.n_cta_m;           // which group of MT row tiles
    const int unit = blockIdx.y / P.n_cta_m;
    const int b = unit / P.Hkv, kvh = unit % P.Hkv;
    const int rows_q = TC_M / P.grp;                  // queries per row tile
    const int q_first = mtc * MT * rows_q;            // first query of the CTA
    const int q_last = TAIL ? P.Dq - 1 : min(P.Dq, q_first + MT * rows_q) - 1;
    const int ctx = P.ctx_len[b];
    const int n_tiles_all = (ctx + q_last + 1 + TC_N - 1) / TC_N;
    const int t_lo = split * P.tiles_per_split;
    const int t_hi = min(n_tiles_all, t_lo + P.tiles_per_split);
    const int n = t_hi > t_lo ? t_hi - t_lo : 0;
    auto part_of = [&](int t) {
        const int mt = mtc * MT + t;
        return P.part + (((size_t)unit * P.n_mtiles + mt) * P.n_split + split) * TC_M * TC_PART;
    };
    // tail mode: the rows of the second tile, all in the first kTailMaxRows;
    // tail warp w keeps its share of the keys in partial rows w * kTailMaxRows + r
    float *part_tail = P.part + (((size_t)unit * P.n_mtiles + 1) * P.n_split + split) * TC_M * TC_PART;

    if (threadIdx.x == 0) {
        mbar_init(&B->q_full, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&B->k_full[s], 1);
            mbar_init(&B->k_empty[s], TAIL ? 1 + kTailWarps : 1);      // the MMAs' commit (+ the tail warps)
            mbar_init(&B->v_full[s], 1);
            mbar_init(&B->v_empty[s], TAIL ? 1 + kTailWarps : 1);
        }
        for (int t = 0; t < MT; ++t) {
            for (int s = 0; s < 2; ++s) {
                mbar_init(&B->s_full[t][s], 1);
                mbar_init(&B->s_free[t][s], 128);
            }
            mbar_init(&B->p_ready[t], 128);
            mbar_init(&B->pv_done[t], 1);
        }
        B->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && n > 0) {
        tc::tmem_alloc(&B->tmem_base, Gm::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    pdl_trigger();      // after the allocation: a started dependent never holds tensor memory first

    if (n == 0) {
        // no key of this split is visible to the CTA's rows: empty partials
        for (int t = 0; t < MT; ++t) {
            float *part = part_of(t);
            for (int i = threadIdx.x; i < TC_M * TC_PART; i += Gm::THREADS) part[i] = (i % TC_PART) == 0 ? kNegBig : 0.f;
        }
        if (TAIL)
            for (int w = 0; w < kTailWarps; ++w)
                for (int i = threadIdx.x; i < P.tail_rows * TC_PART; i += Gm::THREADS)
                    part_tail[w * kTailMaxRows * TC_PART + i] = (i % TC_PART) == 0 ? kNegBig : 0.f;
        return;
    }
    const uint32_t tmem = B->tmem_base;

    // Roles.  Warp 0 lane 0: TMA producer.  Warp 1 lane 0: tcgen05 issuer.
    // Warps 2..5 (and 6..9 for a second tile): softmax.  Tail mode: warps
    // 6 .. 5 + kTailWarps take the tail rows.
    const bool producer = warp == 0 && lane == 0;
    const bool issuer = warp == 1 && lane == 0;
    constexpr int kFirstTailWarp = 2 + 4 * MT;
    if (warp <= 1) {
        if (producer) {
            // -------------------------------------------------- TMA producer --
            tc::prefetch_tmap(&tmQ);
            tc::prefetch_tmap(&tmK);
            tc::prefetch_tmap(&tmV);
            const uint64_t kv_policy = l2_evict_first();
            mbar_arrive_expect_tx(&B->q_full, MT * TC_M * TC_D * 2);
            for (int t = 0; t < MT; ++t) {
                const int qrow = b * P.Dq + q_first + t * rows_q;
                uint8_t *sq = sm + Gm::SM_Q + t * TC_M * TC_D * 2;
                tc::tma_load_3d(sq, &tmQ, 0, kvh * P.grp, qrow, &B->q_full);
                tc::tma_load_3d(sq + TC_M * 128, &tmQ, 64, kvh * P.grp, qrow, &B->q_full);
            }
            for (int j = 0; j < n; ++j) {
                const int s = j % STAGES;
                const uint32_t par = ((j / STAGES) - 1) & 1;
                const int key0 = (t_lo + j) * TC_N;
                if (j >= STAGES && !wait_or_abort(&B->k_empty[s], par, B, P.status, 11)) break;
                uint8_t *sk = sm + Gm::SM_K + s * TC_N * TC_D * 2;
                mbar_arrive_expect_tx(&B->k_full[s], TC_N * TC_D * 2);
                if (P.kv_once) {
                    tc::tma_load_3d_hint(sk, &tmK, 0, key0, unit, &B->k_full[s], kv_policy);
                    tc::tma_load_3d_hint(sk + TC_N * 128, &tmK, 64, key0, unit, &B->k_full[s], kv_policy);
                } else {
                    tc::tma_load_3d(sk, &tmK, 0, key0, unit, &B->k_full[s]);
                    tc::tma_load_3d(sk + TC_N * 128, &tmK, 64, key0, unit, &B->k_full[s]);
                }
                if (j >= STAGES && !wait_or_abort(&B->v_empty[s], par, B, P.status, 12)) break;
                uint8_t *sv = sm + Gm::SM_V + s * TC_N * TC_D * 2;
                mbar_arrive_expect_tx(&B->v_full[s], TC_N * TC_D * 2);
                if (P.kv_once) {
                    tc::tma_load_3d_hint(sv, &tmV, 0, key0, unit, &B->v_full[s], kv_policy);
                    tc::tma_load_3d_hint(sv + TC_N * 128, &tmV, 64, key0, unit, &B->v_full[s], kv_policy);
                } else {
                    tc::tma_load_3d(sv, &tmV, 0, key0, unit, &B->v_full[s]);
                    tc::tma_load_3d(sv + TC_N * 128, &tmV, 64, key0, unit, &B->v_full[s]);
                }
                if (*reinterpret_cast<volatile int32_t *>(&B->abort_flag)) break;
            }
        }
        if (issuer) {
            // --------------------------------------------------- MMA issuer --
            const uint32_t idS = tc::idesc_bf16(TC_M, TC_N, false, false);
            const uint32_t idO = tc::idesc_bf16(TC_M, TC_D, false, true);
            bool ok = wait_or_abort(&B->q_full, 0, B, P.status, 21);
            auto issue_S = [&](int j) -> bool {
                const int s = j % STAGES, sb = j & 1;
                if (!wait_or_abort(&B->k_full[s], (j / STAGES) & 1, B, P.status, 22)) return false;
                const uint32_t sK = smem_u32(sm + Gm::SM_K + s * TC_N * TC_D * 2);
                for (int t = 0; t < MT; ++t) {
                    if (j >= 2 && !wait_or_abort(&B->s_free[t][sb], ((j >> 1) - 1) & 1, B, P.status, 23))
                        return false;
                    tc::fence_after();
                    const uint32_t sQ = smem_u32(sm + Gm::SM_Q + t * TC_M * TC_D * 2);
#pragma unroll
                    for (int kk = 0; kk < TC_D / 16; ++kk) {
                        const uint64_t ad = tc::smem_desc(sQ + (kk >> 2) * (TC_M * 128) + (kk & 3) * 32, 16,
                                                          1024, tc::kSwizzle128B);
                        const uint64_t bd = tc::smem_desc(sK + (kk >> 2) * (TC_N * 128) + (kk & 3) * 32, 16,
                                                          1024, tc::kSwizzle128B);
                        tc::mma_ss(tmem + t * 256 + sb * TC_N, ad, bd, idS, kk > 0);
                    }
                    tc::commit(&B->s_full[t][sb]);
                }
                tc::commit(&B->k_empty[s]);
                return true;
            };
            if (ok) ok = issue_S(0);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n && !issue_S(j + 1)) { ok = false; break; }
                const int s = j % STAGES;
                if (!wait_or_abort(&B->v_full[s], (j / STAGES) & 1, B, P.status, 25)) { ok = false; break; }
                const uint32_t sV = smem_u32(sm + Gm::SM_V + s * TC_N * TC_D * 2);
                for (int t = 0; t < MT; ++t) {
                    if (!wait_or_abort(&B->p_ready[t], j & 1, B, P.status, 24)) { ok = false; break; }
                    tc::fence_after();
                    const uint32_t sP = smem_u32(sm + Gm::SM_P + t * TC_M * TC_N * 2);
#pragma unroll
                    for (int kk = 0; kk < TC_N / 16; ++kk) {
                        // P: K-major, no swizzle; core matrices 8 rows x 16 B,
                        // 128 B apart along K, 1024 B apart along M
                        const uint64_t ad = tc::smem_desc(sP + kk * 256, 128, 1024, tc::kNoSwizzle);
                        // V: MN-major (d contiguous), 128-B swizzle; atoms of 64 d x 8 keys,
                        // next 64 d at +TC_N*128 bytes, next 8 keys at +1024 bytes
                        const uint64_t bd = tc::smem_desc(sV + kk * 2048, TC_N * 128, 1024, tc::kSwizzle128B);
                        tc::mma_ss(tmem + t * 256 + 128, ad, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(&B->pv_done[t]);
                }
                if (!ok) break;
                tc::commit(&B->v_empty[s]);
            }
        }
    } else if (TAIL && warp >= kFirstTailWarp) {
        // ------------------------------------------------ tail rows (mma.sync) --
        // Row r < tail_rows of the second tile (position rows_q + r / grp,
        // head r % grp) against the same K/V tiles.  Transposed products keep
        // the tail rows on the narrow side of m16n8k16 bf16 MMAs: S^T = K Q^T
        // (keys x rows) and O^T += V^T P^T (channels x rows), the K and V
        // operands read from the swizzled tiles by ldmatrix, P^T formed from
        // the S^T fragments by movmatrix.  Lane (gid, tig) holds tail rows
        // 2 tig + e (e = 0, 1).  Tail warp wt takes the 16-key chunks
        // wt * MTS .. wt * MTS + MTS - 1 of every tile.
        constexpr int MTS = TC_N / 16 / kTailWarps;
        const int wt = warp - kFirstTailWarp;
        float *part_w = part_tail + (size_t)wt * kTailMaxRows * TC_PART;
        const int gid = lane >> 2, tig = lane & 3;
        // Q^T fragments (column n = gid: tail row gid)
        uint32_t qb[TC_D / 16][2];
        {
            const bool rv = gid < P.tail_rows;
            const int qpos = rows_q + gid / P.grp;
            const __nv_bfloat16 *qr =
                P.q + (((size_t)b * P.Dq + (rv ? qpos : 0)) * P.Hq + kvh * P.grp + gid % P.grp) * TC_D;
#pragma unroll
            for (int ks = 0; ks < TC_D / 16; ++ks) {
                qb[ks][0] = rv ? *reinterpret_cast<const uint32_t *>(qr + 16 * ks + 2 * tig) : 0u;
                qb[ks][1] = rv ? *reinterpret_cast<const uint32_t *>(qr + 16 * ks + 8 + 2 * tig) : 0u;
            }
        }
        bool rv[2];
        int kmax[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int rr = 2 * tig + e;
            rv[e] = rr < P.tail_rows;
            kmax[e] = ctx + rows_q + rr / P.grp;
        }
        float o[TC_D / 16][4];          // O^T: channels 16 mt + gid (+8) x rows 2 tig + e
#pragma unroll
        for (int i = 0; i < TC_D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m[2] = {kNegBig, kNegBig}, l[2] = {0.f, 0.f};
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int s = j % STAGES;
            if (!__all_sync(0xffffffffu, wait_or_abort(&B->k_full[s], (j / STAGES) & 1, B, P.status, 41))) {
                ok = false;
                break;
            }
            const uint32_t sK = smem_u32(sm + Gm::SM_K + s * TC_N * TC_D * 2);
            float sc[MTS][4];           // S^T: keys 16 (wt MTS + i) + gid (+8) x rows 2 tig + e
#pragma unroll
            for (int i = 0; i < MTS; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < TC_D / 16; ++ks)
#pragma unroll
                for (int i = 0; i < MTS; ++i) {
                    // A = K rows: matrices (keys 16 mt + 8 (mi & 1) .., channel chunk 2 ks + (mi >> 1))
                    const int mt = wt * MTS + i;
                    const int mi = lane >> 3;
                    const int key = 16 * mt + 8 * (mi & 1) + (lane & 7);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(swz_chunk(sK, key, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                    mma_bf16_16816(sc[i], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
            // the stage is refilled by TMA (async proxy) once released: order
            // this warp's generic-proxy reads of it before that
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B->k_empty[s]);
            // causal mask, scale, online softmax per tail row (exp2 domain, lazy rescale)
            const int key0 = (t_lo + j) * TC_N;
            float mx[2] = {kNegBig, kNegBig};
#pragma unroll
            for (int mi2 = 0; mi2 < MTS; ++mi2)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = i & 1;
                    const int key = key0 + 16 * (wt * MTS + mi2) + gid + 8 * (i >> 1);
                    const bool vis = rv[e] && key <= kmax[e];
                    sc[mi2][i] = vis ? sc[mi2][i] * P.scale_log2 : -INFINITY;
                    mx[e] = fmaxf(mx[e], sc[mi2][i]);
                }
            float alpha[2] = {1.f, 1.f};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
                mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
                mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
                if (mx[e] > m[e] + TC_LAZY) {
                    alpha[e] = ex2(m[e] - mx[e]);
                    m[e] = mx[e];
                }
            }
            if (alpha[0] != 1.f || alpha[1] != 1.f) {
                l[0] *= alpha[0];
                l[1] *= alpha[1];
#pragma unroll
                for (int i = 0; i < TC_D / 16; ++i) {
                    o[i][0] *= alpha[0];
                    o[i][1] *= alpha[1];
                    o[i][2] *= alpha[0];
                    o[i][3] *= alpha[1];
                }
            }
            // P^T B fragments: keys 16 kk + 2 tig (+8) of row gid, by transposing
            // the S^T fragment pairs
            uint32_t pb[MTS][2];
#pragma unroll
            for (int mt = 0; mt < MTS; ++mt) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(ex2(sc[mt][0] - m[0]), ex2(sc[mt][1] - m[1]));
                __nv_bfloat162 hi = __floats2bfloat162_rn(ex2(sc[mt][2] - m[0]), ex2(sc[mt][3] - m[1]));
                const float2 fl = __bfloat1622float2(lo), fh = __bfloat1622float2(hi);
                l[0] += fl.x + fh.x;
                l[1] += fl.y + fh.y;
                pb[mt][0] = movmatrix_trans_b16(*reinterpret_cast<uint32_t *>(&lo));
                pb[mt][1] = movmatrix_trans_b16(*reinterpret_cast<uint32_t *>(&hi));
            }
            if (!__all_sync(0xffffffffu, wait_or_abort(&B->v_full[s], (j / STAGES) & 1, B, P.status, 42))) {
                ok = false;
                break;
            }
            const uint32_t sV = smem_u32(sm + Gm::SM_V + s * TC_N * TC_D * 2);
#pragma unroll
            for (int k2 = 0; k2 < MTS; ++k2)
#pragma unroll
                for (int mt = 0; mt < TC_D / 16; ++mt) {
                    // A = V^T: matrices (channels 16 mt + 8 (mi & 1), keys 16 kk + 8 (mi >> 1)),
                    // from key rows, transposed
                    const int kk = wt * MTS + k2;
                    const int mi = lane >> 3;
                    const int key = 16 * kk + 8 * (mi >> 1) + (lane & 7);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(swz_chunk(sV, key, 2 * mt + (mi & 1)), a0, a1, a2, a3);
                    mma_bf16_16816(o[mt], a0, a1, a2, a3, pb[k2][0], pb[k2][1]);
                }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B->v_empty[s]);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
            l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
            l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            if (!rv[e]) continue;
            float *pr = part_w + (size_t)(2 * tig + e) * TC_PART;
            if (gid == 0) {
                pr[0] = ok ? m[e] : kNegBig;
                pr[1] = ok ? l[e] : 0.f;
                pr[2] = 0.f;
                pr[3] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < TC_D / 16; ++mt) {
                pr[4 + 16 * mt + gid] = ok ? o[mt][e] : 0.f;
                pr[4 + 16 * mt + gid + 8] = ok ? o[mt][2 + e] : 0.f;
            }
        }
    } else {
        // --------------------------------------------------- softmax warps --
        const int t = (warp - 2) >> 2;                 // row tile of this warp
        const int wq = warp & 3;                       // TMEM lane quarter
        const int r = wq * 32 + lane;                  // row within the tile
        const int qi = q_first + t * rows_q + r / P.grp;
        const bool row_valid = qi < P.Dq;
        const int kmax = ctx + qi;                     // last visible key
        const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
        const uint32_t tbase = tmem + lane_addr + t * 256;
        float m = kNegBig, l = 0.f;
        uint8_t *sP = sm + Gm::SM_P + t * TC_M * TC_N * 2;
        bool ok = true;
        // a warp whose 32 rows all lie beyond the query block keeps the barrier
        // protocol (same waits and arrivals) but does no softmax work; its P
        // rows and O rows are never read back
        const bool warp_live = __any_sync(0xffffffffu, row_valid);
        for (int j = 0; j < n && !warp_live; ++j) {
            const int sb = j & 1;
            if (!wait_or_abort(&B->s_full[t][sb], (j >> 1) & 1, B, P.status, 34)) { ok = false; break; }
            tc::fence_after();
            tc::fence_before();
            mbar_arrive(&B->s_free[t][sb]);
            if (j > 0 && !wait_or_abort(&B->pv_done[t], (j - 1) & 1, B, P.status, 35)) { ok = false; break; }
            tc::fence_after();
            tc::fence_before();
            mbar_arrive(&B->p_ready[t]);
        }
        for (int j = 0; j < n && warp_live; ++j) {
            const int sb = j & 1;
            if (!wait_or_abort(&B->s_full[t][sb], (j >> 1) & 1, B, P.status, 31)) { ok = false; break; }
            tc::fence_after();
            float s[TC_N];
            {
                uint32_t u[32];
#pragma unroll
                for (int h = 0; h < TC_N / 32; ++h) {
                    tc::ld32(tbase + sb * TC_N + h * 32, u);
                    tc::ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) s[h * 32 + c] = __uint_as_float(u[c]);
                }
            }
            tc::fence_before();
            mbar_arrive(&B->s_free[t][sb]);
            const int key0 = (t_lo + j) * TC_N;
            float mx = kNegBig;
#pragma unroll
            for (int c = 0; c < TC_N; ++c) {
                const bool vis = row_valid && (key0 + c <= kmax);
                s[c] = vis ? s[c] * P.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[c]);
            }
            float alpha = 1.f;
            if (mx > m + TC_LAZY) {
                alpha = ex2(m - mx);
                m = mx;
            }
            float lsum = 0.f;
            uint32_t pk[TC_N / 2];
#pragma unroll
            for (int c = 0; c < TC_N; c += 2) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2(s[c] - m), ex2(s[c + 1] - m));
                const float2 f2 = __bfloat1622float2(h2);
                lsum += f2.x + f2.y;
                pk[c / 2] = *reinterpret_cast<uint32_t *>(&h2);
            }
            l = l * alpha + lsum;
            // the P buffer of this tile and its O are free once PV(j-1) has completed
            if (j > 0 && !wait_or_abort(&B->pv_done[t], (j - 1) & 1, B, P.status, 32)) { ok = false; break; }
            tc::fence_after();
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int h = 0; h < TC_D / 32; ++h) {
                    uint32_t u[32];
                    tc::ld32(tbase + 128 + h * 32, u);
                    tc::ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) u[c] = __float_as_uint(__uint_as_float(u[c]) * alpha);
                    tc::st32(tbase + 128 + h * 32, u);
                }
                tc::st_wait();
            }
            // P row r: 8 chunks of 8 keys, core matrix (r/8, kb) at ((r/8)*8 + kb)*128 + (r%8)*16
#pragma unroll
            for (int kb = 0; kb < TC_N / 8; ++kb) {
                uint4 v;
                v.x = pk[kb * 4 + 0];
                v.y = pk[kb * 4 + 1];
                v.z = pk[kb * 4 + 2];
                v.w = pk[kb * 4 + 3];
                *reinterpret_cast<uint4 *>(sP + ((r >> 3) * 8 + kb) * 128 + (r & 7) * 16) = v;
            }
            fence_async_smem();                  // P (generic writes) before the MMA reads it
            tc::fence_before();
            mbar_arrive(&B->p_ready[t]);
        }
        // epilogue: wait for the last PV, read O, store the partial row
        float *pr = part_of(t) + (size_t)r * TC_PART;
        if (ok && warp_live && wait_or_abort(&B->pv_done[t], (n - 1) & 1, B, P.status, 33)) {
            tc::fence_after();
            pr[0] = m;
            pr[1] = l;
            pr[2] = 0.f;
            pr[3] = 0.f;
#pragma unroll
            for (int h = 0; h < TC_D / 32; ++h) {
                uint32_t u[32];
                tc::ld32(tbase + 128 + h * 32, u);
                tc::ld_wait();
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4 *>(pr + 4 + h * 32 + c) =
                        make_float4(__uint_as_float(u[c]), __uint_as_float(u[c + 1]),
                                    __uint_as_float(u[c + 2]), __uint_as_float(u[c + 3]));
            }
        } else {
            pr[0] = kNegBig;
            pr[1] = 0.f;
            for (int c = 2; c < TC_PART; ++c) pr[c] = 0.f;
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tmem, Gm::TMEM_COLS);
    }
}

// Merge the key splits of the tensor-core kernel.  One thread per (row, 4 channels).
// In tail mode (tail_sub > 1) the last row tile's rows r come in tail_sub
// shares of the keys, at partial rows w * kTailMaxRows + r, merged as splits.
template <typename T>
__global__ void verify_tc_combine(const float *__restrict__ part, int n_split, int n_mtiles, int Hkv,
                                  int Hq, int Dq, int grp, int tail_sub, T *__restrict__ out,
                                  float2 *__restrict__ ml)
{
    pdl_wait();
    pdl_trigger();
    const int item = blockIdx.x;                       // unit * n_mtiles + mt
    const int mt = item % n_mtiles, unit = item / n_mtiles;
    const int b = unit / Hkv, kvh = unit % Hkv;
    const int r = blockIdx.y * 4 + (threadIdx.x >> 5);
    const int c0 = (threadIdx.x & 31) * 4;
    const int qi = mt * (TC_M / grp) + r / grp;
    if (qi >= Dq) return;
    const float *pp = part + (size_t)item * n_split * TC_M * TC_PART + (size_t)r * TC_PART;
    const size_t sstride = (size_t)TC_M * TC_PART;
    const int n_sub = mt == n_mtiles - 1 ? tail_sub : 1;
    const size_t wstride = (size_t)kTailMaxRows * TC_PART;
    float M = kNegBig;
    for (int s = 0; s < n_split; ++s)
        for (int w = 0; w < n_sub; ++w) M = fmaxf(M, pp[s * sstride + w * wstride]);
    float L = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < n_split; ++s)
        for (int w = 0; w < n_sub; ++w) {
            const float *q = pp + s * sstride + w * wstride;
            const float wt = exp2f(q[0] - M);
            L += q[1] * wt;
            const float4 v = *reinterpret_cast<const float4 *>(q + 4 + c0);
            o[0] += v.x * wt;
            o[1] += v.y * wt;
            o[2] += v.z * wt;
            o[3] += v.w * wt;
        }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (ml && c0 == 0) ml[((size_t)b * Dq + qi) * Hq + kvh * grp + r % grp] = make_float2(M, L);
    T *dst = out + (((size_t)b * Dq + qi) * Hq + kvh * grp + r % grp) * TC_D + c0;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = Elem<T>::from_f(o[i] * inv);
}

// ======================================================== CUDA-core kernel ===
constexpr int SIMT_WARPS = 4;

// grid (B*Dq*Hq); warp w of the CTA takes keys k = w, w+4, ...; merged in smem.
template <typename T, int D>
__global__ void __launch_bounds__(SIMT_WARPS * 32)
verify_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   const int32_t *__restrict__ ctx_len, int Dq, int Hq, int Hkv, int L_stride,
                   float scale_log2, T *__restrict__ out)
{
    constexpr int CPL = D / 32;
    const int row = blockIdx.x;                    // (b * Dq + i) * Hq + hq
    const int hq = row % Hq, bi = row / Hq;
    const int b = bi / Dq, i = bi % Dq;
    const int grp = Hq / Hkv;
    const int kvh = hq / grp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkeys = ctx_len[b] + i + 1;
    const T *kb = k + ((size_t)b * Hkv + kvh) * L_stride * D;
    const T *vb = v + ((size_t)b * Hkv + kvh) * L_stride * D;
    float qv[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) qv[c] = Elem<T>::to_f(q[(size_t)row * D + lane * CPL + c]) * scale_log2;
    float m = kNegBig, l = 0.f, o[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[c] = 0.f;
    for (int t = warp; t < nkeys; t += SIMT_WARPS) {
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) s = fmaf(qv[c], Elem<T>::to_f(kb[(size_t)t * D + lane * CPL + c]), s);
        s = warp_sum(s);
        const float mn = fmaxf(m, s);
        const float a = exp2f(m - mn), p = exp2f(s - mn);
        m = mn;
        l = l * a + p;
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[c] = o[c] * a + p * Elem<T>::to_f(vb[(size_t)t * D + lane * CPL + c]);
    }
    __shared__ float wm[SIMT_WARPS], wl[SIMT_WARPS], wo[SIMT_WARPS][D];
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) wo[warp][lane * CPL + c] = o[c];
    __syncthreads();
    if (warp == 0) {
        float M = kNegBig;
        for (int w = 0; w < SIMT_WARPS; ++w) M = fmaxf(M, wm[w]);
        float L = 0.f;
        for (int w = 0; w < SIMT_WARPS; ++w) L += wl[w] * exp2f(wm[w] - M);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            float acc = 0.f;
            for (int w = 0; w < SIMT_WARPS; ++w) acc += wo[w][lane * CPL + c] * exp2f(wm[w] - M);
            out[(size_t)row * D + lane * CPL + c] = Elem<T>::from_f(L > 0.f ? acc / L : 0.f);
        }
    }
}

// ================================================================== host ===
struct TcPlan {
    int n_mtiles, mt_per_cta, n_cta_m, n_split, tiles_per_split, tail_rows;
};

// split_tiles > 0 fixes the number of 64-key tiles per split, so that the
// split boundaries of a row depend on nothing but key positions.
TcPlan tc_plan(int B, int Dq, int Hkv, int grp, int max_ctx, int split_tiles)
{
    TcPlan p;
    p.n_mtiles = (Dq * grp + TC_M - 1) / TC_M;
    // One row tile per CTA: a CTA holding two tiles that share every K/V tile
    // (TcGeom<2>) halves the K/V reads at Dq*grp in (128, 256] but runs one
    // CTA per SM, and its softmax/MMA handoff chain then limits it to about
    // 1.0 ms against 0.77 ms for two single-tile CTAs per SM at Dq = 33.
    p.mt_per_cta = 1;
    p.n_cta_m = p.n_mtiles / p.mt_per_cta;
    // A second tile of at most kTailMaxRows rows (Dq = 33 with 4 query heads
    // per kv head: 4 rows) is done inside the first tile's CTA by a tail warp
    // on the same K/V tiles, instead of by CTAs that repeat the whole tile's
    // work.  Not under a fixed split size: callers that need every row's
    // arithmetic independent of Dq keep all rows on the tcgen05 path.
    p.tail_rows = 0;
    if (split_tiles <= 0 && p.n_mtiles == 2 && Dq * grp - TC_M <= kTailMaxRows) {
        p.tail_rows = Dq * grp - TC_M;
        p.n_cta_m = 1;
    }
    const int tiles = (max_ctx + Dq + TC_N - 1) / TC_N;
    const int items = B * Hkv * p.n_cta_m;
    const int slots = device_sm_count() * (p.mt_per_cta == 1 ? 2 : 1);
    // Split count that minimises waves x (key tiles per CTA + ~4 tiles of
    // fixed cost: setup, partial store) for resident CTAs of equal length.
    int best = 1;
    long best_t = -1;
    for (int s = 1; s <= 32 && s <= tiles; ++s) {
        const int per = (tiles + s - 1) / s;
        const int se = (tiles + per - 1) / per;
        const long waves = ((long)items * se + slots - 1) / slots;
        const long t = waves * (per + 4);
        if (best_t < 0 || t < best_t) {
            best_t = t;
            best = se;
        }
    }
    p.tiles_per_split = (tiles + best - 1) / best;
    if (p.tiles_per_split < 2 && tiles >= 2) p.tiles_per_split = 2;
    if (split_tiles > 0) p.tiles_per_split = split_tiles;
    p.n_split = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    return p;
}

// ===================================================== H2O mass of a verify ==
// The attention mass each key receives from the verify block (H2O ranks
// tokens by accumulated attention, source 3 on the podparley page): for kv
// unit u and key j < ctx_len[b] + Dq, the sum over the block's rows (query i,
// head of the unit's group) that see j (j <= ctx + i) of
// exp2(q.k * scale_log2 - M_row) / L_row, with M_row and L_row the row's final
// max and sum from the verify pass.  The scores are recomputed on the tensor
// cores with the keys on the MMA's M side and the rows on its N side, so a
// warp finishes the mass of its 16 keys on its own: the CTA stages the unit's
// Q rows (and each row's max and 1/sum) once, then every warp streams its own
// 16-key K tiles through a two-stage ring (one bulk copy per key row, padded
// rows for conflict-free ldmatrix), sums the weights over all rows, and adds
// each key's mass to scores[u * scores_stride + j] (each key by one warp).
constexpr int H2O_KT = 16;                      // keys per warp tile
constexpr int H2O_PITCH = TC_D * 2 + 16;        // bytes per staged row
constexpr int H2O_MAXROWS = 272;                // Dq * grp
constexpr int H2O_WARPS = 8;

struct H2oParams {
    const __nv_bfloat16 *q, *k;
    const int32_t *ctx_len;
    const float2 *ml;
    float *scores;
    int32_t *status;
    int Dq, Hq, Hkv, grp, L_stride, keys_per_split, scores_stride, rows_pad;
    float scale_log2;
};

__global__ void __launch_bounds__(H2O_WARPS * 32)
verify_h2o_mass_kernel(H2oParams P)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(128) uint8_t hsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    uint64_t *bars = reinterpret_cast<uint64_t *>(hsm);                               // [warps][2]
    float4 *mlv = reinterpret_cast<float4 *>(hsm + 256);                              // [rows_pad / 2]: (M, 1/L) x 2
    uint8_t *qs = hsm + 256 + P.rows_pad * 8;                                        // [rows_pad][PITCH]
    uint8_t *ring = qs + P.rows_pad * H2O_PITCH + warp * 2 * H2O_KT * H2O_PITCH;     // this warp's [2][16][PITCH]
    const int unit = blockIdx.y, b = unit / P.Hkv, kvh = unit % P.Hkv;
    const int rows = P.Dq * P.grp;
    const int ctx = P.ctx_len[b];
    const int n_keys = ctx + P.Dq;
    const int k_lo = blockIdx.x * P.keys_per_split;
    const int k_hi = min(n_keys, k_lo + P.keys_per_split);
    if (k_lo >= k_hi) return;
    // the unit's rows: Q (bf16, zero beyond `rows`) and (M, 1/L)
    for (int i = threadIdx.x; i < P.rows_pad * (TC_D / 8); i += blockDim.x) {
        const int r = i / (TC_D / 8), ch = i % (TC_D / 8);
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < rows) {
            const size_t row = ((size_t)b * P.Dq + r / P.grp) * P.Hq + kvh * P.grp + r % P.grp;
            u = *reinterpret_cast<const uint4 *>(P.q + row * TC_D + ch * 8);
        }
        *reinterpret_cast<uint4 *>(qs + r * H2O_PITCH + ch * 16) = u;
    }
    for (int i = threadIdx.x; i < P.rows_pad / 2; i += blockDim.x) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * i + e;
            if (r < rows) {
                const float2 m = P.ml[((size_t)b * P.Dq + r / P.grp) * P.Hq + kvh * P.grp + r % P.grp];
                v[2 * e] = m.x;
                v[2 * e + 1] = m.y > 0.f ? 1.f / m.y : 0.f;
            }
        }
        mlv[i] = make_float4(v[0], v[1], v[2], v[3]);
    }
    uint64_t *bar = bars + 2 * warp;
    if (lane == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const __nv_bfloat16 *kb = P.k + (size_t)unit * P.L_stride * TC_D;
    const int nwarps = blockDim.x >> 5;
    // key tiles of this warp: k_lo + 16 (warp + i * nwarps)
    auto issue = [&](int key0, int s) {
        const int nk = min(H2O_KT, k_hi - key0);
        if (lane == 0) mbar_arrive_expect_tx(&bar[s], (uint32_t)nk * TC_D * 2);
        __syncwarp();
        if (lane < nk) bulk_g2s(ring + (s * H2O_KT + lane) * H2O_PITCH, kb + (size_t)(key0 + lane) * TC_D, TC_D * 2,
                                &bar[s]);
    };
    const int step = H2O_KT * nwarps;
    int key0 = k_lo + H2O_KT * warp;
    if (key0 < k_hi) issue(key0, 0);
    if (key0 + step < k_hi) issue(key0 + step, 1);
    const uint32_t qs_u = smem_u32(qs);
    const int n_nt = P.rows_pad / 8;
    for (int it = 0; key0 < k_hi; key0 += step, ++it) {
        const int s = it & 1;
        if (!mbar_wait(&bar[s], (it >> 1) & 1)) {
            report_timeout(P.status, 51);
            if (key0 + step < k_hi) mbar_wait(&bar[s ^ 1], ((it + 1) >> 1) & 1);
            return;
        }
        const uint32_t st = smem_u32(ring + s * H2O_KT * H2O_PITCH);
        // A = K rows of the tile: keys (lane & 7) + 8 ((lane >> 3) & 1), chunk 2 ks + (lane >> 4)
        uint32_t ka[TC_D / 16][4];
#pragma unroll
        for (int ks = 0; ks < TC_D / 16; ++ks)
            ldsm_x4(st + ((lane & 7) + 8 * ((lane >> 3) & 1)) * H2O_PITCH + (2 * ks + (lane >> 4)) * 16, ka[ks][0],
                    ka[ks][1], ka[ks][2], ka[ks][3]);
        // the stage has been read (generic proxy): release it to the refill
        fence_async_smem();
        __syncwarp();
        if (key0 + 2 * step < k_hi) issue(key0 + 2 * step, s);
        const int klo = key0 + gid, khi = key0 + gid + 8;    // this lane's two keys
        const bool all_visible = key0 + H2O_KT - 1 < ctx;     // every row sees every key of the tile
        float mlo = 0.f, mhi = 0.f;
#pragma unroll 2
        for (int nt = 0; nt < n_nt; ++nt) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kp = 0; kp < TC_D / 32; ++kp) {
                // B = Q^T: rows 8 nt + (lane & 7), chunks 4 kp + (lane >> 3)
                uint32_t b0, b1, b2, b3;
                ldsm_x4(qs_u + (8 * nt + (lane & 7)) * H2O_PITCH + (4 * kp + (lane >> 3)) * 16, b0, b1, b2, b3);
                mma_bf16_16816(c, ka[2 * kp][0], ka[2 * kp][1], ka[2 * kp][2], ka[2 * kp][3], b0, b1);
                mma_bf16_16816(c, ka[2 * kp + 1][0], ka[2 * kp + 1][1], ka[2 * kp + 1][2], ka[2 * kp + 1][3], b2, b3);
            }
            // rows 8 nt + 2 tig + e: (M, 1/L)
            const float4 ml = mlv[4 * nt + tig];
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = i & 1;
                p[i] = ex2(c[i] * P.scale_log2 - (e ? ml.z : ml.x)) * (e ? ml.w : ml.y);
            }
            if (!all_visible) {
                // keys of the block itself: row r (query r / grp) sees keys <= ctx + r / grp
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 8 * nt + 2 * tig + (i & 1);
                    const int key = (i >> 1) ? khi : klo;
                    if (key > ctx + r / P.grp) p[i] = 0.f;
                }
            }
            mlo += p[0] + p[1];
            mhi += p[2] + p[3];
        }
        mlo += __shfl_xor_sync(0xffffffffu, mlo, 1);
        mlo += __shfl_xor_sync(0xffffffffu, mlo, 2);
        mhi += __shfl_xor_sync(0xffffffffu, mhi, 1);
        mhi += __shfl_xor_sync(0xffffffffu, mhi, 2);
        if (tig == 0) {
            float *dst = P.scores + (size_t)unit * P.scores_stride;
            if (klo < k_hi) atomicAdd(dst + klo, mlo);
            if (khi < k_hi) atomicAdd(dst + khi, mhi);
        }
    }
}

}  // namespace

bool verify_uses_tensor_cores(vc_dtype dt, int Dq, int Hq, int Hkv, int d)
{
    const int grp = Hq / Hkv;
    return dt == VC_BF16 && d == TC_D && (grp == 1 || grp == 2 || grp == 4 || grp == 8) && Dq >= 1;
}

size_t verify_ws_bytes(vc_dtype dt, int B, int Dq, int Hq, int Hkv, int d, int max_ctx, int split_tiles)
{
    if (!verify_uses_tensor_cores(dt, Dq, Hq, Hkv, d)) return kStatusBytes;
    const TcPlan p = tc_plan(B, Dq, Hkv, Hq / Hkv, max_ctx, split_tiles);
    return kStatusBytes + align256((size_t)B * Hkv * p.n_mtiles * p.n_split * TC_M * TC_PART * 4);
}

cudaError_t verify_attn(const void *q, const void *k, const void *v, vc_dtype dt, const int32_t *ctx_len,
                        int B, int Dq, int Hq, int Hkv, int d, int L_stride, int max_ctx, float sm_scale,
                        void *out, void *ws, cudaStream_t st, int split_tiles, float2 *ml)
{
    const float sl2 = sm_scale * kLog2e;
    if (verify_uses_tensor_cores(dt, Dq, Hq, Hkv, d)) {
        const int grp = Hq / Hkv;
        const TcPlan pl = tc_plan(B, Dq, Hkv, grp, max_ctx, split_tiles);
        CUtensorMap mq, mk, mv;
        if (!tma_map_bf16_3d(&mq, q, TC_D, Hq, (uint64_t)B * Dq, (uint64_t)TC_D * 2, (uint64_t)Hq * TC_D * 2, 64,
                         grp, TC_M / grp) ||
            !tma_map_bf16_3d(&mk, k, TC_D, L_stride, (uint64_t)B * Hkv, (uint64_t)TC_D * 2,
                         (uint64_t)L_stride * TC_D * 2, 64, TC_N, 1) ||
            !tma_map_bf16_3d(&mv, v, TC_D, L_stride, (uint64_t)B * Hkv, (uint64_t)TC_D * 2,
                         (uint64_t)L_stride * TC_D * 2, 64, TC_N, 1))
            return cudaErrorInvalidValue;
        TcParams P;
        P.ctx_len = ctx_len;
        P.q = (const __nv_bfloat16 *)q;
        P.Hq = Hq;
        P.tail_rows = pl.tail_rows;
        P.status = (int32_t *)ws;
        P.part = (float *)((uint8_t *)ws + kStatusBytes);
        P.Hkv = Hkv;
        P.Dq = Dq;
        P.grp = grp;
        P.n_mtiles = pl.n_mtiles;
        P.n_cta_m = pl.n_cta_m;
        // with two row-tile CTAs per unit each K/V tile is read twice, close in
        // time: the second read may find it in L2
        P.kv_once = pl.n_cta_m == 1 ? 1 : 0;
        P.n_split = pl.n_split;
        P.tiles_per_split = pl.tiles_per_split;
        P.scale_log2 = sl2;
        dim3 grid(pl.n_split, B * Hkv * pl.n_cta_m);
        cudaError_t e;
        if (pl.mt_per_cta == 2) {
            auto kern = verify_tc_kernel<2, false>;
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcGeom<2>::SMEM);
            e = launch_pdl(kern, grid, dim3(TcGeom<2>::THREADS), TcGeom<2>::SMEM, st, mq, mk, mv, P);
        } else if (pl.tail_rows > 0) {
            auto kern = verify_tc_kernel<1, true>;
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcGeom<1, true>::SMEM);
            e = launch_pdl(kern, grid, dim3(TcGeom<1, true>::THREADS), TcGeom<1, true>::SMEM, st, mq, mk, mv, P);
        } else {
            auto kern = verify_tc_kernel<1, false>;
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcGeom<1>::SMEM);
            e = launch_pdl(kern, grid, dim3(TcGeom<1>::THREADS), TcGeom<1>::SMEM, st, mq, mk, mv, P);
        }
        if (e != cudaSuccess) return e;
        dim3 cgrid(B * Hkv * pl.n_mtiles, TC_M / 4);
        return launch_pdl(verify_tc_combine<__nv_bfloat16>, cgrid, dim3(128), 0, st, (const float *)P.part,
                          pl.n_split, pl.n_mtiles, Hkv, Hq, Dq, grp, pl.tail_rows > 0 ? kTailWarps : 1,
                          (__nv_bfloat16 *)out, ml);
    }
    const int rows = B * Dq * Hq;
    if (rows == 0) return cudaSuccess;
    if (dt == VC_BF16) {
        if (d == 128)
            verify_simt_kernel<__nv_bfloat16, 128><<<rows, SIMT_WARPS * 32, 0, st>>>(
                (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, ctx_len, Dq, Hq,
                Hkv, L_stride, sl2, (__nv_bfloat16 *)out);
        else
            verify_simt_kernel<__nv_bfloat16, 64><<<rows, SIMT_WARPS * 32, 0, st>>>(
                (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, ctx_len, Dq, Hq,
                Hkv, L_stride, sl2, (__nv_bfloat16 *)out);
    } else {
        if (d == 128)
            verify_simt_kernel<float, 128><<<rows, SIMT_WARPS * 32, 0, st>>>(
                (const float *)q, (const float *)k, (const float *)v, ctx_len, Dq, Hq, Hkv, L_stride, sl2,
                (float *)out);
        else
            verify_simt_kernel<float, 64><<<rows, SIMT_WARPS * 32, 0, st>>>(
                (const float *)q, (const float *)k, (const float *)v, ctx_len, Dq, Hq, Hkv, L_stride, sl2,
                (float *)out);
    }
    return cudaGetLastError();
}

size_t verify_h2o_ws_bytes(int B, int Dq, int Hq, int Hkv, int max_ctx)
{
    return verify_ws_bytes(VC_BF16, B, Dq, Hq, Hkv, TC_D, max_ctx) + align256((size_t)B * Dq * Hq * 8);
}

bool verify_h2o_supported(vc_dtype dt, int Dq, int Hq, int Hkv, int d)
{
    return verify_uses_tensor_cores(dt, Dq, Hq, Hkv, d) && Dq * (Hq / Hkv) <= H2O_MAXROWS;
}

cudaError_t verify_attn_h2o(const void *q, const void *k, const void *v, const int32_t *ctx_len, int B, int Dq,
                            int Hq, int Hkv, int L_stride, int max_ctx, float sm_scale, void *out, float *scores,
                            int scores_stride, void *ws, cudaStream_t st)
{
    const size_t main_ws = verify_ws_bytes(VC_BF16, B, Dq, Hq, Hkv, TC_D, max_ctx);
    float2 *ml = (float2 *)((uint8_t *)ws + main_ws);
    cudaError_t e = verify_attn(q, k, v, VC_BF16, ctx_len, B, Dq, Hq, Hkv, TC_D, L_stride, max_ctx, sm_scale, out,
                                ws, st, 0, ml);
    if (e != cudaSuccess) return e;
    H2oParams P;
    P.q = (const __nv_bfloat16 *)q;
    P.k = (const __nv_bfloat16 *)k;
    P.ctx_len = ctx_len;
    P.ml = ml;
    P.scores = scores;
    P.status = (int32_t *)ws;
    P.Dq = Dq;
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.grp = Hq / Hkv;
    P.L_stride = L_stride;
    P.scores_stride = scores_stride;
    P.scale_log2 = sm_scale * kLog2e;
    const int units = B * Hkv;
    const int rows = Dq * P.grp;
    P.rows_pad = (rows + 7) / 8 * 8;
    const int n_keys = max_ctx + Dq;
    // about two CTAs per SM over the units; splits of whole 16-key tiles per warp pass
    const int want = std::max(1, (2 * device_sm_count() + units - 1) / units);
    const int per = (n_keys + want - 1) / want;
    P.keys_per_split = (per + H2O_KT * H2O_WARPS - 1) / (H2O_KT * H2O_WARPS) * (H2O_KT * H2O_WARPS);
    const int smem = 256 + P.rows_pad * 8 + P.rows_pad * H2O_PITCH + H2O_WARPS * 2 * H2O_KT * H2O_PITCH;
    cudaFuncSetAttribute(verify_h2o_mass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    dim3 grid((n_keys + P.keys_per_split - 1) / P.keys_per_split, units);
    return launch_pdl(verify_h2o_mass_kernel, grid, dim3(32 * H2O_WARPS), smem, st, P);
}

}  // namespace vc
