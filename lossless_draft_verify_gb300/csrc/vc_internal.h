// vc_internal.h -- launchers shared between the kernel files and the C-ABI
// entry points (vc_api.cu).  Arguments are validated by the caller.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/vc.h"

namespace vc {

// quantize.cu
cudaError_t quantize_prefill(const void *k, const void *v, vc_dtype dt, int B, int Hkv, int L,
                             int L_stride, int d, const vc_qcache *c, cudaStream_t st);
cudaError_t qcache_append(const vc_qcache *c, const void *k_new, const void *v_new,
                          const int32_t *n_new, const int32_t *len_base, const int32_t *n_acc,
                          int max_new, int requantize, cudaStream_t st);

// accept.cu
size_t accept_ws_bytes(int B, int D, int V);
cudaError_t accept_tiles(const float *tile_max, const int32_t *tile_idx, int n_tiles, const int32_t *drafts,
                         int B, int D, int32_t *n_acc, int32_t *next_tok, cudaStream_t st);
// The per-sequence counters in ws are left at zero by every call; with
// clear_counters they are also zeroed on the stream first.
cudaError_t accept(const void *logits, vc_dtype dt, const int32_t *drafts, int B, int D, int V,
                   int32_t *n_acc, int32_t *next_tok, void *ws, cudaStream_t st, bool clear_counters = false);

// draft_attn.cu
size_t draft_ws_bytes(const vc_cache_view *view, int Hq);
cudaError_t draft_attn(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq,
                       float sm_scale, void *out, void *ws, cudaStream_t st);

// draft_attn.cu, H2O variant (dense bf16 and KIVI views): also adds each
// token's attention mass, summed over the query heads of its kv head, to scores.
size_t draft_h2o_ws_bytes(const vc_cache_view *view, int Hq);
cudaError_t draft_attn_h2o(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq, float sm_scale,
                           void *out, float *scores, int scores_stride, const int32_t *kept_idx, int kept_stride,
                           void *ws, cudaStream_t st);

// verify_attn.cu
// split_tiles > 0: fixed key splits of split_tiles x 64 keys (row results then
// do not depend on B or Dq); 0: splits chosen to fill the GPU.
size_t verify_ws_bytes(vc_dtype dt, int B, int Dq, int Hq, int Hkv, int d, int max_ctx, int split_tiles = 0);
bool verify_uses_tensor_cores(vc_dtype dt, int Dq, int Hq, int Hkv, int d);
cudaError_t verify_attn(const void *q, const void *k, const void *v, vc_dtype dt,
                        const int32_t *ctx_len, int B, int Dq, int Hq, int Hkv, int d,
                        int L_stride, int max_ctx, float sm_scale, void *out, void *ws,
                        cudaStream_t st, int split_tiles = 0, float2 *ml = nullptr);
// H2O variant (tensor-core shapes, Dq * Hq / Hkv <= 272 rows): the verify
// pass, then each key's attention mass summed over the block's rows added to
// scores (a second pass over K with the rows' final max and sum).
size_t verify_h2o_ws_bytes(int B, int Dq, int Hq, int Hkv, int max_ctx);
bool verify_h2o_supported(vc_dtype dt, int Dq, int Hq, int Hkv, int d);
cudaError_t verify_attn_h2o(const void *q, const void *k, const void *v, const int32_t *ctx_len, int B, int Dq,
                            int Hq, int Hkv, int L_stride, int max_ctx, float sm_scale, void *out, float *scores,
                            int scores_stride, void *ws, cudaStream_t st);

// drop.cu
size_t drop_ws_bytes(int B, int H, int L);
cudaError_t drop_tokens(const float *scores, const void *k, const void *v, vc_dtype dt, int B,
                        int H, int L, int d, int64_t keep_top, int64_t keep_recent,
                        int32_t *kept_idx, void *k_out, void *v_out, void *ws, cudaStream_t st);

// gemm.cu: y = x W (+ resid), x [M][ldx] (first K columns), W [K][N].  The
// summation order of an output element depends on (N, K, plan) and the
// device, never on M.  ws: gemm_ws_bytes bytes of fp32 partials (bf16 path);
// counters: kGemmMaxTiles words that are zero on entry and left zero (the last
// CTA of each output tile sums the partials), or null (a separate reduction).
constexpr int kGemmRowInvariant = 0;   // forward passes (verify, plain decoding, prefill)
constexpr int kGemmDecode = 1;         // draft steps (M <= 128)
// Flag OR-ed into the plan of gemm(): the weights cannot be written by work
// still pending on the stream (the decoder's own weights), so the kernel may
// request its first weight slices before the previous kernel completes.
constexpr int kGemmEarlyWeights = 1 << 4;
constexpr int kGemmMaxTiles = 16384;
constexpr size_t kGemmCounterBytes = (size_t)kGemmMaxTiles * 4;
bool gemm_uses_tensor_cores(vc_dtype dt, int N, int K);
int gemm_splits(int N, int K, int plan);
size_t gemm_ws_bytes(vc_dtype dt, int M, int N, int K, int plan = kGemmRowInvariant);
// rms_eps >= 0: x is the raw residual stream and every output row is scaled by
// 1 / sqrt(mean(x_row^2) + rms_eps), i.e. the product of rmsnorm(x) (draft-step
// products only: gemm_rms_ok; no residual)
cudaError_t gemm(const void *x, const void *w, const void *resid, void *out, vc_dtype dt, int M, int N, int K,
                 int ldx, void *ws, unsigned int *counters, int32_t *status, cudaStream_t st,
                 int plan = kGemmRowInvariant, float *amax_val = nullptr, int32_t *amax_idx = nullptr,
                 float rms_eps = -1.f);
bool gemm_rms_ok(vc_dtype dt, int M, int N, int K, int ldx, int plan);
// whether the argmax epilogue is available for this shape and plan (tensor-core
// path, and one K split or per-tile counters)
bool gemm_argmax_ok(vc_dtype dt, int M, int N, int K, int plan, bool have_counters);
// act [M][F] = silu(g) * u for the product x W with W [K][2F] whose columns hold
// gate and up interleaved per 64 (columns 128 t + j: gate 64 t + j, 128 t + 64 + j:
// up 64 t + j), g and u rounded to bf16 first: the SwiGLU epilogue of the
// tensor-core GEMM, for bf16 products the plan leaves unsplit
bool gemm_swiglu_ok(vc_dtype dt, int F, int K, int plan);
cudaError_t gemm_swiglu(const void *x, const void *w, void *act, vc_dtype dt, int M, int F, int K, int ldx,
                        int32_t *status, cudaStream_t st, int plan, float rms_eps = -1.f);
constexpr int kGemmTileN = 128;     // columns per argmax tile

// host_util.cu
int device_sm_count();
// 3-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
bool tma_map_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                     uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

}  // namespace vc
