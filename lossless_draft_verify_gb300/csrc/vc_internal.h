// vc_internal.h -- launchers shared between the kernel files and the C-ABI
// entry points (vc_api.cu).  Arguments are validated by the caller.
#pragma once

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
cudaError_t accept(const void *logits, vc_dtype dt, const int32_t *drafts, int B, int D, int V,
                   int32_t *n_acc, int32_t *next_tok, void *ws, cudaStream_t st);

// draft_attn.cu
size_t draft_ws_bytes(const vc_cache_view *view, int Hq);
cudaError_t draft_attn(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq,
                       float sm_scale, void *out, void *ws, cudaStream_t st);

// verify_attn.cu
size_t verify_ws_bytes(vc_dtype dt, int B, int Dq, int Hq, int Hkv, int d, int max_ctx);
bool verify_uses_tensor_cores(vc_dtype dt, int Dq, int Hq, int Hkv, int d);
cudaError_t verify_attn(const void *q, const void *k, const void *v, vc_dtype dt,
                        const int32_t *ctx_len, int B, int Dq, int Hq, int Hkv, int d,
                        int L_stride, int max_ctx, float sm_scale, void *out, void *ws,
                        cudaStream_t st);

// drop.cu
size_t drop_ws_bytes(int B, int H, int L);
cudaError_t drop_tokens(const float *scores, const void *k, const void *v, vc_dtype dt, int B,
                        int H, int L, int d, int64_t keep_top, int64_t keep_recent,
                        int32_t *kept_idx, void *k_out, void *v_out, void *ws, cudaStream_t st);

}  // namespace vc
