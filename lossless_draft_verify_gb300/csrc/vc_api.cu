// vc_api.cu -- the C-ABI entry points declared in include/vc.h: host-side
// argument validation, then dispatch to the kernel launchers.
#include <cstring>

#include "vc_common.cuh"
#include "vc_internal.h"

using namespace vc;

namespace {

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline size_t esize(vc_dtype dt) { return dt == VC_BF16 ? 2 : 4; }
inline bool dtype_ok(vc_dtype dt) { return dt == VC_BF16 || dt == VC_F32; }
inline vc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? VC_OK : VC_ERR_CUDA; }
// Largest B * (D + 1) acceptance serves: one CTA row of the grid per logit row.
constexpr long kAcceptMaxRows = 65535;
inline bool is_memory_type(const void *p, cudaMemoryType t)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == t;
}

bool qcache_ok(const vc_qcache *c)
{
    if (!c || !c->records || !c->k_res || !c->v_res || !c->n_groups || !c->seq_len) return false;
    if (c->B <= 0 || c->Hkv <= 0 || (c->d != 64 && c->d != 128)) return false;
    if ((c->cfg.bits != 2 && c->cfg.bits != 4) || c->cfg.group != 32 || c->cfg.residual < 0) return false;
    if (c->cfg.rotate != 0 && c->cfg.rotate != 1) return false;
    if (c->max_groups < 0 || c->res_cap < c->cfg.residual + c->cfg.group) return false;
    if (!dtype_ok(c->res_dtype)) return false;
    if (!aligned(c->records, 256) || !aligned(c->k_res, 16) || !aligned(c->v_res, 16)) return false;
    return true;
}

// One CTA waits, with the library's bounded wait, on an mbarrier that nothing
// completes: the wait gives up and records a timeout (where = 77).
__global__ void wait_probe_kernel(int32_t *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) report_timeout(status, 77);
}

// Pacing of an emulated slower link: chunk i of a paced copy may start only
// at t0 + i * ns_per_chunk, t0 being the time the first pace kernel ran.  One
// thread sleeps until its deadline (at most max_ns past t0, so every wait
// ends).
__global__ void pace_kernel(uint64_t *t0, int first, uint64_t offset_ns, uint64_t max_ns)
{
    if (first) {
        *t0 = globaltimer_ns();
        return;
    }
    const uint64_t start = *t0;
    const uint64_t deadline = start + (offset_ns < max_ns ? offset_ns : max_ns);
    while (globaltimer_ns() < deadline) __nanosleep(2000);
}

}  // namespace

extern "C" {

const char *vc_status_str(vc_status s)
{
    switch (s) {
    case VC_OK: return "ok";
    case VC_ERR_INVALID: return "invalid argument";
    case VC_ERR_UNSUPPORTED: return "unsupported configuration";
    case VC_ERR_CUDA: return "CUDA runtime error";
    case VC_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char *vc_version(void) { return "vericache-gb300 0.1 (sm_103a)"; }

vc_status vc_check(cudaStream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    return cuda_status(e);
}

vc_status vc_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!ws || ws_bytes < (size_t)kStatusBytes || !aligned(ws, 256)) return VC_ERR_INVALID;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

vc_status vc_poll_status(void *ws, cudaStream_t stream)
{
    if (!ws) return VC_ERR_INVALID;
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return VC_ERR_CUDA;
    if (word != 0) {
        e = cudaMemsetAsync(ws, 0, sizeof(word), stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return VC_ERR_CUDA;
        return VC_ERR_TIMEOUT;
    }
    return VC_OK;
}

size_t vc_record_bytes(int bits, int d)
{
    if ((bits != 2 && bits != 4) || d <= 0 || d % 32) return 0;
    return (size_t)2 * 32 * d * bits / 8 + (size_t)8 * d;
}

vc_status vc_quantize_kv(const void *k, const void *v, vc_dtype dt, int B, int Hkv, int L, int L_stride,
                         int d, vc_qcache *cache, cudaStream_t stream)
{
    if (!k || !v || !qcache_ok(cache)) return VC_ERR_INVALID;
    if (!dtype_ok(dt) || dt != cache->res_dtype) return VC_ERR_INVALID;
    if (B != cache->B || Hkv != cache->Hkv || d != cache->d) return VC_ERR_INVALID;
    if (L < 0 || L_stride < L || !aligned(k, 16) || !aligned(v, 16)) return VC_ERR_INVALID;
    const int G = cache->cfg.group, R = cache->cfg.residual;
    const int nq = (L - R > 0) ? ((L - R) / G) * G : 0;
    if (nq / G > cache->max_groups || L - nq > cache->res_cap) return VC_ERR_INVALID;
    return cuda_status(quantize_prefill(k, v, dt, B, Hkv, L, L_stride, d, cache, stream));
}

vc_status vc_qcache_append(vc_qcache *cache, const void *k_new, const void *v_new, const int32_t *n_new,
                           int max_new, int requantize, cudaStream_t stream)
{
    if (!qcache_ok(cache) || !k_new || !v_new || !n_new || max_new < 0) return VC_ERR_INVALID;
    if (max_new == 0) return VC_OK;
    return cuda_status(qcache_append(cache, k_new, v_new, n_new, nullptr, nullptr, max_new, requantize,
                                     stream));
}

vc_status vc_qcache_commit(vc_qcache *cache, const void *k_blk, const void *v_blk, const int32_t *round_len,
                           const int32_t *n_acc, int Dq, cudaStream_t stream)
{
    if (!qcache_ok(cache) || !k_blk || !v_blk || !round_len || !n_acc || Dq <= 0) return VC_ERR_INVALID;
    return cuda_status(qcache_append(cache, k_blk, v_blk, nullptr, round_len, n_acc, Dq, 1, stream));
}

int64_t vc_drop_kept_count(int64_t L, vc_drop_cfg cfg)
{
    if (L < 0 || cfg.keep_top < 0 || cfg.keep_recent < 0) return -1;
    const int64_t R = cfg.keep_recent < L ? cfg.keep_recent : L;
    const int64_t cand = L - R;
    return (cfg.keep_top < cand ? cfg.keep_top : cand) + R;
}

size_t vc_drop_tokens_workspace_bytes(int B, int H, int L)
{
    if (B <= 0 || H <= 0 || L < 0) return 0;
    return drop_ws_bytes(B, H, L);
}

vc_status vc_drop_tokens(const float *scores, const void *k, const void *v, vc_dtype dt, int B, int H, int L,
                         int d, vc_drop_cfg cfg, int32_t *kept_idx, void *k_out, void *v_out, void *ws,
                         size_t ws_bytes, cudaStream_t stream)
{
    if (!scores || !k || !v || !kept_idx || !k_out || !v_out || !ws) return VC_ERR_INVALID;
    if (!dtype_ok(dt) || B <= 0 || H <= 0 || L < 0 || d <= 0) return VC_ERR_INVALID;
    if (cfg.keep_top < 0 || cfg.keep_recent < 0) return VC_ERR_INVALID;
    if ((d * esize(dt)) % 16 || !aligned(k, 16) || !aligned(v, 16) || !aligned(k_out, 16) ||
        !aligned(v_out, 16) || !aligned(ws, 256))
        return VC_ERR_INVALID;
    if (ws_bytes < drop_ws_bytes(B, H, L)) return VC_ERR_INVALID;
    return cuda_status(drop_tokens(scores, k, v, dt, B, H, L, d, cfg.keep_top, cfg.keep_recent, kept_idx,
                                   k_out, v_out, ws, stream));
}

size_t vc_draft_attn_workspace_bytes(const vc_cache_view *view, int Hq)
{
    if (!view) return 0;
    if (view->kind == VC_CACHE_KIVI && !qcache_ok(view->kivi)) return 0;
    if (view->kind == VC_CACHE_DENSE && (view->B <= 0 || view->Hkv <= 0 || view->max_len < 0)) return 0;
    return draft_ws_bytes(view, Hq);
}

vc_status vc_draft_attn(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq, float sm_scale,
                        void *out, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!q || !view || !out || !ws || !dtype_ok(q_dt) || !aligned(ws, 256)) return VC_ERR_INVALID;
    int Hkv, d;
    if (view->kind == VC_CACHE_KIVI) {
        if (!qcache_ok(view->kivi)) return VC_ERR_INVALID;
        Hkv = view->kivi->Hkv;
        d = view->kivi->d;
        if (Hq <= 0 || Hq % Hkv || Hq / Hkv > 4) return VC_ERR_UNSUPPORTED;
    } else if (view->kind == VC_CACHE_DENSE) {
        if (!view->k || !view->v || !view->seq_len || !dtype_ok(view->dt)) return VC_ERR_INVALID;
        if (view->B <= 0 || view->Hkv <= 0 || view->L_stride < view->max_len || view->max_len < 0)
            return VC_ERR_INVALID;
        if (view->d != 64 && view->d != 128) return VC_ERR_UNSUPPORTED;
        if (view->dt != q_dt) return VC_ERR_INVALID;
        if (!aligned(view->k, 16) || !aligned(view->v, 16)) return VC_ERR_INVALID;
        Hkv = view->Hkv;
        d = view->d;
        if (Hq <= 0 || Hq % Hkv || Hq / Hkv > 4) return VC_ERR_UNSUPPORTED;
    } else {
        return VC_ERR_INVALID;
    }
    (void)d;
    if (ws_bytes < draft_ws_bytes(view, Hq)) return VC_ERR_INVALID;
    return cuda_status(draft_attn(q, q_dt, view, Hq, sm_scale, out, ws, stream));
}

size_t vc_draft_attn_h2o_workspace_bytes(const vc_cache_view *view, int Hq)
{
    if (!view || Hq <= 0) return 0;
    if (view->kind == VC_CACHE_KIVI) return qcache_ok(view->kivi) ? draft_h2o_ws_bytes(view, Hq) : 0;
    if (view->kind != VC_CACHE_DENSE || view->dt != VC_BF16 || view->B <= 0 || view->Hkv <= 0 ||
        view->max_len < 0)
        return 0;
    return draft_h2o_ws_bytes(view, Hq);
}

vc_status vc_draft_attn_h2o(const void *q, vc_dtype q_dt, const vc_cache_view *view, int Hq, float sm_scale,
                            void *out, float *scores, int scores_stride, const int32_t *kept_idx, int kept_stride,
                            void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!q || !view || !out || !scores || !ws || !aligned(ws, 256)) return VC_ERR_INVALID;
    if (view->kind == VC_CACHE_KIVI) {
        // rows of a KIVI cache are positions 0 .. seq_len - 1 themselves
        const vc_qcache *c = view->kivi;
        if (!qcache_ok(c) || !dtype_ok(q_dt) || kept_idx) return VC_ERR_INVALID;
        if (Hq <= 0 || Hq % c->Hkv || Hq / c->Hkv > 4) return VC_ERR_UNSUPPORTED;
        if ((long)scores_stride < (long)c->max_groups * c->cfg.group + c->res_cap) return VC_ERR_INVALID;
        if (ws_bytes < draft_h2o_ws_bytes(view, Hq)) return VC_ERR_INVALID;
        return cuda_status(
            draft_attn_h2o(q, q_dt, view, Hq, sm_scale, out, scores, scores_stride, nullptr, 0, ws, stream));
    }
    if (view->kind != VC_CACHE_DENSE || view->dt != VC_BF16 || q_dt != VC_BF16) return VC_ERR_UNSUPPORTED;
    if (!view->k || !view->v || !view->seq_len || view->B <= 0 || view->Hkv <= 0) return VC_ERR_INVALID;
    if (view->L_stride < view->max_len || view->max_len < 0) return VC_ERR_INVALID;
    if (view->d != 64 && view->d != 128) return VC_ERR_UNSUPPORTED;
    if (Hq <= 0 || Hq % view->Hkv || Hq / view->Hkv > 4) return VC_ERR_UNSUPPORTED;
    if (!aligned(view->k, 16) || !aligned(view->v, 16) || !aligned(q, 4)) return VC_ERR_INVALID;
    if (kept_idx ? kept_stride < view->max_len : scores_stride < view->max_len) return VC_ERR_INVALID;
    if (ws_bytes < draft_h2o_ws_bytes(view, Hq)) return VC_ERR_INVALID;
    return cuda_status(draft_attn_h2o(q, q_dt, view, Hq, sm_scale, out, scores, scores_stride, kept_idx, kept_stride,
                                      ws, stream));
}

size_t vc_verify_attn_workspace_bytes(vc_dtype dt, int B, int Dq, int Hq, int Hkv, int d, int max_ctx)
{
    if (!dtype_ok(dt) || B <= 0 || Dq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_ctx < 0) return 0;
    return verify_ws_bytes(dt, B, Dq, Hq, Hkv, d, max_ctx);
}

vc_status vc_verify_attn(const void *q, const void *k, const void *v, vc_dtype dt, const int32_t *ctx_len,
                         int B, int Dq, int Hq, int Hkv, int d, int L_stride, int max_ctx, float sm_scale,
                         void *out, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!q || !k || !v || !ctx_len || !out || !ws || !dtype_ok(dt)) return VC_ERR_INVALID;
    if (B <= 0 || Dq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_ctx < 0) return VC_ERR_INVALID;
    if (d != 64 && d != 128) return VC_ERR_UNSUPPORTED;
    if (L_stride < max_ctx + Dq) return VC_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(ws, 256)) return VC_ERR_INVALID;
    if (ws_bytes < verify_ws_bytes(dt, B, Dq, Hq, Hkv, d, max_ctx)) return VC_ERR_INVALID;
    if (!verify_uses_tensor_cores(dt, Dq, Hq, Hkv, d) && Hq / Hkv > 64) return VC_ERR_UNSUPPORTED;
    return cuda_status(verify_attn(q, k, v, dt, ctx_len, B, Dq, Hq, Hkv, d, L_stride, max_ctx, sm_scale, out,
                                   ws, stream));
}

size_t vc_verify_attn_h2o_workspace_bytes(int B, int Dq, int Hq, int Hkv, int d, int max_ctx)
{
    if (B <= 0 || Dq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_ctx < 0) return 0;
    if (!verify_h2o_supported(VC_BF16, Dq, Hq, Hkv, d)) return 0;
    return verify_h2o_ws_bytes(B, Dq, Hq, Hkv, max_ctx);
}

vc_status vc_verify_attn_h2o(const void *q, const void *k, const void *v, const int32_t *ctx_len, int B, int Dq,
                             int Hq, int Hkv, int d, int L_stride, int max_ctx, float sm_scale, void *out,
                             float *scores, int scores_stride, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!q || !k || !v || !ctx_len || !out || !scores || !ws) return VC_ERR_INVALID;
    if (B <= 0 || Dq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_ctx < 0) return VC_ERR_INVALID;
    if (!verify_h2o_supported(VC_BF16, Dq, Hq, Hkv, d)) return VC_ERR_UNSUPPORTED;
    if (L_stride < max_ctx + Dq || scores_stride < max_ctx + Dq) return VC_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(ws, 256)) return VC_ERR_INVALID;
    if (ws_bytes < verify_h2o_ws_bytes(B, Dq, Hq, Hkv, max_ctx)) return VC_ERR_INVALID;
    return cuda_status(verify_attn_h2o(q, k, v, ctx_len, B, Dq, Hq, Hkv, L_stride, max_ctx, sm_scale, out, scores,
                                       scores_stride, ws, stream));
}

size_t vc_accept_workspace_bytes(int B, int D, int V)
{
    if (B <= 0 || D < 0 || V <= 0) return 0;
    return accept_ws_bytes(B, D, V);
}

vc_status vc_accept(const void *logits, vc_dtype dt, const int32_t *drafts, int B, int D, int V,
                    int32_t *n_acc, int32_t *next_tok, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!logits || !n_acc || !next_tok || !ws || !dtype_ok(dt)) return VC_ERR_INVALID;
    if (B <= 0 || D < 0 || D > 1024 || V <= 0 || (D > 0 && !drafts)) return VC_ERR_INVALID;
    if ((long)B * (D + 1) > kAcceptMaxRows) return VC_ERR_INVALID;
    if (!aligned(ws, 256) || ws_bytes < accept_ws_bytes(B, D, V)) return VC_ERR_INVALID;
    return cuda_status(accept(logits, dt, drafts, B, D, V, n_acc, next_tok, ws, stream));
}

vc_status vc_accept_tiles(const float *tile_max, const int32_t *tile_idx, int n_tiles, const int32_t *drafts, int B,
                          int D, int32_t *n_acc, int32_t *next_tok, cudaStream_t stream)
{
    if (!tile_max || !tile_idx || !n_acc || !next_tok) return VC_ERR_INVALID;
    if (B <= 0 || D < 0 || D > 1024 || n_tiles <= 0 || (D > 0 && !drafts)) return VC_ERR_INVALID;
    return cuda_status(accept_tiles(tile_max, tile_idx, n_tiles, drafts, B, D, n_acc, next_tok, stream));
}

vc_status vc_wait_probe(void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!ws || ws_bytes < (size_t)kStatusBytes || !aligned(ws, 256)) return VC_ERR_INVALID;
    wait_probe_kernel<<<1, 32, 0, stream>>>((int32_t *)ws);
    return cuda_status(cudaGetLastError());
}

vc_status vc_swap_in_paced(void *dst_dev, const void *src_pinned_host, size_t bytes, double gbps,
                           size_t chunk_bytes, void *pace_ws, cudaStream_t side_stream, cudaEvent_t done)
{
    if (!dst_dev || !src_pinned_host || !pace_ws || !aligned(pace_ws, 16)) return VC_ERR_INVALID;
    if (!(gbps > 0.0) || chunk_bytes == 0) return VC_ERR_INVALID;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, src_pinned_host) != cudaSuccess || a.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return VC_ERR_INVALID;
    }
    if (bytes && (!is_memory_type((const uint8_t *)src_pinned_host + bytes - 1, cudaMemoryTypeHost) ||
                  !is_memory_type(dst_dev, cudaMemoryTypeDevice) ||
                  !is_memory_type((const uint8_t *)dst_dev + bytes - 1, cudaMemoryTypeDevice)))
        return VC_ERR_INVALID;
    const double ns_per_byte = 1.0 / gbps;            // GB/s = bytes per ns
    const uint64_t max_ns = 30000000000ull;           // no chunk waits past 30 s
    uint64_t *t0 = (uint64_t *)pace_ws;
    pace_kernel<<<1, 1, 0, side_stream>>>(t0, 1, 0, max_ns);
    for (size_t off = 0; off < bytes; off += chunk_bytes) {
        const size_t n = bytes - off < chunk_bytes ? bytes - off : chunk_bytes;
        if (off > 0) pace_kernel<<<1, 1, 0, side_stream>>>(t0, 0, (uint64_t)(off * ns_per_byte), max_ns);
        if (cudaMemcpyAsync((uint8_t *)dst_dev + off, (const uint8_t *)src_pinned_host + off, n,
                            cudaMemcpyHostToDevice, side_stream) != cudaSuccess)
            return VC_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return VC_ERR_CUDA;
    if (done && cudaEventRecord(done, side_stream) != cudaSuccess) return VC_ERR_CUDA;
    return VC_OK;
}

vc_status vc_swap_in(void *dst_dev, const void *src_pinned_host, size_t bytes, cudaStream_t side_stream,
                     cudaEvent_t done)
{
    if (!dst_dev || !src_pinned_host) return VC_ERR_INVALID;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, src_pinned_host) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_INVALID;
    }
    if (a.type != cudaMemoryTypeHost) return VC_ERR_INVALID;   // pageable or device memory
    cudaPointerAttributes ad;
    if (cudaPointerGetAttributes(&ad, dst_dev) != cudaSuccess || ad.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        return VC_ERR_INVALID;
    }
    if (bytes && (!is_memory_type((const uint8_t *)src_pinned_host + bytes - 1, cudaMemoryTypeHost) ||
                  !is_memory_type((const uint8_t *)dst_dev + bytes - 1, cudaMemoryTypeDevice)))
        return VC_ERR_INVALID;                                 // the range leaves the allocation
    if (bytes) {
        cudaError_t e = cudaMemcpyAsync(dst_dev, src_pinned_host, bytes, cudaMemcpyHostToDevice, side_stream);
        if (e != cudaSuccess) return VC_ERR_CUDA;
    }
    if (done && cudaEventRecord(done, side_stream) != cudaSuccess) return VC_ERR_CUDA;
    return VC_OK;
}

vc_status vc_swap_in_rows(void *dst_dev, const void *src_pinned_host, size_t row_bytes, size_t rows,
                          size_t pitch_rows, size_t blocks, cudaStream_t side_stream, cudaEvent_t done)
{
    if (!dst_dev || !src_pinned_host || rows > pitch_rows) return VC_ERR_INVALID;
    if (row_bytes && blocks && pitch_rows && rows) {
        const size_t pitch = row_bytes * pitch_rows, width = row_bytes * rows;
        const size_t last = (blocks - 1) * pitch + width - 1;       // the last byte copied
        if (!is_memory_type(src_pinned_host, cudaMemoryTypeHost) ||
            !is_memory_type((const uint8_t *)src_pinned_host + last, cudaMemoryTypeHost) ||
            !is_memory_type(dst_dev, cudaMemoryTypeDevice) ||
            !is_memory_type((const uint8_t *)dst_dev + last, cudaMemoryTypeDevice))
            return VC_ERR_INVALID;                                 // pageable, or the range leaves the allocation
        cudaError_t e = cudaMemcpy2DAsync(dst_dev, pitch, src_pinned_host, pitch, width, blocks,
                                          cudaMemcpyHostToDevice, side_stream);
        if (e != cudaSuccess) return VC_ERR_CUDA;
    }
    if (done && cudaEventRecord(done, side_stream) != cudaSuccess) return VC_ERR_CUDA;
    return VC_OK;
}

}  // extern "C"
