// accept_noalloc.cu -- greedy acceptance for callers that cannot allocate
// device memory.
//
// vc_accept() needs a small device workspace from its caller.  Some callers
// cannot provide one: code running inside another framework whose device
// memory all belongs to that framework's pool, plugin hosts that hand out no
// allocator, and latency-critical loops where a cudaMalloc/cudaFree would
// synchronize the device.  vc_accept_noalloc() serves them with a scratch
// buffer that lives in this library's own static device memory.
//
// The buffer is a file-scope __device__ array of kScratchBytes bytes; every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on a
// device (with that device current) looks up its address with
// cudaGetSymbolAddress and caches it.  All calls on a device share the one
// buffer: two calls that overlap on the GPU (different streams, no ordering)
// race on it.  The per-sequence counters that must start at zero are cleared
// on the stream by every call; the rest of the buffer keeps whatever the last
// call left there and is fully rewritten before it is read.
#include <mutex>

#include "vc_common.cuh"
#include "vc_internal.h"

namespace {

// Largest problem served: B <= 1024 sequences and B * (D + 1) <= 16384 logit
// rows.  The workspace layout of vc_accept for that size is 256 (status) +
// 4096 (counters) + 16384 rows * 4 splits * 8 bytes (partial argmax) bytes.
constexpr int kMaxB = 1024;
constexpr int kMaxRows = 16384;
constexpr size_t kScratchBytes = 256 + 4096 + (size_t)kMaxRows * 4 * 8;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_accept_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device (looked up once).
vc_status scratch_for_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return VC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return VC_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return VC_OK;
}

}  // namespace

extern "C" vc_status vc_accept_noalloc(const void *logits, vc_dtype dt, const int32_t *drafts, int B, int D,
                                       int V, int32_t *n_acc, int32_t *next_tok, cudaStream_t stream)
{
    if (!logits || !n_acc || !next_tok || (dt != VC_BF16 && dt != VC_F32)) return VC_ERR_INVALID;
    if (B <= 0 || D < 0 || D > 1024 || V <= 0 || (D > 0 && !drafts)) return VC_ERR_INVALID;
    // sizes beyond the static buffer are refused before anything is enqueued
    if (B > kMaxB || (long)B * (D + 1) > kMaxRows) return VC_ERR_INVALID;
    if (vc::accept_ws_bytes(B, D, V) > kScratchBytes) return VC_ERR_INVALID;
    void *ws = nullptr;
    const vc_status s = scratch_for_current_device(&ws);
    if (s != VC_OK) return s;
    const cudaError_t e = vc::accept(logits, dt, drafts, B, D, V, n_acc, next_tok, ws, stream);
    return e == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}
