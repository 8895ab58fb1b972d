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
// cudaGetSymbolAddress and caches it.  The address belongs to the CUDA
// context the module was loaded in, so the cache is keyed on the unique id
// of the calling thread's current context: after a cudaDeviceReset, or from
// another context on the same device, the next call looks the address up
// again (and that call, like the first, must not be inside a stream
// capture).  All calls on a device share the one
// buffer: two calls that overlap on the GPU (different streams, no ordering)
// race on it.  The per-sequence counters that must start at zero are cleared
// on the stream by every call; the rest of the buffer keeps whatever the last
// call left there and is fully rewritten before it is read.
#include <cuda.h>

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
struct Cached {
    unsigned long long ctx_id;
    void *ptr;
};
Cached g_cache[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Driver entry points for the current context and its process-unique id,
// obtained through the runtime (no link-time dependency on libcuda).
bool driver_fns(CtxGetCurrentFn *cur, CtxGetIdFn *id)
{
    static std::once_flag once;
    static CtxGetCurrentFn f_cur = nullptr;
    static CtxGetIdFn f_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
            r1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
            r2 == cudaDriverEntryPointSuccess) {
            f_cur = reinterpret_cast<CtxGetCurrentFn>(p);
            f_id = reinterpret_cast<CtxGetIdFn>(q);
        } else {
            cudaGetLastError();
        }
    });
    *cur = f_cur;
    *id = f_id;
    return f_cur && f_id;
}

// Unique id of the calling thread's current context, 0 if there is none yet.
unsigned long long current_ctx_id(CtxGetCurrentFn cur, CtxGetIdFn id)
{
    CUcontext c = nullptr;
    unsigned long long v = 0;
    if (cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    if (id(c, &v) != CUDA_SUCCESS) return 0;
    return v;
}

// Device address of the scratch buffer in the current device's current
// context (looked up once per context).
vc_status scratch_for_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return VC_ERR_UNSUPPORTED;
    CtxGetCurrentFn cur;
    CtxGetIdFn idf;
    if (!driver_fns(&cur, &idf)) return VC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long id = current_ctx_id(cur, idf);
    if (id != 0 && g_cache[dev].ptr && g_cache[dev].ctx_id == id) {
        *out = g_cache[dev].ptr;
        return VC_OK;
    }
    // First call in this context (or the runtime has not made one current
    // yet): the lookup loads the module and binds the device's context.
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return VC_ERR_CUDA;
    }
    g_cache[dev] = Cached{current_ctx_id(cur, idf), p};
    *out = p;
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
    const cudaError_t e = vc::accept(logits, dt, drafts, B, D, V, n_acc, next_tok, ws, stream, true);
    return e == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}
