// lightning_attn_backward_noalloc: the backward pass with its scratch space
// in a fixed array inside this library instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory when they call
// the backward pass -- for example code running under another framework's
// memory manager, which owns the device pool and does not allow raw
// cudaMalloc calls, or a serving or training loop that must not call
// cudaMalloc in its steady state because cudaMalloc can synchronise the
// device.  Such callers still pass their inputs and outputs; only the
// scratch of the time-reversed copies of the CUDA-core path comes from here
// (the tensor-core path needs none).
//
// The array lives in device memory of every GPU that loads the library, from
// module load until the process exits.  Its address is looked up once per
// device (cudaGetSymbolAddress on the first call made with that device
// current), and again if the device's context has been destroyed and made
// anew since (cudaDeviceReset); the array's name in host code is only a
// stand-in for the symbol and must never be passed to a kernel.  All calls share the one array, so
// calls that overlap on the GPU (different streams, or different host
// threads, without ordering between them) race on it and give wrong results;
// calls serialised on one stream are safe.  Nothing in the array needs to
// start at zero: every byte the backward pass reads from it was written
// earlier in the same call.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "la_internal.h"
#include "lightning_attn.h"

namespace la {
namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_backward_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context the address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Unique id of the current context (0 if it cannot be read).  A device whose
// primary context was destroyed (cudaDeviceReset) and made again gets a new
// id, and the module holding the array may then sit at a new address.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_backward_scratch on the current device, looked up with
// cudaGetSymbolAddress on the first call for that device and again whenever
// the device's context has changed since.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // (id 0 -- no context made current yet -- always looks the address up;
    // the lookup itself makes the runtime set up the device's context)
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_backward_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace la

extern "C" int64_t lightning_attn_backward_noalloc_max_bytes(void) {
    return (int64_t)la::kScratchBytes;
}

extern "C" la_status lightning_attn_backward_noalloc(
    const void *q, const void *k, const void *v, const float *decay, const int32_t *cu_seqlens,
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, int32_t head_dim, int32_t chunk,
    la_dtype dtype, const void *d_out, void *d_q, void *d_k, void *d_v, void *stream) {
    // every argument check of the workspace entry point comes first, so
    // errors, empty calls and unsupported block sizes report as they do there
    bool work = false, needs_ws = false;
    const la_status chk = la::backward_check(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                             num_heads, head_dim, chunk, dtype, d_out, d_q, d_k,
                                             d_v, &work, &needs_ws);
    if (chk != LA_OK || !work) return chk;
    // the tensor-core path (bf16, head_dim 128) uses no scratch: no size limit
    if (!needs_ws)
        return lightning_attn_backward(q, k, v, decay, cu_seqlens, num_seqs, total_tokens,
                                       num_heads, head_dim, chunk, dtype, d_out, d_q, d_k, d_v,
                                       nullptr, 0, stream);
    const int64_t need =
        lightning_attn_backward_workspace_bytes(total_tokens, num_heads, head_dim, dtype);
    if (need < 0 || need > (int64_t)la::kScratchBytes) {
        la::set_last_error(
            "backward_noalloc: %lld bytes of scratch needed (total_tokens * num_heads * "
            "head_dim too large), the built-in array holds %lld",
            (long long)need, (long long)la::kScratchBytes);
        return LA_ERR_INVALID_ARG;
    }
    void *scratch = nullptr;
    const cudaError_t e = la::scratch_address(&scratch);
    if (e != cudaSuccess) {
        la::set_last_error("backward_noalloc: scratch address lookup failed: %s",
                           cudaGetErrorString(e));
        return LA_ERR_CUDA;
    }
    return lightning_attn_backward(q, k, v, decay, cu_seqlens, num_seqs, total_tokens, num_heads,
                                   head_dim, chunk, dtype, d_out, d_q, d_k, d_v, scratch,
                                   (int64_t)la::kScratchBytes, stream);
}
