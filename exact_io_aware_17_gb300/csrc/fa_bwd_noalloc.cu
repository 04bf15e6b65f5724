// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs a scratch buffer from its caller.  Some callers cannot provide one: an operator
// plugin that a host framework hands only its input and output buffers, or code that must not call
// cudaMalloc because that call can synchronise the whole device.  This entry point uses a fixed
// scratch array compiled into the library instead, and then runs exactly the same kernels as fa_bwd.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds
// kNoallocScratchBytes of it until the process exits.  Host code cannot use the array's name as a
// device address, so the address is looked up once per device with cudaGetSymbolAddress (on the
// first call made while that device is current) and cached.

#include <atomic>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)FA_BWD_NOALLOC_MAX_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, void* stream) {
    using namespace fa;
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (need > kNoallocScratchBytes)
        return set_error(FA_ERR_INVALID_ARG,
                         "fa_bwd_noalloc: B=%d H=%d N=%d d=%d needs %zu bytes of scratch, more than the %zu bytes "
                         "of the library's static scratch; use fa_bwd with a caller-provided workspace",
                         B, H, N, d, need, kNoallocScratchBytes);
    void* scratch = nullptr;
    if (need > 0) {
        cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess)
            return set_error(FA_ERR_CUDA, "fa_bwd_noalloc: cudaGetSymbolAddress of the static scratch failed: %s",
                             cudaGetErrorString(e));
    }
    // fa_bwd checks every other argument and clears, before use, every part of the scratch that
    // must start at zero.
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, scratch, kNoallocScratchBytes, stream);
}
