// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs a scratch buffer from its caller.  Some callers cannot provide one: an operator
// plugin that a host framework hands only its input and output buffers, or code that must not call
// cudaMalloc because that call can synchronise the whole device.  This entry point uses a fixed
// scratch array compiled into the library instead, and then runs exactly the same kernels as fa_bwd.
//
// The array is a file-scope __device__ variable: every GPU that loads this library holds
// kNoallocScratchBytes of it until the process exits.  Host code cannot use the array's name as a
// device address, so the address is looked up with cudaGetSymbolAddress while the device is current.
// The lookup is cached per device together with the CUDA context it was made in: after a
// cudaDeviceReset the device gets a new primary context, the module is loaded again and the array may
// move, so a changed context makes the next call look the address up again.

#include <cudaTypedefs.h>

#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)FA_BWD_NOALLOC_MAX_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct ScratchEntry {
    CUcontext ctx;
    void* addr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

cudaError_t current_context(CUcontext* out) {
    static PFN_cuCtxGetCurrent_v4000 get = nullptr;
    if (!get) {
        cudaDriverEntryPointQueryResult qres;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &qres);
        if (e != cudaSuccess) return e;
        if (qres != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        get = (PFN_cuCtxGetCurrent_v4000)fn;
    }
    return get(out) == CUDA_SUCCESS ? cudaSuccess : cudaErrorContextIsDestroyed;
}

// Device address of the scratch array in the current device's current context.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CUcontext ctx = nullptr;
    if ((e = current_context(&ctx)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& ent = g_scratch[dev];
    if (ctx == nullptr || ent.addr == nullptr || ent.ctx != ctx) {
        // The lookup also makes the runtime bind the device's primary context to this thread if nothing
        // had yet, so the context is read again after it.
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess) return e;
        if ((e = current_context(&ctx)) != cudaSuccess) return e;
        ent.ctx = ctx;
        ent.addr = p;
    }
    *out = ent.addr;
    return cudaSuccess;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, void* stream) {
    using namespace fa;
    static const char* kFn = "fa_bwd_noalloc";
    const BwdTiming timing = take_bwd_main_events();
    fa_status st = check_bwd_shape(kFn, B, H, N, d, scale);
    if (st) return st;
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (need > kNoallocScratchBytes)
        return set_error(FA_ERR_INVALID_ARG,
                         "fa_bwd_noalloc: B=%d H=%d N=%d d=%d needs %zu bytes of scratch, more than the %zu bytes "
                         "of the library's static scratch; use fa_bwd with a caller-provided workspace",
                         B, H, N, d, need, kNoallocScratchBytes);
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return set_error(FA_ERR_CUDA, "fa_bwd_noalloc: cudaGetSymbolAddress of the static scratch failed: %s",
                         cudaGetErrorString(e));
    // The backward checks every other argument and clears, before use, every part of the scratch that
    // must start at zero.
    return bwd_entry(kFn, q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, scratch, kNoallocScratchBytes,
                     stream, timing);
}
