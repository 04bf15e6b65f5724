// bf16 attention backward on the sm_103a tensor cores (placeholder: status word only).
#include "fa_internal.h"

namespace fa {
namespace {
__device__ int g_bwd_status;
}

int bwd_tc_read_and_clear_status(cudaStream_t st) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_bwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    return v;
}

}  // namespace fa
