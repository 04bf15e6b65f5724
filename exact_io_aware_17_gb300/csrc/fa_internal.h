// Host-side declarations shared by the translation units of libfa.so (no device code here).
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fa.h"

namespace fa {

// Shape of one attention call: B*H independent heads of N rows and head size d.
struct Shape {
    int B, H, N, d;
    int64_t heads() const { return (int64_t)B * H; }
    int64_t rows() const { return heads() * N; }
};

// Records a message for fa_last_error_string() and returns `st`.
fa_status set_error(fa_status st, const char* fmt, ...);

// Each kernel translation unit owns one device status word; these read it (after a stream sync)
// and clear it.  They return the first nonzero code recorded, or 0.
int fwd_tc_read_and_clear_status(cudaStream_t s);
int bwd_tc_read_and_clear_status(cudaStream_t s);

// Workspace sections of the backward pass (byte offsets from the workspace base).
struct BwdWorkspace {
    size_t dq_acc, row_d, lse2, total;
};
BwdWorkspace bwd_workspace_layout(const Shape& s);
// Rows per head of the backward's per-row arrays: N rounded up to the 128-query step of the kernel.
inline int bwd_padded_rows(int N) { return (N + 127) / 128 * 128; }

// Budget of the kernels' bounded waits (~2 s of clock), and whether the tensor-core kernels withhold their
// Q loads with a ~10 ms budget so that their first wait runs out.  The latter is only ever set by an
// explicit fa_test_force_wait_timeout(1) call, which tests of the failure path make.
struct WaitPolicy {
    long long budget_cycles;
    int starve;
};
WaitPolicy wait_policy();

// Multiprocessor count of the current device (cached per device).
int device_sm_count();

// Makes a kernel's dynamic shared-memory limit on the current device at least `bytes` (the attribute call is
// made only when the limit has to rise).
cudaError_t set_max_dynamic_smem(const void* func, int bytes);

// Launches `kernel` with programmatic stream serialisation: it may start while the kernel ahead of it on
// `st` is finishing, and must itself wait (griddepcontrol.wait) before it reads anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Encodes a TMA descriptor for a bf16 [heads, N, d] array (d innermost) with boxes of 64 columns x
// `box_rows` rows x 1 head and 128-byte swizzling; rows beyond N read as zero.  Encoded maps are cached by
// their arguments (address, shape, box), so repeated calls on the same buffers cost a table lookup.
cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int N, int64_t heads, int box_rows);
// fp32 [heads][N][d] viewed as (d, N, heads), boxes of box_cols x box_rows (box_cols * 4 bytes a multiple of
// 16; 128 bytes when swizzled): the dQ accumulator as the target of tensor reduce-adds.  swizzle128: the
// shared-memory box has 128-byte swizzling (16-byte chunk c of row r at chunk c ^ (r % 8)).
cudaError_t make_tmap_f32_3d(CUtensorMap* map, const float* base, int d, int N, int64_t heads, int box_cols,
                             int box_rows, bool swizzle128);

// Launchers (return cudaGetLastError() of their launches).
cudaError_t launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, const Shape& s,
                          float scale, cudaStream_t st, bool stepnorm);
cudaError_t launch_fwd_simt_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                const Shape& s, float scale, cudaStream_t st);
// Events recorded around the backward's main kernel (both null: none), see fa_debug_time_bwd_main.
struct BwdTiming {
    cudaEvent_t start, stop;
};
cudaError_t launch_bwd_tc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, const Shape& s, float scale,
                          void* workspace, cudaStream_t st, BwdTiming timing);

// Checks of the backward's shape, scale and head size (FA_OK or the error, message recorded with `fn`).
fa_status check_bwd_shape(const char* fn, int B, int H, int N, int d, float scale);
// The backward entry point under the name `fn`: every argument check, then the launches.
fa_status bwd_entry(const char* fn, const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                    void* workspace, size_t workspace_bytes, void* stream, BwdTiming timing);

// The events that the calling thread's next backward call records around its main kernel (both null:
// none); taking them clears them, so each backward entry point takes them first, whether it then launches
// or fails its checks (fa_debug_time_bwd_main).
BwdTiming take_bwd_main_events();

// Adds n to the process-wide count of kernels this library has launched (read by fa_kernel_launches).
void count_launches(int n);
std::atomic<unsigned long long>& launch_counter();

}  // namespace fa
