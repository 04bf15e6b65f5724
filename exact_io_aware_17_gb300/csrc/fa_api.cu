// C entry points of libfa.so: argument checks, workspace layout, dispatch to the kernels.
// The declarations and their contracts are in include/fa.h.

#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <mutex>
#include <stdlib.h>
#include <stdarg.h>
#include <stdio.h>

#include "fa_internal.h"

namespace fa {

static thread_local char g_last_error[512] = "";
static thread_local cudaEvent_t g_bwd_main_events[2] = {nullptr, nullptr};

BwdTiming take_bwd_main_events() {
    const BwdTiming t{g_bwd_main_events[0], g_bwd_main_events[1]};
    g_bwd_main_events[0] = g_bwd_main_events[1] = nullptr;
    return t;
}

fa_status set_error(fa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

std::atomic<unsigned long long>& launch_counter() {
    static std::atomic<unsigned long long> n{0};
    return n;
}
void count_launches(int n) { launch_counter().fetch_add((unsigned long long)n, std::memory_order_relaxed); }

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

BwdWorkspace bwd_workspace_layout(const Shape& s) {
    BwdWorkspace w;
    const size_t rows = (size_t)s.rows();
    const size_t padded = (size_t)s.heads() * bwd_padded_rows(s.N);
    w.dq_acc = 0;
    w.row_d = round256(rows * (size_t)s.d * sizeof(float));
    w.lse2 = w.row_d + round256(padded * sizeof(float));
    w.total = w.lse2 + round256(padded * sizeof(float));
    return w;
}

static cudaError_t tmap_encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult qres;
        void* fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qres);
        if (e != cudaSuccess) return e;
        if (qres != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    *out = encode;
    return cudaSuccess;
}

// Encoded tensor maps, keyed by everything that goes into them (a map holds the array's address, its shape
// and the box, nothing of the device or context), so that repeated calls on the same buffers skip the
// driver's encoding.  A small table with round-robin replacement, shared by all threads.
namespace {
struct TmapKey {
    const void* base;
    int64_t heads;
    int d, N, box_cols, box_rows, dtype;
    bool operator==(const TmapKey& o) const {
        return base == o.base && heads == o.heads && d == o.d && N == o.N && box_cols == o.box_cols &&
               box_rows == o.box_rows && dtype == o.dtype;
    }
};
constexpr int kTmapCacheSize = 64;
struct TmapEntry {
    bool used;
    TmapKey key;
    CUtensorMap map;
};
TmapEntry g_tmap_cache[kTmapCacheSize];
int g_tmap_next = 0;
std::mutex g_tmap_mu;

bool tmap_lookup(const TmapKey& k, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    for (const TmapEntry& e : g_tmap_cache)
        if (e.used && e.key == k) {
            *out = e.map;
            return true;
        }
    return false;
}

void tmap_store(const TmapKey& k, const CUtensorMap& map) {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    TmapEntry& e = g_tmap_cache[g_tmap_next];
    g_tmap_next = (g_tmap_next + 1) % kTmapCacheSize;
    e.used = true;
    e.key = k;
    e.map = map;
}
}  // namespace

cudaError_t set_max_dynamic_smem(const void* func, int bytes) {
    // The limit set so far per kernel and device: the attribute call is made only to raise it.
    static std::mutex mu;
    static struct {
        const void* func;
        int dev, bytes;
    } set[256];
    static int n_set = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    int i = 0;
    while (i < n_set && !(set[i].func == func && set[i].dev == dev)) ++i;
    if (i < n_set && set[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (i < n_set) set[i].bytes = bytes;
    else if (n_set < 256) set[n_set++] = {func, dev, bytes};
    return cudaSuccess;
}

cudaError_t make_tmap_f32_3d(CUtensorMap* map, const float* base, int d, int N, int64_t heads, int box_cols,
                             int box_rows, bool swizzle128) {
    const TmapKey key{base, heads, d, N, box_cols, box_rows, swizzle128 ? 2 : 1};
    if (tmap_lookup(key, map)) return cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    cudaError_t e = tmap_encoder(&encode);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    tmap_store(key, *map);
    return cudaSuccess;
}

cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int N, int64_t heads, int box_rows) {
    const TmapKey key{base, heads, d, N, 64, box_rows, 0};
    if (tmap_lookup(key, map)) return cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    cudaError_t e = tmap_encoder(&encode);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    tmap_store(key, *map);
    return cudaSuccess;
}

static std::atomic<int> g_force_wait_timeout{0};

WaitPolicy wait_policy() {
    if (g_force_wait_timeout.load(std::memory_order_relaxed))
        return WaitPolicy{20000000LL, 1};  // ~10 ms, and the kernels' Q loads withheld
    return WaitPolicy{4000000000LL, 0};   // ~2 s: no legitimate wait comes near it
}

int device_sm_count() {
    static int counts[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        counts[dev] = n;
    }
    return counts[dev];
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Common checks of every entry point; returns FA_OK or the error (message already recorded).
static fa_status check_shape(const char* fn, int B, int H, int N, int d, float scale) {
    if (B < 1 || H < 1 || N < 1 || d < 1)
        return set_error(FA_ERR_INVALID_ARG, "%s: B, H, N, d must be >= 1 (got B=%d H=%d N=%d d=%d)", fn, B, H, N, d);
    if ((int64_t)B * H > INT32_MAX || (int64_t)N * d > INT32_MAX)
        return set_error(FA_ERR_INVALID_ARG, "%s: B*H and N*d must fit in int32", fn);
    if (!isfinite(scale) || !(scale > 0.f))
        return set_error(FA_ERR_INVALID_ARG, "%s: scale must be finite and > 0 (got %g)", fn, (double)scale);
    return FA_OK;
}

static fa_status check_ptrs(const char* fn, const void* const* ptrs, const char* const* names, int n) {
    for (int i = 0; i < n; ++i) {
        if (!ptrs[i]) return set_error(FA_ERR_INVALID_ARG, "%s: %s is NULL", fn, names[i]);
        if (!aligned16(ptrs[i])) return set_error(FA_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, names[i]);
    }
    return FA_OK;
}

static fa_status launch_result(const char* fn, cudaError_t e) {
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return FA_OK;
}


fa_status check_bwd_shape(const char* fn, int B, int H, int N, int d, float scale) {
    fa_status st = check_shape(fn, B, H, N, d, scale);
    if (st) return st;
    if (d != 64 && d != 128) return set_error(FA_ERR_UNSUPPORTED, "%s: d must be 64 or 128 (got %d)", fn, d);
    return FA_OK;
}

fa_status bwd_entry(const char* fn, const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                    void* workspace, size_t workspace_bytes, void* stream, BwdTiming timing) {
    g_last_error[0] = 0;
    fa_status st = check_bwd_shape(fn, B, H, N, d, scale);
    if (st) return st;
    const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
    const char* names[] = {"q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv", "workspace"};
    if ((st = check_ptrs(fn, ptrs, names, 10))) return st;
    if ((uintptr_t)workspace & 255u) return set_error(FA_ERR_INVALID_ARG, "%s: workspace is not 256-byte aligned", fn);
    Shape s{B, H, N, d};
    BwdWorkspace w = bwd_workspace_layout(s);
    if (workspace_bytes < w.total)
        return set_error(FA_ERR_INVALID_ARG, "%s: workspace holds %zu bytes, needs %zu", fn, workspace_bytes, w.total);
    return launch_result(fn, launch_bwd_tc(q, k, v, o, dout, lse, dq, dk, dv, s, scale, workspace,
                                           (cudaStream_t)stream, timing));
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_last_error_string(void) { return g_last_error; }

unsigned long long fa_kernel_launches(void) { return fa::launch_counter().load(std::memory_order_relaxed); }

void fa_debug_time_bwd_main(void* start_event, void* stop_event) {
    g_bwd_main_events[0] = (cudaEvent_t)start_event;
    g_bwd_main_events[1] = (cudaEvent_t)stop_event;
}

void fa_test_force_wait_timeout(int enable) { g_force_wait_timeout.store(enable != 0, std::memory_order_relaxed); }

static fa_status fwd_common(const char* fn, const void* q, const void* k, const void* v, void* o, float* lse, int B,
                            int H, int N, int d, float scale, void* stream, bool stepnorm) {
    g_last_error[0] = 0;
    fa_status st = check_shape(fn, B, H, N, d, scale);
    if (st) return st;
    const void* ptrs[] = {q, k, v, o, lse};
    const char* names[] = {"q", "k", "v", "o", "lse"};
    if ((st = check_ptrs(fn, ptrs, names, 5))) return st;
    if (d != 64 && d != 128) return set_error(FA_ERR_UNSUPPORTED, "%s: d must be 64 or 128 (got %d)", fn, d);
    Shape s{B, H, N, d};
    return launch_result(fn, launch_fwd_tc(q, k, v, o, lse, s, scale, (cudaStream_t)stream, stepnorm));
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, void* stream) {
    return fwd_common("fa_fwd", q, k, v, o, lse, B, H, N, d, scale, stream, false);
}

fa_status fa_fwd_stepnorm(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int N, int d, float scale, void* stream) {
    return fwd_common("fa_fwd_stepnorm", q, k, v, o, lse, B, H, N, d, scale, stream, true);
}

fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                     int B, int H, int N, int d, float scale, void* stream) {
    g_last_error[0] = 0;
    fa_status st = check_shape("fa_fwd_f32", B, H, N, d, scale);
    if (st) return st;
    const void* ptrs[] = {q, k, v, o, lse};
    const char* names[] = {"q", "k", "v", "o", "lse"};
    if ((st = check_ptrs("fa_fwd_f32", ptrs, names, 5))) return st;
    if (d > 128 || d % 4 != 0)
        return set_error(FA_ERR_UNSUPPORTED, "fa_fwd_f32: d must be a multiple of 4 and <= 128 (got %d)", d);
    Shape s{B, H, N, d};
    return launch_result("fa_fwd_f32", launch_fwd_simt_f32(q, k, v, o, lse, s, scale, (cudaStream_t)stream));
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return bwd_workspace_layout(Shape{B, H, N, d}).total;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return fa::bwd_entry("fa_bwd", q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, workspace, workspace_bytes,
                         stream, fa::take_bwd_main_events());
}

fa_status fa_check_status(void* stream) {
    g_last_error[0] = 0;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return set_error(FA_ERR_CUDA, "fa_check_status: %s", cudaGetErrorString(e));
    int codes[] = {fwd_tc_read_and_clear_status(s), bwd_tc_read_and_clear_status(s)};
    for (int c : codes) {
        if (c < 0) return set_error(FA_ERR_CUDA, "fa_check_status: could not read the device status word");
        if (c) return set_error(FA_ERR_TIMEOUT, "fa_check_status: a kernel gave up a bounded wait (code %d)", c);
    }
    return FA_OK;
}

}  // extern "C"
