// CUDA-core (SIMT) forward of exact attention in fp32 (fa_fwd_f32): no operand is rounded to a
// tensor-core type, for callers that need fp32 results.
//
// Method: "账房先生的奔命：Flash Attention 与内存 I/O 革命" §六 (Tiling + Online Softmax).  K and V
// are streamed through shared memory in blocks of 32 keys; each warp keeps, per query row, the
// running max m, the running exp-sum l and an unnormalised output accumulator that is multiplied by
// exp(m_old - m_new) whenever the max grows (the rescale of the FlashAttention fable on
// ckw19810413.github.io, section 兩大核心魔法).  Only O and LSE = m + ln l are written.
//
// Thread mapping: one warp owns kRows query rows; lane l computes the score of key l of the staged
// block, and owns output columns c = l, l+32, l+64, l+96 of the accumulators.

#include <math.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 4;
constexpr int kRows = 4;        // rows per warp
constexpr int kBlk = 32;        // keys (or queries) staged per step
constexpr int kMaxD = 128;
constexpr int kCols = kMaxD / 32;

__device__ __forceinline__ float to_f(float x) { return x; }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }

__device__ __forceinline__ float warp_max(float x) {
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Copies rows [r0, r0+kBlk) of a [N, d] head into shared memory as fp32 with row pitch d+1
// (the odd pitch keeps lane-per-row reads free of bank conflicts); rows >= N are zero.
template <typename T>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int r0, int N, int d) {
    const int pitch = d + 1;
    for (int idx = threadIdx.x; idx < kBlk * d; idx += blockDim.x) {
        int r = idx / d, c = idx - r * d;
        float x = 0.f;
        if (r0 + r < N) x = to_f(src[(size_t)(r0 + r) * d + c]);
        dst[r * pitch + c] = x;
    }
}

// ---------------------------------------------------------------------------------------------
// Forward.  grid = B*H*ceil(N / (kWarps*kRows)) (head-major), block = kWarps*32.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                T* __restrict__ o, float* __restrict__ lse, int N, int d, int blocks_per_head, float scale) {
    extern __shared__ float smem[];
    const int pitch = d + 1;
    float* ks = smem;                       // [kBlk][pitch]
    float* vs = ks + kBlk * pitch;          // [kBlk][pitch]
    float* qs = vs + kBlk * pitch;          // [kWarps*kRows][d]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = blockIdx.x / blocks_per_head;
    const int blk = blockIdx.x % blocks_per_head;
    const T* qh = q + head * N * d;
    const T* kh = k + head * N * d;
    const T* vh = v + head * N * d;
    const int row0 = blk * (kWarps * kRows) + warp * kRows;

    for (int idx = threadIdx.x; idx < kWarps * kRows * d; idx += blockDim.x) {
        int r = idx / d, c = idx - r * d;
        int gr = blk * (kWarps * kRows) + r;
        qs[idx] = gr < N ? to_f(qh[(size_t)gr * d + c]) : 0.f;
    }
    const float* qw = qs + warp * kRows * d;

    float m[kRows], l[kRows], acc[kRows][kCols];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int t = 0; t < kCols; ++t) acc[r][t] = 0.f;
    }

    for (int j0 = 0; j0 < N; j0 += kBlk) {
        __syncthreads();
        stage_rows(ks, kh, j0, N, d);
        stage_rows(vs, vh, j0, N, d);
        __syncthreads();

        // scores of this lane's key against the warp's rows
        float s[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) s[r] = 0.f;
        for (int c = 0; c < d; ++c) {
            float kc = ks[lane * pitch + c];
#pragma unroll
            for (int r = 0; r < kRows; ++r) s[r] = fmaf(qw[r * d + c], kc, s[r]);
        }
        const bool valid = j0 + lane < N;
        float p[kRows], alpha[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            s[r] = valid ? s[r] * scale : -INFINITY;
            float m_new = fmaxf(m[r], warp_max(s[r]));
            alpha[r] = (m[r] == -INFINITY) ? 0.f : expf(m[r] - m_new);
            p[r] = valid ? expf(s[r] - m_new) : 0.f;
            l[r] = alpha[r] * l[r] + warp_sum(p[r]);
            m[r] = m_new;
#pragma unroll
            for (int t = 0; t < kCols; ++t) acc[r][t] *= alpha[r];
        }
        for (int jj = 0; jj < kBlk; ++jj) {
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float pj = __shfl_sync(0xffffffffu, p[r], jj);
#pragma unroll
                for (int t = 0; t < kCols; ++t) {
                    int c = lane + 32 * t;
                    if (c < d) acc[r][t] = fmaf(pj, vs[jj * pitch + c], acc[r][t]);
                }
            }
        }
    }

#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        int gr = row0 + r;
        if (gr >= N) continue;
        float inv = 1.f / l[r];
#pragma unroll
        for (int t = 0; t < kCols; ++t) {
            int c = lane + 32 * t;
            if (c < d) o[(head * N + gr) * d + c] = from_f<T>(acc[r][t] * inv);
        }
        if (lane == 0) lse[head * N + gr] = m[r] + logf(l[r]);
    }
}

template <typename T>
cudaError_t launch_fwd(const T* q, const T* k, const T* v, T* o, float* lse, const Shape& s,
                       float scale, cudaStream_t st) {
    const int rows_per_block = kWarps * kRows;
    const int bph = (s.N + rows_per_block - 1) / rows_per_block;
    if ((long long)bph * s.heads() > INT32_MAX) return cudaErrorInvalidConfiguration;
    const unsigned grid = (unsigned)(bph * s.heads());
    size_t smem = sizeof(float) * (2 * kBlk * (s.d + 1) + kWarps * kRows * s.d);
    cudaError_t e = set_max_dynamic_smem((const void*)fwd_simt_kernel<T>, (int)smem);
    if (e != cudaSuccess) return e;
    fwd_simt_kernel<T><<<grid, kWarps * 32, smem, st>>>(q, k, v, o, lse, s.N, s.d, bph, scale);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_fwd_simt_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                const Shape& s, float scale, cudaStream_t st) {
    return launch_fwd<float>(q, k, v, o, lse, s, scale, st);
}

}  // namespace fa
