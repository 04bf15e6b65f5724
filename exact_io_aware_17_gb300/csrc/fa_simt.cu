// CUDA-core (SIMT) kernels of exact attention: the fp32 forward, and bf16 forward/backward kernels
// that use no tensor cores.
//
// Method: "账房先生的奔命：Flash Attention 与内存 I/O 革命" §六 (Tiling + Online Softmax).  K and V
// are streamed through shared memory in blocks of 32 keys; each warp keeps, per query row, the
// running max m, the running exp-sum l and an unnormalised output accumulator that is multiplied by
// exp(m_old - m_new) whenever the max grows (the rescale of the FlashAttention fable on
// ckw19810413.github.io, section 兩大核心魔法).  Only O and LSE = m + ln l are written.
// The backward recomputes P = exp(scale q.k - LSE) pair by pair (§七 重计算 of the same page).
//
// Thread mapping: one warp owns ROWS query rows (forward, dQ) or ROWS key rows (dK/dV); lane l
// handles key (or query) l of the staged block for the dot products, and output columns
// c = l, l+32, l+64, l+96 for the accumulators.

#include <cuda_bf16.h>
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
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

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
// Forward.  grid = (ceil(N / (kWarps*kRows)), B*H), block = kWarps*32.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                T* __restrict__ o, float* __restrict__ lse, int N, int d, float scale) {
    extern __shared__ float smem[];
    const int pitch = d + 1;
    float* ks = smem;                       // [kBlk][pitch]
    float* vs = ks + kBlk * pitch;          // [kBlk][pitch]
    float* qs = vs + kBlk * pitch;          // [kWarps*kRows][d]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = blockIdx.y;
    const T* qh = q + head * N * d;
    const T* kh = k + head * N * d;
    const T* vh = v + head * N * d;
    const int row0 = blockIdx.x * (kWarps * kRows) + warp * kRows;

    for (int idx = threadIdx.x; idx < kWarps * kRows * d; idx += blockDim.x) {
        int r = idx / d, c = idx - r * d;
        int gr = blockIdx.x * (kWarps * kRows) + r;
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

// ---------------------------------------------------------------------------------------------
// Backward, row term: D_i = sum_c dO_ic * O_ic.  One warp per row.
template <typename T>
__global__ void bwd_rowdot_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                  float* __restrict__ row_d, int64_t rows, int d) {
    int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32) acc = fmaf(to_f(o[row * d + c]), to_f(dout[row * d + c]), acc);
    acc = warp_sum(acc);
    if (lane == 0) row_d[row] = acc;
}

// dK, dV: each warp owns kRows key rows and walks all query blocks.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
bwd_dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ dout, const float* __restrict__ lse,
                     const float* __restrict__ row_d, T* __restrict__ dk, T* __restrict__ dv,
                     int N, int d, float scale) {
    extern __shared__ float smem[];
    const int pitch = d + 1;
    float* qs = smem;                      // [kBlk][pitch]
    float* dos = qs + kBlk * pitch;        // [kBlk][pitch]
    float* ls = dos + kBlk * pitch;        // [kBlk]
    float* ds_ = ls + kBlk;                // [kBlk]
    float* kw_all = ds_ + kBlk;            // [kWarps*kRows][d]  key rows
    float* vw_all = kw_all + kWarps * kRows * d;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = blockIdx.y;
    const size_t hoff = head * (size_t)N * d;
    const int key0 = blockIdx.x * (kWarps * kRows);
    for (int idx = threadIdx.x; idx < kWarps * kRows * d; idx += blockDim.x) {
        int r = idx / d, c = idx - r * d;
        bool ok = key0 + r < N;
        kw_all[idx] = ok ? to_f(k[hoff + (size_t)(key0 + r) * d + c]) : 0.f;
        vw_all[idx] = ok ? to_f(v[hoff + (size_t)(key0 + r) * d + c]) : 0.f;
    }
    const float* kw = kw_all + warp * kRows * d;
    const float* vw = vw_all + warp * kRows * d;

    float adk[kRows][kCols], adv[kRows][kCols];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kCols; ++t) adk[r][t] = adv[r][t] = 0.f;

    for (int i0 = 0; i0 < N; i0 += kBlk) {
        __syncthreads();
        stage_rows(qs, q + hoff, i0, N, d);
        stage_rows(dos, dout + hoff, i0, N, d);
        if (threadIdx.x < kBlk) {
            int i = i0 + threadIdx.x;
            ls[threadIdx.x] = i < N ? lse[head * N + i] : INFINITY;
            ds_[threadIdx.x] = i < N ? row_d[head * N + i] : 0.f;
        }
        __syncthreads();
        const bool valid = i0 + lane < N;
        float s[kRows], dp[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) s[r] = dp[r] = 0.f;
        for (int c = 0; c < d; ++c) {
            float qc = qs[lane * pitch + c], dc = dos[lane * pitch + c];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                s[r] = fmaf(qc, kw[r * d + c], s[r]);
                dp[r] = fmaf(dc, vw[r * d + c], dp[r]);
            }
        }
        float p[kRows], dsv[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            p[r] = valid ? expf(s[r] * scale - ls[lane]) : 0.f;
            dsv[r] = p[r] * (dp[r] - ds_[lane]);
        }
        for (int ii = 0; ii < kBlk; ++ii) {
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float pi = __shfl_sync(0xffffffffu, p[r], ii);
                float di = __shfl_sync(0xffffffffu, dsv[r], ii);
#pragma unroll
                for (int t = 0; t < kCols; ++t) {
                    int c = lane + 32 * t;
                    if (c < d) {
                        adv[r][t] = fmaf(pi, dos[ii * pitch + c], adv[r][t]);
                        adk[r][t] = fmaf(di, qs[ii * pitch + c], adk[r][t]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        int gj = key0 + warp * kRows + r;
        if (gj >= N) continue;
#pragma unroll
        for (int t = 0; t < kCols; ++t) {
            int c = lane + 32 * t;
            if (c < d) {
                dk[hoff + (size_t)gj * d + c] = from_f<T>(adk[r][t] * scale);
                dv[hoff + (size_t)gj * d + c] = from_f<T>(adv[r][t]);
            }
        }
    }
}

// dQ: each warp owns kRows query rows and walks all key blocks.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
bwd_dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ dout, const float* __restrict__ lse,
                   const float* __restrict__ row_d, T* __restrict__ dq, int N, int d, float scale) {
    extern __shared__ float smem[];
    const int pitch = d + 1;
    float* ks = smem;
    float* vs = ks + kBlk * pitch;
    float* qw_all = vs + kBlk * pitch;            // [kWarps*kRows][d]
    float* dow_all = qw_all + kWarps * kRows * d;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = blockIdx.y;
    const size_t hoff = head * (size_t)N * d;
    const int row0 = blockIdx.x * (kWarps * kRows);
    for (int idx = threadIdx.x; idx < kWarps * kRows * d; idx += blockDim.x) {
        int r = idx / d, c = idx - r * d;
        bool ok = row0 + r < N;
        qw_all[idx] = ok ? to_f(q[hoff + (size_t)(row0 + r) * d + c]) : 0.f;
        dow_all[idx] = ok ? to_f(dout[hoff + (size_t)(row0 + r) * d + c]) : 0.f;
    }
    const float* qw = qw_all + warp * kRows * d;
    const float* dow = dow_all + warp * kRows * d;
    float lr[kRows], dr[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        int gi = row0 + warp * kRows + r;
        lr[r] = gi < N ? lse[head * N + gi] : INFINITY;
        dr[r] = gi < N ? row_d[head * N + gi] : 0.f;
    }
    float adq[kRows][kCols];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int t = 0; t < kCols; ++t) adq[r][t] = 0.f;

    for (int j0 = 0; j0 < N; j0 += kBlk) {
        __syncthreads();
        stage_rows(ks, k + hoff, j0, N, d);
        stage_rows(vs, v + hoff, j0, N, d);
        __syncthreads();
        const bool valid = j0 + lane < N;
        float s[kRows], dp[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) s[r] = dp[r] = 0.f;
        for (int c = 0; c < d; ++c) {
            float kc = ks[lane * pitch + c], vc = vs[lane * pitch + c];
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                s[r] = fmaf(qw[r * d + c], kc, s[r]);
                dp[r] = fmaf(dow[r * d + c], vc, dp[r]);
            }
        }
        float dsv[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            float p = valid ? expf(s[r] * scale - lr[r]) : 0.f;
            dsv[r] = p * (dp[r] - dr[r]);
        }
        for (int jj = 0; jj < kBlk; ++jj) {
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                float dj = __shfl_sync(0xffffffffu, dsv[r], jj);
#pragma unroll
                for (int t = 0; t < kCols; ++t) {
                    int c = lane + 32 * t;
                    if (c < d) adq[r][t] = fmaf(dj, ks[jj * pitch + c], adq[r][t]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        int gi = row0 + warp * kRows + r;
        if (gi >= N) continue;
#pragma unroll
        for (int t = 0; t < kCols; ++t) {
            int c = lane + 32 * t;
            if (c < d) dq[hoff + (size_t)gi * d + c] = from_f<T>(adq[r][t] * scale);
        }
    }
}

template <typename T>
cudaError_t launch_fwd(const T* q, const T* k, const T* v, T* o, float* lse, const Shape& s,
                       float scale, cudaStream_t st) {
    const int rows_per_block = kWarps * kRows;
    dim3 grid((s.N + rows_per_block - 1) / rows_per_block, (unsigned)s.heads());
    size_t smem = sizeof(float) * (2 * kBlk * (s.d + 1) + kWarps * kRows * s.d);
    cudaFuncSetAttribute(fwd_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    fwd_simt_kernel<T><<<grid, kWarps * 32, smem, st>>>(q, k, v, o, lse, s.N, s.d, scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                const Shape& s, float scale, cudaStream_t st) {
    return launch_fwd<float>(q, k, v, o, lse, s, scale, st);
}

cudaError_t launch_fwd_simt_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const Shape& s, float scale, cudaStream_t st) {
    using T = __nv_bfloat16;
    return launch_fwd<T>((const T*)q, (const T*)k, (const T*)v, (T*)o, lse, s, scale, st);
}

cudaError_t launch_bwd_simt_bf16(const void* q, const void* k, const void* v, const void* o,
                                 const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                 const Shape& s, float scale, float* row_d, cudaStream_t st) {
    using T = __nv_bfloat16;
    const int64_t rows = s.rows();
    bwd_rowdot_kernel<T><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>((const T*)o, (const T*)dout, row_d, rows, s.d);
    const int per_block = kWarps * kRows;
    dim3 grid((s.N + per_block - 1) / per_block, (unsigned)s.heads());
    size_t smem = sizeof(float) * (2 * kBlk * (s.d + 1) + 2 * kBlk + 2 * kWarps * kRows * s.d);
    cudaFuncSetAttribute(bwd_dkdv_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    bwd_dkdv_simt_kernel<T><<<grid, kWarps * 32, smem, st>>>((const T*)q, (const T*)k, (const T*)v,
                                                             (const T*)dout, lse, row_d, (T*)dk, (T*)dv,
                                                             s.N, s.d, scale);
    size_t smem_q = sizeof(float) * (2 * kBlk * (s.d + 1) + 2 * kWarps * kRows * s.d);
    cudaFuncSetAttribute(bwd_dq_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
    bwd_dq_simt_kernel<T><<<grid, kWarps * 32, smem_q, st>>>((const T*)q, (const T*)k, (const T*)v,
                                                             (const T*)dout, lse, row_d, (T*)dq,
                                                             s.N, s.d, scale);
    return cudaGetLastError();
}

}  // namespace fa
