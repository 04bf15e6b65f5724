// bf16 attention backward on the sm_103a tensor cores (tcgen05 + TMA + tensor memory).
//
// The pages keep P out of device memory in the backward pass too: it is recomputed from Q, K and the
// saved statistic ("账房先生的奔命：Flash Attention 与内存 I/O 革命" §七 重计算).  The gradient formulas
// themselves are the textbook derivative of O = softmax(scale Q K^T) V:
//     P = exp(scale S - LSE),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D_i = dO_i . O_i,
//     dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels per call:
//   bwd_prep_kernel   -D_i and -LSE_i * log2(e) per query row (padded to a multiple of 64 rows per head;
//                     pad rows get 0 and -inf so they contribute nothing), and zeroes the fp32 dQ
//                     accumulator.  Negated so that the main kernel applies them with packed-pair adds.
//   bwd_tc_kernel     one CTA per (head, block of 128 keys).  K_j, V_j stay in shared memory; the CTA
//                     walks every block of 64 queries i:
//                         S^T  = K_j Q_i^T            K_j as bf16 from tensor memory; fp32 result,
//                                                     double buffered
//                         dP^T = V_j dO_i^T
//                         P^T  = exp2(S^T scale log2e - LSE2_i)    thread = key row; packed fp32
//                                                     pairs (f32x2) for the element-wise work
//                         dS^T = P^T o (dP^T - D_i)
//                         dV_j += P^T dO_i            P^T as bf16 from tensor memory
//                         dK_j += dS^T Q_i            dS^T as bf16 from tensor memory
//                         dQ_i^T = K_j^T dS^T         dS^T as bf16 from shared memory, into the
//                                                     S^T buffer of the step (free once dV used P^T)
//                     and adds dQ_i into the fp32 accumulator with bulk reduce-add copies.
//   bwd_dq_convert    dQ = bf16(scale * accumulator).
//
// Warp roles of bwd_tc_kernel (320 threads): warps 0-3 own the 128 key rows (softmax gradient and the
// dK/dV epilogue), warps 4-7 drain dQ^T (thread = head-dimension index) into the accumulator,
// warp 8 issues TMA loads, warp 9 allocates tensor memory and issues the MMAs.
//
// For d = 64 the dQ^T product still uses M = 128: the A operand's second 64-row half points at a
// zeroed shared-memory block, and the rows it produces are ignored.
//
// TMEM columns: two step buffers [0,64) and [64,128), each holding S^T, then P^T as bf16 over its
// first 32 columns, then dQ^T; dP^T [128,192) (dS^T as bf16 over its first 32); K_j as bf16 [192,192+D/2)
// (the A operand of S^T: it stays resident, so S^T reads only Q_i from shared memory); dV [256,256+D),
// dK [256+D,256+2D).  Three of the five products have N = 64 (the query step), and those MMAs set
// this kernel's pace.

#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

__device__ int g_bwd_status;

constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 64;   // queries per step
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 3;

struct BwdBarriers {
    uint64_t kv_full;
    uint64_t qdo_full[kStages];
    uint64_t qdo_empty[kStages];
    uint64_t s_full[2];
    uint64_t dp_full;
    uint64_t p_ready;
    uint64_t ds_ready;
    uint64_t dq_full;
    uint64_t dq_empty;
    uint64_t ds_free[2];
    uint64_t dkdv_full;
    uint64_t ka_ready;
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kChunkK = BK * 128;          // one 64-column chunk of a K or V tile
    static constexpr uint32_t kChunkQ = BQ * 128;          // one 64-column chunk of a Q or dO tile
    static constexpr uint32_t kKBytes = BK * D * 2;
    static constexpr uint32_t kQBytes = BQ * D * 2;
    static constexpr uint32_t kOffK = 0;
    static constexpr uint32_t kOffZero = kOffK + kKBytes;   // d = 64: zero half that pads K^T to M = 128
    static constexpr uint32_t kZeroBytes = (D == 64) ? kChunkK : 0;
    static constexpr uint32_t kOffV = kOffZero + kZeroBytes;
    static constexpr uint32_t kOffQ = kOffV + kKBytes;
    static constexpr uint32_t kOffDO = kOffQ + kStages * kQBytes;
    static constexpr uint32_t kDSBytes = BK * BQ * 2;      // dS^T tile: 128 key rows x 128 bytes
    static constexpr uint32_t kOffDS = kOffDO + kStages * kQBytes;
    static constexpr uint32_t kDQBytes = BQ * D * 4;       // fp32 dQ staging [BQ][D]
    static constexpr uint32_t kOffDQ = kOffDS + 2 * kDSBytes;
    static constexpr uint32_t kRowBytes = BQ * 4;          // LSE2 or D of one query block
    static constexpr uint32_t kOffRows = kOffDQ + kDQBytes; // [stage][2][BQ] floats
    static constexpr uint32_t kOffBar = kOffRows + kStages * 2 * kRowBytes;
    static constexpr uint32_t kSmemBytes = kOffBar + sizeof(BwdBarriers) + 1024;
    static constexpr uint32_t kColDP = 128, kColKA = 192, kColDV = 256, kColDK = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t col_s(int b) { return (uint32_t)b * 64; }
};

template <int D>
__device__ void bwd_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                             const CUtensorMap* tm_do, const float* lse2, const float* row_d, uint8_t* smem,
                             BwdBarriers* bars, int head, int k0, int Tq, int Npad) {
    using C = BwdCfg<D>;
    volatile int* abort_flag = &bars->abort;
    const uint64_t pol_keep = policy_evict_last();
    mbar_expect_tx(&bars->kv_full, 2 * C::kKBytes);
    for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(smem + C::kOffK + c * C::kChunkK, tm_k, &bars->kv_full, c * 64, k0, head, pol_keep);
        tma_load_3d(smem + C::kOffV + c * C::kChunkK, tm_v, &bars->kv_full, c * 64, k0, head, pol_keep);
    }
    int issued = 0;
    for (int i = 0; i < Tq; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(&bars->qdo_empty[s], ((i / kStages) - 1) & 1, abort_flag)) break;
        uint64_t* bar = &bars->qdo_full[s];
        mbar_expect_tx(bar, 2 * C::kQBytes + 2 * C::kRowBytes);
        for (int c = 0; c < C::kChunks; ++c) {
            tma_load_3d(smem + C::kOffQ + s * C::kQBytes + c * C::kChunkQ, tm_q, bar, c * 64, i * BQ, head, pol_keep);
            tma_load_3d(smem + C::kOffDO + s * C::kQBytes + c * C::kChunkQ, tm_do, bar, c * 64, i * BQ, head,
                        pol_keep);
        }
        float* rows = reinterpret_cast<float*>(smem + C::kOffRows) + s * 2 * BQ;
        const size_t r0 = (size_t)head * Npad + (size_t)i * BQ;
        bulk_load(rows, lse2 + r0, C::kRowBytes, bar);
        bulk_load(rows + BQ, row_d + r0, C::kRowBytes, bar);
        issued = i + 1;
    }
    drain_wait(&bars->kv_full, 0);
    for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        drain_wait(&bars->qdo_full[i % kStages], (i / kStages) & 1);
}

template <int D>
__device__ void bwd_mma(uint8_t* smem, BwdBarriers* bars, uint32_t tmem, int Tq) {
    using C = BwdCfg<D>;
    volatile int* abort_flag = &bars->abort;
    constexpr uint32_t idS = idesc_bf16_f32(BK, BQ, 0, 0);   // S^T (A from TMEM), dP^T (A K-major); B K-major [q][d]
    constexpr uint32_t idG = idesc_bf16_f32(BK, D, 0, 1);    // dV, dK: A from TMEM, B MN-major [q][d]
    constexpr uint32_t idQ = idesc_bf16_f32(128, BQ, 1, 1);  // dQ^T: A = K^T (MN-major), B = dS^T (MN-major)
    // Operand descriptors are built once; each use only adds a constant byte offset.  K-major views
    // serve S^T and dP^T; MN-major views of the same tiles serve dV, dK and dQ^T.
    const uint64_t kV = sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    const uint64_t kQ = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t kDO = sdesc_sw128(smem_u32(smem + C::kOffDO), 16, 1024);
    const uint64_t mQ = sdesc_sw128(smem_u32(smem + C::kOffQ), C::kChunkQ, 1024);
    const uint64_t mDO = sdesc_sw128(smem_u32(smem + C::kOffDO), C::kChunkQ, 1024);
    const uint64_t mK = sdesc_sw128(smem_u32(smem + C::kOffK), C::kChunkK, 1024);
    const uint64_t mDS = sdesc_sw128(smem_u32(smem + C::kOffDS), C::kDSBytes, 1024);

    // S^T = K Q_i^T with K from tensor memory and Q_i K-major over the head dimension.
    auto s_mma = [&](uint64_t b0, uint32_t dst) {
        const uint32_t d = tmem + dst, a = tmem + C::kColKA;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            mma_ts(d, a + kk * 8, sdesc_advance(b0, (kk / 4) * C::kChunkQ + (kk % 4) * 32), idS, kk > 0);
    };
    // dP^T = V dO_i^T with both tiles K-major over the head dimension.
    auto qk_like = [&](uint64_t a0, uint64_t b0, uint32_t dst) {
        const uint32_t d = tmem + dst;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(d, sdesc_advance(a0, (kk / 4) * C::kChunkK + (kk % 4) * 32),
                   sdesc_advance(b0, (kk / 4) * C::kChunkQ + (kk % 4) * 32), idS, kk > 0);
    };
    // G += A[tmem] B_tile with B MN-major over the query block (dV or dK).
    auto grad = [&](uint32_t a_col, uint64_t b0, uint32_t dst, bool acc) {
        const uint32_t d = tmem + dst, a = tmem + a_col;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
            mma_ts(d, a + kk * 8, sdesc_advance(b0, kk * 16 * 128), idG, (acc || kk > 0) ? 1u : 0u);
    };
    // dQ^T = K^T dS^T over the 128 keys, into the step's buffer.
    auto dq = [&](int buf) {
        const uint32_t d = tmem + C::col_s(buf);
        const uint64_t b0 = sdesc_advance(mDS, buf * C::kDSBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
            mma_ss(d, sdesc_advance(mK, kk * 16 * 128), sdesc_advance(b0, kk * 16 * 128), idQ, kk > 0);
    };

    bool ok = mbar_wait_poll(&bars->kv_full, 0, abort_flag) && mbar_wait_poll(&bars->qdo_full[0], 0, abort_flag) &&
              mbar_wait_poll(&bars->ka_ready, 0, abort_flag);
    if (ok) {
        tc_fence_after();
        s_mma(kQ, C::col_s(0));
        mma_commit(&bars->s_full[0]);
        qk_like(kV, kDO, C::kColDP);
        mma_commit(&bars->dp_full);
    }
    for (int i = 0; ok && i < Tq; ++i) {
        const int s = i % kStages;
        const int s1 = (i + 1) % kStages;
        const int buf = i & 1;
        if (i + 1 < Tq) {
            if (!(ok = mbar_wait_poll(&bars->qdo_full[s1], ((i + 1) / kStages) & 1, abort_flag))) break;
            // Buffer buf^1 last held dQ^T of step i-1: it must have been drained.
            if (i > 0 && !(ok = mbar_wait_poll(&bars->dq_empty, (i - 1) & 1, abort_flag))) break;
            tc_fence_after();
            s_mma(sdesc_advance(kQ, s1 * C::kQBytes), C::col_s(buf ^ 1));
            mma_commit(&bars->s_full[buf ^ 1]);
        }
        if (!(ok = mbar_wait_poll(&bars->p_ready, i & 1, abort_flag))) break;
        tc_fence_after();
        grad(C::col_s(buf), sdesc_advance(mDO, s * C::kQBytes), C::kColDV, i > 0);
        if (!(ok = mbar_wait_poll(&bars->ds_ready, i & 1, abort_flag))) break;
        tc_fence_after();
        grad(C::kColDP, sdesc_advance(mQ, s * C::kQBytes), C::kColDK, i > 0);
        mma_commit(&bars->qdo_empty[s]);
        dq(buf);
        mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free[buf]);
        if (i + 1 < Tq) {
            qk_like(kV, sdesc_advance(kDO, s1 * C::kQBytes), C::kColDP);
            mma_commit(&bars->dp_full);
        }
    }
    if (ok) mma_commit(&bars->dkdv_full);
    mma_commit(&bars->mma_done);
    drain_wait(&bars->mma_done, 0);
}

// Warps 0-3: thread = key row.  Recomputes P^T, forms dS^T, then writes dK and dV.
template <int D>
__device__ void bwd_softgrad(uint8_t* smem, BwdBarriers* bars, uint32_t tmem, __nv_bfloat16* __restrict__ dk,
                             __nv_bfloat16* __restrict__ dv, int head, int k0, int N, int Tq, float scale,
                             float scale_log2) {
    using C = BwdCfg<D>;
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r = warp * 32 + lane;                       // key row in the block, = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const bool valid_key = k0 + r < N;
    uint8_t* ds_tile = smem + C::kOffDS;
    const float* rows_base = reinterpret_cast<const float*>(smem + C::kOffRows);

    // K row r into tensor memory as packed bf16 pairs: the resident A operand of S^T.
    if (!warp_wait(&bars->kv_full, 0, abort_flag)) return;
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c) {
        uint32_t w[32];
        const uint8_t* krow = smem + C::kOffK + c * C::kChunkK + r * 128;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint4 x = *reinterpret_cast<const uint4*>(krow + ((p ^ (r & 7)) << 4));
            w[4 * p] = x.x;
            w[4 * p + 1] = x.y;
            w[4 * p + 2] = x.z;
            w[4 * p + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + C::kColKA + c * 32, w);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars->ka_ready);

    bool ok = true;
    for (int i = 0; i < Tq; ++i) {
        const int s = i % kStages;
        const int buf = i & 1;
        if (!(ok = warp_wait(&bars->s_full[buf], (i >> 1) & 1, abort_flag))) break;
        if (!(ok = warp_wait(&bars->qdo_full[s], (i / kStages) & 1, abort_flag))) break;
        tc_fence_after();
        const float* lse2 = rows_base + s * 2 * BQ;
        const float* drow = lse2 + BQ;
        uint32_t sr[2][32];
        tmem_ld32(tmem + lane_off + C::col_s(buf), sr[0]);
        tmem_ld32(tmem + lane_off + C::col_s(buf) + 32, sr[1]);
        tmem_ld_wait();
        uint64_t p2[BQ / 2];
        {
            const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < BQ / 2; ++c) {
                const int q = (2 * c) / 32, e = (2 * c) % 32;
                const uint64_t x2 = ffma2(f2_pack(__uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1])), sl2,
                                          *reinterpret_cast<const uint64_t*>(lse2 + 2 * c));
                float x0, x1;
                f2_unpack(x2, x0, x1);
                const float p0 = valid_key ? ex2(x0) : 0.f, p1 = valid_key ? ex2(x1) : 0.f;
                p2[c] = f2_pack(p0, p1);
                pk[c] = pack_bf16(p0, p1);
            }
            tmem_st32(tmem + lane_off + C::col_s(buf), pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_ready);

        if (!(ok = warp_wait(&bars->dp_full, i & 1, abort_flag))) break;
        tc_fence_after();
        uint32_t dr[2][32];
        tmem_ld32(tmem + lane_off + C::kColDP, dr[0]);
        tmem_ld32(tmem + lane_off + C::kColDP + 32, dr[1]);
        tmem_ld_wait();
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int q = (2 * c) / 32, e = (2 * c) % 32;
            const uint64_t g2 = fadd2(f2_pack(__uint_as_float(dr[q][e]), __uint_as_float(dr[q][e + 1])),
                                      *reinterpret_cast<const uint64_t*>(drow + 2 * c));
            float d0, d1;
            f2_unpack(fmul2(p2[c], g2), d0, d1);
            pk[c] = pack_bf16(d0, d1);
        }
        tmem_st32(tmem + lane_off + C::kColDP, pk);
        // dS^T row r into the shared tile (128-byte rows, 16-byte chunks XOR-swizzled by r % 8).
        if (i >= 2 && !(ok = warp_wait(&bars->ds_free[buf], ((i >> 1) - 1) & 1, abort_flag))) break;
        uint8_t* row = ds_tile + buf * C::kDSBytes + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(row + ((ch ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
    }
    if (!ok) return;
    if (!warp_wait(&bars->dkdv_full, 0, abort_flag)) return;
    tc_fence_after();
    const size_t base = ((size_t)head * N + k0 + r) * D;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const uint32_t col = g == 0 ? C::kColDV : C::kColDK;
        const float mul = g == 0 ? 1.f : scale;
        __nv_bfloat16* out = g == 0 ? dv : dk;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t x[32];
            tmem_ld32(tmem + lane_off + col + q * 32, x);
            tmem_ld_wait();
            uint32_t pk2[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
                pk2[c] = pack_bf16(__uint_as_float(x[2 * c]) * mul, __uint_as_float(x[2 * c + 1]) * mul);
            if (valid_key) {
                uint4* dst = reinterpret_cast<uint4*>(out + base + q * 32);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    dst[c] = make_uint4(pk2[4 * c], pk2[4 * c + 1], pk2[4 * c + 2], pk2[4 * c + 3]);
            }
        }
    }
}

// Warps 4-7: thread = head-dimension index c.  Moves dQ_i^T out of tensor memory and adds it into the
// fp32 accumulator [head][N][D] with one bulk reduce-add per query block.
template <int D>
__device__ void bwd_dq_drain(uint8_t* smem, BwdBarriers* bars, uint32_t tmem, float* __restrict__ dq_acc, int head,
                             int N, int Tq) {
    using C = BwdCfg<D>;
    volatile int* abort_flag = &bars->abort;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;
    const int c = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool active = quarter * 32 < D;
    float* stage = reinterpret_cast<float*>(smem + C::kOffDQ);
    const bool leader = threadIdx.x == 128;

    // Every warp reaches both named barriers in every step, even after a wait gave up, so that no
    // warp of this group can be left waiting on the others.
    bool failed = false;
    for (int i = 0; i < Tq; ++i) {
        if (!failed && !warp_wait(&bars->dq_full, i & 1, abort_flag)) failed = true;
        uint32_t x[2][32];
        if (!failed) {
            tc_fence_after();
            if (active) {
                tmem_ld32(tmem + lane_off + C::col_s(i & 1), x[0]);
                tmem_ld32(tmem + lane_off + C::col_s(i & 1) + 32, x[1]);
                tmem_ld_wait();
            }
            tc_fence_before();
            mbar_arrive(&bars->dq_empty);
        }
        if (leader) bulk_wait_group_read<0>();
        named_bar_sync(1, 128);
        if (!failed && active) {
#pragma unroll
            for (int q = 0; q < BQ; ++q) stage[q * D + c] = __uint_as_float(x[q / 32][q % 32]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader && !failed && !*abort_flag) {
            const int rows = min(BQ, N - i * BQ);
            bulk_reduce_add_f32(dq_acc + ((size_t)head * N + (size_t)i * BQ) * D, stage, (uint32_t)(rows * D * 4));
            bulk_commit_group();
        }
    }
    if (leader) bulk_wait_group<0>();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const float* __restrict__ lse2, const float* __restrict__ row_d, float* __restrict__ dq_acc,
              __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int N, int Npad,
              int blocks_per_head, float scale, float scale_log2, long long wait_budget) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    BwdBarriers* bars = reinterpret_cast<BwdBarriers*>(smem + C::kOffBar);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // 1-D grid, head-major: the CTAs of one head walk the same Q/dO blocks, which stay in L2.
    const int head = blockIdx.x / blocks_per_head;
    const int k0 = (blockIdx.x % blocks_per_head) * BK;
    const int Tq = Npad / BQ;

    if (threadIdx.x == 0) {
        s_wait_budget = wait_budget;
        mbar_init(&bars->kv_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->qdo_full[s], 1);
            mbar_init(&bars->qdo_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->s_full[b], 1);
            mbar_init(&bars->ds_free[b], 1);
        }
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->p_ready, 128);
        mbar_init(&bars->ds_ready, 128);
        mbar_init(&bars->dq_full, 1);
        mbar_init(&bars->dq_empty, 128);
        mbar_init(&bars->dkdv_full, 1);
        mbar_init(&bars->ka_ready, 128);
        mbar_init(&bars->mma_done, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if constexpr (C::kZeroBytes > 0) {
        uint4* z = reinterpret_cast<uint4*>(smem + C::kOffZero);
        for (uint32_t idx = threadIdx.x; idx < C::kZeroBytes / 16; idx += kThreads) z[idx] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == kTmaWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == kTmaWarp) {
        if (lane == 0) bwd_producer<D>(&tm_q, &tm_k, &tm_v, &tm_do, lse2, row_d, smem, bars, head, k0, Tq, Npad);
    } else if (warp == kMmaWarp) {
        if (lane == 0) bwd_mma<D>(smem, bars, tmem, Tq);
    } else if (warp < 4) {
        bwd_softgrad<D>(smem, bars, tmem, dk, dv, head, k0, N, Tq, scale, scale_log2);
    } else {
        bwd_dq_drain<D>(smem, bars, tmem, dq_acc, head, N, Tq);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0 && bars->abort) atomicCAS(&g_bwd_status, 0, (int)FA_ERR_TIMEOUT);
}

// -D_i = -(dO_i . O_i) and -LSE2_i = -LSE_i log2(e) into [head][Npad] arrays (pad rows: 0 and -inf);
// zeroes the fp32 dQ accumulator.  D/8 threads share a row (16-byte loads of O and dO), each warp takes
// 2 * 32 / (D/8) rows per pass, so enough bytes are in flight to stream at HBM speed.
template <int D>
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ lse, float* __restrict__ row_d, float* __restrict__ lse2,
                                float* __restrict__ dq_acc, int N, int Npad, int64_t heads) {
    constexpr int kTpr = D / 8;          // threads per row
    constexpr int kRpw = 32 / kTpr;      // rows per warp and pass
    const int lane = threadIdx.x & 31;
    const int sub = lane / kTpr, part = lane % kTpr;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t warp_id = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t rows = heads * Npad;
    for (int64_t base = warp_id * 2 * kRpw; base < rows; base += nwarps * 2 * kRpw) {
        float acc[2];
        int64_t w[2];
        bool valid[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            w[u] = base + u * kRpw + sub;
            const int64_t h = w[u] / Npad;
            const int r = (int)(w[u] - h * Npad);
            valid[u] = w[u] < rows && r < N;
            acc[u] = 0.f;
            if (valid[u]) {
                const size_t off = ((size_t)h * N + r) * D + part * 8;
                const uint4 a = *reinterpret_cast<const uint4*>(o + off);
                const uint4 g = *reinterpret_cast<const uint4*>(dout + off);
                const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
                const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 fa = __bfloat1622float2(a2[t]), fg = __bfloat1622float2(g2[t]);
                    acc[u] = fmaf(fa.x, fg.x, fmaf(fa.y, fg.y, acc[u]));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int off = kTpr / 2; off; off >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], off);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (part != 0 || w[u] >= rows) continue;
            const int64_t h = w[u] / Npad;
            const int r = (int)(w[u] - h * Npad);
            row_d[w[u]] = valid[u] ? -acc[u] : 0.f;
            lse2[w[u]] = valid[u] ? -lse[(size_t)h * N + r] * 1.4426950408889634f : -INFINITY;
        }
    }
    const int64_t n4 = heads * (int64_t)N * D / 4;
    float4* z = reinterpret_cast<float4*>(dq_acc);
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n4; idx += (int64_t)gridDim.x * blockDim.x)
        z[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator), four elements per thread, grid-stride.
__global__ void bwd_dq_convert_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, float scale,
                                      int64_t n4) {
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n4;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(dq_acc)[idx];
        uint2 out;
        out.x = pack_bf16(a.x * scale, a.y * scale);
        out.y = pack_bf16(a.z * scale, a.w * scale);
        reinterpret_cast<uint2*>(dq)[idx] = out;
    }
}

template <int D>
cudaError_t launch(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, const Shape& s, float scale, void* workspace, cudaStream_t st) {
    using C = BwdCfg<D>;
    const BwdWorkspace w = bwd_workspace_layout(s);
    char* ws = (char*)workspace;
    float* dq_acc = (float*)(ws + w.dq_acc);
    float* row_d = (float*)(ws + w.row_d);
    float* lse2 = (float*)(ws + w.lse2);
    const int Npad = bwd_padded_rows(s.N);
    const int blocks = device_sm_count() * 4;
    bwd_prep_kernel<D><<<blocks, 256, 0, st>>>((const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, lse, row_d,
                                               lse2, dq_acc, s.N, Npad, s.heads());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap tq, tk, tv, tdo;
    if ((e = make_tmap_bf16_3d(&tq, q, s.d, s.N, s.heads(), BQ)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tdo, dout, s.d, s.N, s.heads(), BQ)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tk, k, s.d, s.N, s.heads(), BK)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tv, v, s.d, s.N, s.heads(), BK)) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int bph = (s.N + BK - 1) / BK;
    if ((long long)bph * s.heads() > INT32_MAX) return cudaErrorInvalidConfiguration;
    const unsigned grid = (unsigned)(bph * s.heads());
    bwd_tc_kernel<D><<<grid, kThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, lse2, row_d, dq_acc,
                                                            (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, s.N, Npad, bph, scale,
                                                            scale * 1.4426950408889634f, wait_policy().budget_cycles);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_dq_convert_kernel<<<blocks, 256, 0, st>>>(dq_acc, (__nv_bfloat16*)dq, scale, s.heads() * (int64_t)s.N * D / 4);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, const Shape& s, float scale,
                          void* workspace, cudaStream_t st) {
    return s.d == 128 ? launch<128>(q, k, v, o, dout, lse, dq, dk, dv, s, scale, workspace, st)
                      : launch<64>(q, k, v, o, dout, lse, dq, dk, dv, s, scale, workspace, st);
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
