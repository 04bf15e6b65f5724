// bf16 attention backward on the sm_103a tensor cores (tcgen05 + TMA + tensor memory).
//
// The pages keep P out of device memory in the backward pass too: it is recomputed from Q, K and the
// saved statistic ("账房先生的奔命：Flash Attention 与内存 I/O 革命" §七 重计算).  The gradient formulas
// themselves are the textbook derivative of O = softmax(scale Q K^T) V:
//     P = exp(scale S - LSE),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D_i = dO_i . O_i,
//     dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels per call:
//   bwd_prep_kernel   -D_i and -LSE_i * log2(e) per query row (padded to a multiple of 128 rows per head;
//                     pad rows get 0 and -inf so they contribute nothing), and zeroes the fp32 dQ
//                     accumulator.  Negated so that the main kernel applies them with packed-pair adds.
//   bwd_tc_kernel     one CTA per (head, block of 128 keys).  K_j, V_j stay in shared memory; the CTA
//                     walks every block of 128 queries i:
//                         S^T  = K_j Q_i^T              fp32 in tensor memory
//                         dP^T = V_j dO_i^T
//                         P^T  = exp2(S^T scale log2e - LSE2_i)    thread = key row; packed fp32
//                                                       pairs (f32x2) for the element-wise work
//                         dS^T = P^T o (dP^T - D_i)
//                         dV_j += P^T dO_i              P^T as bf16 from tensor memory
//                         dK_j += dS^T Q_i              dS^T as bf16 from tensor memory
//                         dQ_i = dS K_j                 dS as bf16 from shared memory (the slot's dS^T
//                                                       read MN-major), queries as tensor-memory lanes
//                     and adds dQ_i into the fp32 accumulator with tensor reduce-add copies.
//   bwd_dq_convert    dQ = bf16(scale * accumulator).
// The main and conversion kernels are programmatic dependents of the kernel before them: the prep kernel
// releases the main kernel at its start, whose TMA thread loads K and V and only then waits for the prep
// kernel's results; the conversion kernel launches as the main kernel's CTAs finish and waits for them.  The
// backward measured 0.8 % faster at N = 8192 d = 128, 2.6 % at N = 2048 and 2.3 % at B=4 H=16 N=2048 d = 64.
//
// At d = 128 every product is 128 x 128 x 128 (M = 128 keys or queries, N = 128 queries or head
// dimensions): N = 128 is the narrowest tcgen05 shape that runs at the full rate, which 64-query steps
// (three of five products at N = 64) did not reach.  Tensor memory then holds exactly S^T, dP^T, dV and
// dK (4 x 128 columns at d = 128), with dQ reusing the columns of dP^T; at d = 64 dQ has 64 columns of its
// own.  The MMAs of step i run in the order dV(i), S^T(i+1), dK(i), dQ(i), dP^T(i+1): the next S^T goes
// right behind dV (its columns held P^T, which dV has just read), so forming P(i+1) overlaps dK and dQ on
// the tensor core.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two warpgroups that own the same 128 key rows
// (tensor-memory lanes) and split each step's queries, 64 each, for P^T and dS^T; for dQ the lanes are
// the step's 128 queries and the warpgroups split the head dimension, d / 2 columns each, which they move
// out of tensor memory (thread = query row) and stage.  At the end warps 0-3 write dV and warps 4-7 dK.
// Warp 8 issues the TMA loads and every reduce-add, warp 9 allocates tensor memory and issues the MMAs.
//
// Shared memory (d = 128: 226 KB): K and V resident, two Q stages, and two slots that each hold a step's dO
// tile, then its dS^T (once dV has read dO), then the first warpgroup's fp32 dQ columns (once dQ has read
// dS^T) as d / 64 [128][32] blocks, 128-byte swizzled and written with 16-byte stores; the TMA thread adds
// each block into the accumulator with one tensor reduce and loads the dO tile of step i + 2 there by
// 64-column chunks, each once the block under it has been read (one barrier for the whole tile).  The
// second warpgroup's blocks have a buffer of their own, which the TMA thread adds only after it has issued
// that dO load: with the second half's reduce issued first (from that warpgroup's own leader thread) the dO
// tile queued behind it in the copy unit, which cost 11 % of the backward at d = 128.  At the end the K and V
// tiles' space takes the bf16 rows of dK and dV, so that they leave in whole-row stores.  The kernel has no static shared memory, so its dynamic region starts aligned and
// needs no slack.
//
// (An earlier layout formed dQ^T = K^T dS^T at d = 128, thread = head-dimension index, each warp staging a
// [64][32] stripe with scalar stores: once the tensor-memory loads were widened to 64 columns, the present
// layout measured 0.6-0.7 % faster, and it serves both head sizes.)

#include <cuda_bf16.h>
#include <math.h>
#include <type_traits>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

__device__ int g_bwd_status;

constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 128;  // queries per step
constexpr int HQ = 64;   // queries per warpgroup half of a step
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;

struct BwdBarriers {
    uint64_t kv_full;
    uint64_t q_full[2];            // Q tile + LSE2 and -D rows of a step
    uint64_t q_empty[2];           // dK of that step has read the Q tile
    uint64_t do_full[2];           // a step's dO tile is in its slot
    uint64_t dv_done[2];           // dV of that step has read dO: the slot takes dS^T
    uint64_t staged_a[2];          // the first warpgroup's dQ columns are staged in the slot
    uint64_t s_full;
    uint64_t dp_full;
    uint64_t p_ready;              // both halves' P^T of a step are in tensor memory (256 arrivals)
    uint64_t ds_ready[2];          // a half's dS^T is in tensor memory (d = 128: and in the step's slot)
    uint64_t ds_smem;              // d = 64: both halves' dS^T are in the step's slot (what dQ reads)
    uint64_t dq_full;
    uint64_t dq_empty;
    uint64_t staged_b;             // the second warpgroup's dQ columns are in their staging buffer
    uint64_t stage_b_free;         // ... and their reduce has read them (arrived by the TMA thread)
    uint64_t dkdv_full;
    uint64_t mma_done;
    uint32_t tmem_base;
    WaitCtl wait;
};

// Shared memory.  K and V stay resident; Q has two stages.  Each step's dO tile lives in one of two
// slots, and the slot is reused within the step: once dV has read dO it takes the step's dS^T (the A
// operand of dQ), and once dQ has read that it takes the first warpgroup's fp32 dQ columns, which the
// TMA thread adds into the accumulator before loading the dO tile of step i + 2 there.  The second
// warpgroup's columns have a buffer of their own.
template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kChunkK = BK * 128;          // one 64-column chunk of a K or V tile
    static constexpr uint32_t kChunkQ = BQ * 128;          // one 64-column chunk of a Q or dO tile
    static constexpr uint32_t kKBytes = BK * D * 2;
    static constexpr uint32_t kQBytes = BQ * D * 2;
    static constexpr uint32_t kDSChunk = BK * 128;         // dS^T of one half: 128 key rows x 64 queries
    // dQ = dS K is formed with the step's queries as tensor-memory lanes (M = 128, N = d); the two
    // warpgroups split its d columns, and each stages [128 queries][d / 2] fp32.
    static constexpr uint32_t kHalfDQBytes = BQ * (D / 2) * 4;   // fp32 dQ of one warpgroup (16 or 32 KB)
    static constexpr uint32_t kSlotBytes = 2 * kDSChunk;   // holds a dO tile, dS^T or a half's dQ rows
    static constexpr uint32_t kOffK = 0;
    static constexpr uint32_t kOffV = kOffK + kKBytes;
    static constexpr uint32_t kOffQ = kOffV + kKBytes;
    static constexpr uint32_t kOffSlot = kOffQ + 2 * kQBytes;
    static constexpr uint32_t kOffStageB = kOffSlot + 2 * kSlotBytes;   // the second half's dQ rows
    // A warpgroup's dQ columns are staged as [BQ][32] fp32 blocks (128-byte swizzled, written by 16-byte
    // stores), d / 64 of them, each added into the accumulator by one tensor reduce.
    static constexpr int kDqBlocks = D / 64;
    // d = 64: dS ready for dK (tensor memory) is signalled before the shared-memory copy for dQ, which
    // waits for dV to have read the slot; a barrier of its own covers that copy.  At d = 128 one signal
    // after both measured as fast (and 0.7 % faster at N = 32768).
    static constexpr bool kEarlyDsReady = D == 64;
    static constexpr uint32_t kDqBlockBytes = BQ * 32 * 4;
    static constexpr uint32_t kRowBytes = BQ * 4;          // LSE2 or -D of one query block
    static constexpr uint32_t kOffRows = kOffStageB + kHalfDQBytes;    // [q stage][LSE2 | -D][BQ] floats
    static constexpr uint32_t kOffBar = kOffRows + 2 * 2 * kRowBytes;
    static constexpr uint32_t kSmemNeed = kOffBar + sizeof(BwdBarriers);
    // Room to align the region to 1024 bytes if the dynamic shared memory does not start aligned (it
    // does when the kernel has no static shared memory, which is the case here).
    static constexpr uint32_t kAlignSlack = kSmemNeed + 1024 <= 232448 ? 1024 : 232448 - kSmemNeed;
    static constexpr uint32_t kSmemBytes = kSmemNeed + kAlignSlack;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    // dQ reuses the columns of dP^T at d = 128 (all 512 are taken); at d = 64 it has spare columns of its
    // own, so the next dP^T need not wait for it to be moved out.
    static constexpr bool kOwnDQ = D == 64;
    static constexpr uint32_t kColDQ = kOwnDQ ? 256 + 2 * D : kColDP;
    static_assert(kColDQ + D <= 512, "tensor memory columns");
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kQBytes <= kSlotBytes && kHalfDQBytes <= kSlotBytes, "slot contents");
    static_assert(kDqBlocks * kDqBlockBytes == kHalfDQBytes && kDqBlocks == kChunks, "one block per dO chunk");
    static_assert(kSmemNeed <= 232448, "shared memory per CTA");
};

// Query block visited at step i by a CTA whose walk starts at block `rot`.
__device__ __forceinline__ int qblock(int i, int rot, int Tq) {
    const int b = i + rot % Tq;
    return b < Tq ? b : b - Tq;
}

template <int D>
__device__ void bwd_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                             const CUtensorMap* tm_do, const CUtensorMap* tm_dq, const float* lse2, const float* row_d,
                             float* __restrict__ dq_acc, uint8_t* smem, BwdBarriers* bars, int head, int k0, int N,
                             int Tq, int Npad, int rot, int starve) {
    using C = BwdCfg<D>;
    WaitCtl* wc = &bars->wait;
    const uint64_t pol_keep = policy_evict_last();
    mbar_expect_tx(&bars->kv_full, 2 * C::kKBytes);
    for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(smem + C::kOffK + c * C::kChunkK, tm_k, &bars->kv_full, c * 64, k0, head, pol_keep);
        tma_load_3d(smem + C::kOffV + c * C::kChunkK, tm_v, &bars->kv_full, c * 64, k0, head, pol_keep);
    }
    // The kernel may start while the prep kernel is still running: K and V are inputs of the call, but the
    // row terms and the zeroed accumulator are the prep kernel's, and only this thread touches them.
    griddep_wait();
    // The first warpgroup's dQ columns of step j end up in slot j % 2 as d / 64 [BQ][32] blocks.  This
    // thread adds each block into the accumulator once the warpgroup has staged them (rows past N are
    // clipped by the tensor map) and reloads the slot once the reduces have read it, so it owns the slot's
    // whole cycle.  Block c lies under chunk c of the dO tile that reloads the slot and is its own bulk
    // group, so that chunk c can load as soon as that block has been read.
    auto reduce_first_half = [&](int j) -> bool {
        const int t = j & 1;
        const int q0 = qblock(j, rot, Tq) * BQ;
        if (!mbar_wait(&bars->staged_a[t], (j >> 1) & 1, wc)) return false;
        for (int w = 0; w < C::kDqBlocks; ++w) {
            tma_reduce_add_3d(tm_dq, smem + C::kOffSlot + t * C::kSlotBytes + w * C::kDqBlockBytes, 32 * w, q0, head);
            bulk_commit_group();
        }
        return true;
    };
    // The second warpgroup's dQ columns of step j, from their own buffer, added after the dO loads so that
    // those do not queue behind them; the buffer is handed back once the reduce has read it.
    auto reduce_second_half = [&](int j) -> bool {
        if (!mbar_wait(&bars->staged_b, j & 1, wc)) return false;
        const int q0 = qblock(j, rot, Tq) * BQ;
        for (int b = 0; b < C::kDqBlocks; ++b)
            tma_reduce_add_3d(tm_dq, smem + C::kOffStageB + b * C::kDqBlockBytes, D / 2 + 32 * b, q0, head);
        bulk_commit_group();
        return true;
    };
    auto free_stage_b = [&]() {
        bulk_wait_group_read<0>();
        mbar_arrive(&bars->stage_b_free);
    };
    int q_issued = 0, do_issued = 0;
    bool ok = true;
    for (int i = 0; i < Tq && ok; ++i) {
        const int s = i & 1;
        const int qb = qblock(i, rot, Tq);
        if (i >= 2 && !(ok = mbar_wait(&bars->q_empty[s], ((i >> 1) - 1) & 1, wc))) break;
        // starve != 0 withholds the Q loads so that the first waits on them run out: the failure path of
        // the bounded waits, exercised by the tests with a short budget.
        if (!starve) {
            uint64_t* bar = &bars->q_full[s];
            mbar_expect_tx(bar, C::kQBytes + 2 * C::kRowBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(smem + C::kOffQ + s * C::kQBytes + c * C::kChunkQ, tm_q, bar, c * 64, qb * BQ, head,
                            pol_keep);
            float* rows = reinterpret_cast<float*>(smem + C::kOffRows) + s * 2 * BQ;
            const size_t r0 = (size_t)head * Npad + (size_t)qb * BQ;
            bulk_load(rows, lse2 + r0, C::kRowBytes, bar);
            bulk_load(rows + BQ, row_d + r0, C::kRowBytes, bar);
            q_issued = i + 1;
        }

        if (i >= 2) {
            if (i >= 3) free_stage_b();
            if (!(ok = reduce_first_half(i - 2))) break;
        }
        for (int c = 0; c < C::kChunks; ++c) {
            // Chunk c overwrites the block of reduce group c (the groups are read in order).
            if (i >= 2) {
                if (C::kChunks == 2 && c == 0) bulk_wait_group_read<1>();
                else bulk_wait_group_read<0>();
            }
            if (c == 0) mbar_expect_tx(&bars->do_full[s], C::kQBytes);
            tma_load_3d(smem + C::kOffSlot + s * C::kSlotBytes + c * C::kChunkQ, tm_do, &bars->do_full[s], c * 64,
                        qb * BQ, head, pol_keep);
        }
        do_issued = i + 1;
        if (i >= 2 && !(ok = reduce_second_half(i - 2))) break;
    }
    for (int j = (Tq > 2 ? Tq - 2 : 0); ok && j < Tq; ++j) {
        if (j >= 1) free_stage_b();
        ok = reduce_first_half(j) && reduce_second_half(j);
    }
    bulk_wait_group<0>();
    // Copies still in flight must land before the CTA can exit.
    drain_wait(&bars->kv_full, 0, wc);
    for (int i = (q_issued > 2 ? q_issued - 2 : 0); i < q_issued; ++i) drain_wait(&bars->q_full[i & 1], (i >> 1) & 1, wc);
    for (int i = (do_issued > 2 ? do_issued - 2 : 0); i < do_issued; ++i)
        drain_wait(&bars->do_full[i & 1], (i >> 1) & 1, wc);
}

// MMA order of step i: dV(i), S^T(i+1), dK(i), dQ(i), dP^T(i+1).  S^T of the next step goes right
// behind dV (its columns held P^T, which dV has just read), so the softmax warps can form P(i+1) while
// the tensor core works on dK and dQ; at d = 128 dP^T(i+1) waits until dQ(i) has left its columns.
template <int D>
__device__ void bwd_mma(uint8_t* smem, BwdBarriers* bars, uint32_t tmem, int Tq) {
    using C = BwdCfg<D>;
    WaitCtl* wc = &bars->wait;
    constexpr uint32_t idS = idesc_bf16_f32(BK, BQ, 0, 0);   // S^T, dP^T: A and B K-major over the head dimension
    constexpr uint32_t idG = idesc_bf16_f32(BK, D, 0, 1);    // dV, dK: A from TMEM, B MN-major [q][d]
    // dQ: A = dS read MN-major from the slot's dS^T, B = K (MN-major over d).
    constexpr uint32_t idQ = idesc_bf16_f32(BQ, D, 1, 1);
    // Operand descriptors are built once; each use only adds a constant byte offset.  K-major views
    // serve S^T and dP^T; MN-major views of the same tiles serve dV, dK and dQ.
    const uint64_t kK = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t kV = sdesc_sw128(smem_u32(smem + C::kOffV), 16, 1024);
    const uint64_t kQ = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t kDO = sdesc_sw128(smem_u32(smem + C::kOffSlot), 16, 1024);
    const uint64_t mQ = sdesc_sw128(smem_u32(smem + C::kOffQ), C::kChunkQ, 1024);
    const uint64_t mDO = sdesc_sw128(smem_u32(smem + C::kOffSlot), C::kChunkQ, 1024);
    const uint64_t mK = sdesc_sw128(smem_u32(smem + C::kOffK), C::kChunkK, 1024);
    const uint64_t mDS = sdesc_sw128(smem_u32(smem + C::kOffSlot), C::kDSChunk, 1024);

    // X^T = A B^T over the head dimension, both tiles K-major (S^T = K Q^T, dP^T = V dO^T).
    auto qk_like = [&](uint64_t a0, uint64_t b0, uint32_t dst) {
        const uint32_t d = tmem + dst;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(d, sdesc_advance(a0, (kk / 4) * C::kChunkK + (kk % 4) * 32),
                   sdesc_advance(b0, (kk / 4) * C::kChunkQ + (kk % 4) * 32), idS, kk > 0);
    };
    // G += A[tmem] B_tile over one half's 64 queries, B MN-major over the head dimension (dV or dK).
    auto grad = [&](uint32_t a_col, uint64_t b0, int half, uint32_t dst, bool acc) {
        const uint32_t d = tmem + dst, a = tmem + a_col + half * HQ;
#pragma unroll
        for (int kk = 0; kk < HQ / 16; ++kk)
            mma_ts(d, a + kk * 8, sdesc_advance(b0, (half * (HQ / 16) + kk) * 16 * 128), idG,
                   (acc || kk > 0) ? 1u : 0u);
    };
    // dQ = dS K over the 128 keys: at d = 128 into the columns of dP^T (free once dK used dS^T), at d = 64
    // into columns of its own.
    auto dq = [&](uint64_t ds0) {
        const uint32_t d = tmem + C::kColDQ;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
            mma_ss(d, sdesc_advance(ds0, kk * 16 * 128), sdesc_advance(mK, kk * 16 * 128), idQ, kk > 0);
    };

    bool ok = mbar_wait_poll(&bars->kv_full, 0, wc) && mbar_wait_poll(&bars->q_full[0], 0, wc);
    if (ok) {
        tc_fence_after();
        qk_like(kK, kQ, C::kColS);
        mma_commit(&bars->s_full);
        if ((ok = mbar_wait_poll(&bars->do_full[0], 0, wc))) {
            tc_fence_after();
            qk_like(kV, kDO, C::kColDP);
            mma_commit(&bars->dp_full);
        }
    }
    for (int i = 0; ok && i < Tq; ++i) {
        const int s = i & 1, s1 = s ^ 1;
        const uint64_t bdo = sdesc_advance(mDO, s * C::kSlotBytes), bq = sdesc_advance(mQ, s * C::kQBytes);
        // dV waits for both halves' P^T at once: one barrier test fewer per step for this thread, whose
        // every test costs the tensor core idle cycles, measured faster than starting on the first half
        // (1.3 % at d = 128, N = 8192; 2.4 % at N = 32768; 0.8 % at d = 64, N = 2048).
        if (!(ok = mbar_wait_poll(&bars->p_ready, i & 1, wc))) break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h) grad(C::kColS, bdo, h, C::kColDV, i > 0 || h > 0);
        mma_commit(&bars->dv_done[s]);
        if (i + 1 < Tq) {
            if (!(ok = mbar_wait_poll(&bars->q_full[s1], ((i + 1) >> 1) & 1, wc))) break;
            tc_fence_after();
            qk_like(kK, sdesc_advance(kQ, s1 * C::kQBytes), C::kColS);
            mma_commit(&bars->s_full);
        }
        for (int h = 0; h < 2; ++h) {
            if (!(ok = mbar_wait_poll(&bars->ds_ready[h], i & 1, wc))) break;
            tc_fence_after();
            grad(C::kColDP, bq, h, C::kColDK, i > 0 || h > 0);
        }
        if (!ok) break;
        mma_commit(&bars->q_empty[s]);
        // dQ reads both halves' dS^T from the slot (at d = 128 ds_ready already covered it).
        if constexpr (C::kEarlyDsReady) {
            if (!(ok = mbar_wait_poll(&bars->ds_smem, i & 1, wc))) break;
            tc_fence_after();
        }
        // At d = 64 dQ has its own columns, which dQ of step i-1 must have left: each warpgroup arrives on
        // ds_smem(i) only after it has moved dQ(i-1) out (program order, behind that drain's tcgen05 fence),
        // so the wait on ds_smem above covers it and this thread saves a barrier test per step.
        static_assert(!C::kOwnDQ || C::kEarlyDsReady, "dQ's own columns are freed through ds_smem");
        dq(sdesc_advance(mDS, s * C::kSlotBytes));
        mma_commit(&bars->dq_full);
        if (i + 1 < Tq) {
            // One test for the whole dO tile: testing its two 64-column chunks separately, so that dP^T
            // could start on the first, measured 1.1-1.5 % slower at d = 128.
            if (!(ok = mbar_wait_poll(&bars->do_full[s1], ((i + 1) >> 1) & 1, wc))) break;
            // At d = 128 the columns of dP^T hold dQ of step i until it has been moved out.
            if (!C::kOwnDQ && !(ok = mbar_wait_poll(&bars->dq_empty, i & 1, wc))) break;
            tc_fence_after();
            qk_like(kV, sdesc_advance(kDO, s1 * C::kSlotBytes), C::kColDP);
            mma_commit(&bars->dp_full);
        }
    }
    if (ok) mma_commit(&bars->dkdv_full);
    mma_commit(&bars->mma_done);
    drain_wait(&bars->mma_done, 0, wc);
}

// Warps 0-7 write dV (0-3) and dK (4-7, scaled) once every MMA has completed.  The K and V tiles are free
// by then: each thread converts its key row to bf16 and puts it in the V (dV) or K (dK) tile's space,
// 16-byte chunks XOR-swizzled by the row; then each warp copies its own 32 rows out, a warp's 16-byte
// stores covering whole rows (two at d = 128, four at d = 64), where one row per thread would touch 32
// rows of memory per store.  A call rather than inlined code: inlined, its registers shaped the step loop
// of bwd_softgrad (this copy inlined made the d = 64 backward 2.4 % slower; called, it is 1.5-1.8 % faster
// than the one-row-per-thread stores at every N, and at d = 128 0.3 % faster at N = 8192, 1.8 % at 2048).
template <int D>
__device__ __noinline__ void bwd_write_dkdv(uint8_t* smem, uint32_t tmem, __nv_bfloat16* __restrict__ dk,
                                                   __nv_bfloat16* __restrict__ dv, int head, int k0, int N, float scale) {
    using C = BwdCfg<D>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = warp / 4, quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t col = half == 0 ? C::kColDV : C::kColDK;
    const float mul = half == 0 ? 1.f : scale;
    __nv_bfloat16* out = half == 0 ? dv : dk;
    uint8_t* tile = smem + (half == 0 ? C::kOffV : C::kOffK);
    constexpr int kRowChunks = D / 8;                 // 16-byte chunks in a bf16 row
    constexpr int kRowsPerStore = 32 / kRowChunks;    // rows one warp store covers
#pragma unroll
    for (int q2 = 0; q2 < D / 64; ++q2) {
        uint32_t y[2][32];
        tmem_ld64(tmem + lane_off + col + q2 * 64, y);
        tmem_ld_wait();
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int c = q2 * 8 + b * 4 + c4;
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16(__uint_as_float(y[b][8 * c4 + 2 * e]) * mul,
                                     __uint_as_float(y[b][8 * c4 + 2 * e + 1]) * mul);
                *reinterpret_cast<uint4*>(tile + r * (D * 2) + ((c ^ (r & (kRowChunks - 1))) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
    }
    __syncwarp();
    const int sub = lane / kRowChunks, c = lane % kRowChunks;
#pragma unroll
    for (int it = 0; it < 32 / kRowsPerStore; ++it) {
        const int rr = quarter * 32 + it * kRowsPerStore + sub;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + rr * (D * 2) + ((c ^ (rr & (kRowChunks - 1))) << 4));
        if (k0 + rr < N)
            *reinterpret_cast<uint4*>(out + ((size_t)head * N + k0 + rr) * D + c * 8) = v;
    }
}

// Warps 0-7.  Thread = key row r of the CTA (tensor-memory lane) in the softmax-gradient part, where
// `half` selects queries [64 half, 64 half + 64) of each step, and query row r of the step in the dQ
// part, where `half` selects head-dimension columns [d/2 half, d/2 half + d/2).
// Order of step i: dS(i), P(i+1), then dQ(i) out of tensor memory (P(0) comes first).
template <int D>
__device__ void bwd_softgrad(uint8_t* smem, BwdBarriers* bars, uint32_t tmem, float* __restrict__ dq_acc,
                             const CUtensorMap* tm_dq, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                             int head, int k0, int N, int Tq, int rot, float scale, float scale_log2) {
    using C = BwdCfg<D>;
    WaitCtl* wc = &bars->wait;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = warp / 4, quarter = warp % 4;
    const int r = quarter * 32 + lane;                    // key row in the block, = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool valid_key = k0 + r < N;
    const bool all_keys_valid = k0 + BK <= N;   // CTA-uniform: only the head's last key block masks
    const float* rows_base = reinterpret_cast<const float*>(smem + C::kOffRows);
    const uint64_t sl2 = f2_pack(scale_log2, scale_log2);

    // P(j) for this half: P^T as bf16 pairs over the first 32 of the half's 64 columns of S^T; the fp32
    // values stay in p2 for dS(j).
    uint64_t p2[HQ / 2];
    auto form_p = [&](int j) -> bool {
        if (!warp_wait(&bars->s_full, j & 1, wc)) return false;
        if (!warp_wait(&bars->q_full[j & 1], (j >> 1) & 1, wc)) return false;
        tc_fence_after();
        const float* lse2 = rows_base + (j & 1) * 2 * BQ + half * HQ;
        uint32_t sr[2][32];
        tmem_ld64(tmem + lane_off + C::kColS + half * HQ, sr);
        tmem_ld_wait();
        uint32_t pk[32];
        // The row terms come in 16-byte loads (two query pairs each), and key rows past N are masked only in
        // the head's last key block: with both the backward measured 2 % faster at d = 128 and 4-6 % at d = 64.
        const float4* lse4 = reinterpret_cast<const float4*>(lse2);
        auto body = [&](auto all_valid) {
#pragma unroll
            for (int c2 = 0; c2 < HQ / 4; ++c2) {
                const float4 l = lse4[c2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int c = 2 * c2 + u;
                    const int q = (2 * c) / 32, e = (2 * c) % 32;
                    const uint64_t x2 = ffma2(f2_pack(__uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1])), sl2,
                                              u == 0 ? f2_pack(l.x, l.y) : f2_pack(l.z, l.w));
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    float p0 = ex2(x0), p1 = ex2(x1);
                    if constexpr (!decltype(all_valid)::value) {
                        p0 = valid_key ? p0 : 0.f;
                        p1 = valid_key ? p1 : 0.f;
                    }
                    p2[c] = f2_pack(p0, p1);
                    pk[c] = pack_bf16(p0, p1);
                }
            }
        };
        if (all_keys_valid) body(std::true_type{});
        else body(std::false_type{});
        tmem_st32(tmem + lane_off + C::kColS + half * HQ, pk);
        tmem_st_wait();
        tc_fence_before();
        // A warpgroup cannot arrive for step j + 1 before the phase of step j completes: P(j + 1) needs
        // S^T(j + 1), which the MMA thread issues only after that phase.
        mbar_arrive(&bars->p_ready);
        return true;
    };

    bool ok = Tq > 0 && form_p(0);
    for (int i = 0; ok && i < Tq; ++i) {
        const int s = i & 1;
        // dS(i) = P(i) o (dP(i) - D).
        if (!(ok = warp_wait(&bars->dp_full, i & 1, wc))) break;
        tc_fence_after();
        const float4* drow4 = reinterpret_cast<const float4*>(rows_base + s * 2 * BQ + BQ + half * HQ);
        uint32_t pk[32];
        {
            uint32_t dr[2][32];
            tmem_ld64(tmem + lane_off + C::kColDP + half * HQ, dr);
            tmem_ld_wait();
#pragma unroll
            for (int c2 = 0; c2 < HQ / 4; ++c2) {
                const float4 dv4 = drow4[c2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int c = 2 * c2 + u;
                    const int q = (2 * c) / 32, e = (2 * c) % 32;
                    const uint64_t g2 = fadd2(f2_pack(__uint_as_float(dr[q][e]), __uint_as_float(dr[q][e + 1])),
                                              u == 0 ? f2_pack(dv4.x, dv4.y) : f2_pack(dv4.z, dv4.w));
                    float d0, d1;
                    f2_unpack(fmul2(p2[c], g2), d0, d1);
                    pk[c] = pack_bf16(d0, d1);
                }
            }
        }
        tmem_st32(tmem + lane_off + C::kColDP + half * HQ, pk);
        if constexpr (C::kEarlyDsReady) {
            // dK reads dS^T from tensor memory: signal it now, not after the shared-memory copy below,
            // which has to wait until dV has read the dO tile in the slot.
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->ds_ready[half]);
        }
        // dS^T row r into this half's chunk of the step's slot (128-byte rows, 16-byte chunks XOR-swizzled
        // by r % 8) for dQ, once dV has read the dO tile there.
        if (!(ok = warp_wait(&bars->dv_done[s], (i >> 1) & 1, wc))) break;
        uint8_t* row = smem + C::kOffSlot + s * C::kSlotBytes + half * C::kDSChunk + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(row + ((ch ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        fence_proxy_async_smem();
        if constexpr (C::kEarlyDsReady) {
            mbar_arrive(&bars->ds_smem);
        } else {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->ds_ready[half]);
        }

        if (i + 1 < Tq && !(ok = form_p(i + 1))) break;

        // dQ_i: thread = query row r of the step, this warpgroup's d / 2 columns, staged as row r of d / 64
        // [BQ][32] fp32 blocks with 16-byte stores, 16-byte chunks XOR-swizzled by r % 8 (the tensor map's
        // 128-byte swizzle): the first warpgroup's in the step's slot (dQ has read its dS^T), the second's in
        // its own buffer once the previous step's reduce has read it.
        if (!(ok = warp_wait(&bars->dq_full, i & 1, wc))) break;
        tc_fence_after();
        uint32_t x[D / 64][32];
        if constexpr (D == 128) tmem_ld64(tmem + lane_off + C::kColDQ + (D / 2) * half, x);
        else tmem_ld32(tmem + lane_off + C::kColDQ + (D / 2) * half, x[0]);
        tmem_ld_wait();
        tc_fence_before();
        if constexpr (!C::kOwnDQ) mbar_arrive(&bars->dq_empty);
        if (half == 1 && i > 0 && !(ok = warp_wait(&bars->stage_b_free, (i - 1) & 1, wc))) break;
        uint8_t* rowp = smem + (half == 0 ? C::kOffSlot + s * C::kSlotBytes : C::kOffStageB) + r * 128;
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(rowp + b * C::kDqBlockBytes + ((j ^ (lane & 7)) << 4)) =
                    make_uint4(x[b][4 * j], x[b][4 * j + 1], x[b][4 * j + 2], x[b][4 * j + 3]);
        fence_proxy_async_smem();
        mbar_arrive(half == 0 ? &bars->staged_a[s] : &bars->staged_b);
    }
    if (!ok) return;
    if (!warp_wait(&bars->dkdv_full, 0, wc)) return;
    tc_fence_after();
    bwd_write_dkdv<D>(smem, tmem, dk, dv, head, k0, N, scale);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse2, const float* __restrict__ row_d, float* __restrict__ dq_acc,
              __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int N, int Npad,
              int blocks_per_head, float scale, float scale_log2, long long wait_budget, int starve) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024 - (smem_u32(smem_raw) & 1023)) & 1023;
    if (pad > C::kAlignSlack) {   // cannot happen without static shared memory; never touch memory past the end
        if (threadIdx.x == 0) atomicCAS(&g_bwd_status, 0, (int)FA_ERR_CUDA);
        return;
    }
    uint8_t* smem = smem_raw + pad;
    BwdBarriers* bars = reinterpret_cast<BwdBarriers*>(smem + C::kOffBar);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // 1-D grid, head-major: the CTAs of one head walk the same Q/dO blocks, which stay in L2.
    const int head = blockIdx.x / blocks_per_head;
    const int k0 = (blockIdx.x % blocks_per_head) * BK;
    const int Tq = Npad / BQ;
    // Every CTA of a head walks the query blocks starting at its own key-block index, so that at any time
    // the CTAs add into different dQ rows instead of all contending for the same ones in L2.
    const int rot = blockIdx.x % blocks_per_head;

    if (threadIdx.x == 0) {
        bars->wait.budget = wait_budget;
        mbar_init(&bars->kv_full, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->q_full[t], 1);
            mbar_init(&bars->q_empty[t], 1);
            mbar_init(&bars->do_full[t], 1);
            mbar_init(&bars->dv_done[t], 1);
            mbar_init(&bars->staged_a[t], 128);
            mbar_init(&bars->ds_ready[t], 128);
        }
        mbar_init(&bars->staged_b, 128);
        mbar_init(&bars->p_ready, 256);
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->dq_full, 1);
        mbar_init(&bars->dq_empty, 256);
        mbar_init(&bars->ds_smem, 256);
        mbar_init(&bars->stage_b_free, 1);
        mbar_init(&bars->dkdv_full, 1);
        mbar_init(&bars->mma_done, 1);
        bars->wait.abort = 0;
        fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
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
        if (lane == 0)
            bwd_producer<D>(&tm_q, &tm_k, &tm_v, &tm_do, &tm_dq, lse2, row_d, dq_acc, smem, bars, head, k0, N, Tq, Npad, rot,
                            starve);
    } else if (warp == kMmaWarp) {
        if (lane == 0) bwd_mma<D>(smem, bars, tmem, Tq);
    } else {
        bwd_softgrad<D>(smem, bars, tmem, dq_acc, &tm_dq, dk, dv, head, k0, N, Tq, rot, scale, scale_log2);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0 && bars->wait.abort) atomicCAS(&g_bwd_status, 0, (int)FA_ERR_TIMEOUT);
}

// -D_i = -(dO_i . O_i) and -LSE2_i = -LSE_i log2(e) into [head][Npad] arrays (pad rows: 0 and -inf);
// zeroes the fp32 dQ accumulator.  D/8 threads share a row (16-byte loads of O and dO), each warp takes
// 2 * 32 / (D/8) rows per pass, so enough bytes are in flight to stream at HBM speed.
template <int D>
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ lse, float* __restrict__ row_d, float* __restrict__ lse2,
                                float* __restrict__ dq_acc, int N, int Npad, int64_t heads) {
    griddep_launch_dependents();
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
    griddep_wait();   // launched to start while the main kernel finishes: its reduce-adds must be complete
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
                   void* dq, void* dk, void* dv, const Shape& s, float scale, void* workspace, cudaStream_t st,
                   BwdTiming timing) {
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
    count_launches(1);

    CUtensorMap tq, tk, tv, tdo, tdq;
    if ((e = make_tmap_bf16_3d(&tq, q, s.d, s.N, s.heads(), BQ)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tdo, dout, s.d, s.N, s.heads(), BQ)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tk, k, s.d, s.N, s.heads(), BK)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tv, v, s.d, s.N, s.heads(), BK)) != cudaSuccess) return e;
    // The dQ staging boxes: [BQ rows][32 columns], 128-byte swizzled.
    if ((e = make_tmap_f32_3d(&tdq, dq_acc, s.d, s.N, s.heads(), 32, BQ, true)) != cudaSuccess)
        return e;
    e = set_max_dynamic_smem((const void*)bwd_tc_kernel<D>, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int bph = (s.N + BK - 1) / BK;
    if ((long long)bph * s.heads() > INT32_MAX) return cudaErrorInvalidConfiguration;
    const unsigned grid = (unsigned)(bph * s.heads());
    const WaitPolicy wp = wait_policy();
    if (timing.start && (e = cudaEventRecord(timing.start, st)) != cudaSuccess) return e;
    if ((e = launch_dependent(bwd_tc_kernel<D>, dim3(grid), dim3(kThreads), C::kSmemBytes, st, tq, tk, tv, tdo, tdq,
                              lse2, row_d, dq_acc, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, s.N, Npad, bph, scale,
                              scale * 1.4426950408889634f, wp.budget_cycles, wp.starve)) != cudaSuccess)
        return e;
    count_launches(1);
    if (timing.stop && (e = cudaEventRecord(timing.stop, st)) != cudaSuccess) return e;
    if ((e = launch_dependent(bwd_dq_convert_kernel, dim3(blocks), dim3(256), 0, st, dq_acc, (__nv_bfloat16*)dq, scale,
                              s.heads() * (int64_t)s.N * D / 4)) != cudaSuccess)
        return e;
    count_launches(1);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_tc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, const Shape& s, float scale,
                          void* workspace, cudaStream_t st, BwdTiming timing) {
    return s.d == 128 ? launch<128>(q, k, v, o, dout, lse, dq, dk, dv, s, scale, workspace, st, timing)
                      : launch<64>(q, k, v, o, dout, lse, dq, dk, dv, s, scale, workspace, st, timing);
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
