// bf16 attention forward on the sm_103a tensor cores (tcgen05 + TMA + tensor memory).
//
// Method ("账房先生的奔命：Flash Attention 与内存 I/O 革命" §六, Tiling + Online Softmax): a CTA owns two
// tiles of 128 query rows (Q0, Q1) and streams K_j, V_j (128 keys each) through a shared-memory ring.
// For every K/V block and both Q tiles:
//     S = Q K_j^T                                   tcgen05.mma, fp32 in tensor memory (TMEM)
//     m_new = max(m, rowmax(scale S))               one thread owns one row: no shuffles
//     P = exp(scale S - m_new), l = a l + rowsum P  a = exp(m - m_new)
//     O = a O + P V_j                               P goes back to TMEM as bf16 and feeds the MMA
// and only O / l (bf16) and LSE = m + ln l (fp32) are written to global memory (the 技术解读 section of
// "算珠楼的掌簿人": only the output and the statistics return to HBM).  The rescale by
// exp(m_old - m_new) is the identity of the FlashAttention fable on ckw19810413.github.io (兩大核心魔法).
//
// Rescale skipping: the reference max used in the exponent is only moved when the row max grows by
// more than 2^8 (in the log2 domain).  O and l always share that reference, so O / l and
// m + ln l are unchanged; the skipped rescales only bound P by 256 instead of 1.
//
// kStepNorm (fa_fwd_stepnorm) instead keeps O normalised after every block, the per-step update rule
// that "账房先生的奔命" §六 prints:  O_new = exp(m_old - m_new) (l_old / l_new) O_old + exp(S - m_new) V / l_new.
// P is divided by l_new before the MMA, O is rescaled in tensor memory on every block, and nothing is
// divided at the end.  It gives the same results up to rounding and exists to measure what the
// unnormalised accumulator saves.
//
// Warp roles (320 threads): warps 0-3 own Q0's rows, warps 4-7 own Q1's rows (thread = row = TMEM
// lane), warp 8 issues TMA loads, warp 9 allocates TMEM and issues the MMAs.  While one warpgroup
// exponentiates its S tile the tensor cores run the other tile's MMAs.
//
// Work: a CTA takes a pair of adjacent 128-row tiles of one head (a head-major 1-D grid).  When the
// pairs do not fill the GPU's last wave, those last pairs run as 2-CTA clusters instead: each CTA of a
// cluster streams half of the K/V blocks, rank 1 hands its unnormalised O, m and l to rank 0 through
// distributed shared memory, and rank 0 merges the halves,
//     m = max(m0, m1),  l = 2^(m0-m) l0 + 2^(m1-m) l1,  O = (2^(m0-m) O0 + 2^(m1-m) O1) / l,
// the same exp-sum factorisation as the online rescale.  The last wave then takes half as long.  The
// clusters' launch is a programmatic dependent of the full waves' (every CTA releases it at its start), so
// its CTAs take SMs as the full waves leave them instead of waiting for the whole first launch to drain:
// the forward measured 1.1 % faster at N = 8192 d = 128, 3.3 % at N = 2048 and 4.5 % at B=4 H=16 N=2048
// d = 64.
//
// TMEM columns at d = 128: S0/P0 [0,128), S1/P1 [128,256), O0 [256,384), O1 [384,512).  At d = 64 S rotates
// through three buffers [0,128), [128,256), [256,384) (S of the next tile is formed while the softmax works
// on the current one), O0 [384,448), O1 [448,512); K and V share one barrier per ring stage.

#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

using namespace ptx;

__device__ int g_fwd_status;

constexpr int BM = 128;  // query rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;  // keys per K/V block
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kMaxStages = 4;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdBarriers {
    uint64_t q_full[2];
    uint64_t k_full[kMaxStages];
    uint64_t v_full[kMaxStages];
    uint64_t kv_empty[kMaxStages];
    uint64_t s_full[2][2];   // [tile][block parity]: S of a tile's block j is in TMEM
    uint64_t p_full[2][2];   // [tile][block parity]: P of a tile's block j is in TMEM
    uint64_t o_full[2];
    uint64_t pv_done[2];   // d = 64, per-step normalisation: PV of a tile has completed (before O is rescaled)
    uint64_t mma_done;
    uint32_t tmem_base;
    WaitCtl wait;
};

template <int D>
struct FwdCfg {
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kChunks = D / 64;                 // 64-column (128-byte) swizzle chunks
    static constexpr uint32_t kChunkQ = BM * 128;          // bytes of one chunk of a Q tile
    static constexpr uint32_t kChunkKV = BN * 128;
    static constexpr uint32_t kQBytes = BM * D * 2;
    static constexpr uint32_t kKVBytes = BN * D * 2;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + 2 * kQBytes;
    static constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
    static constexpr uint32_t kOffBar = kOffV + kStages * kKVBytes;
    static constexpr uint32_t kSmemBytes = kOffBar + sizeof(FwdBarriers) + 1024;  // + alignment slack
    // d = 64 leaves room for a third S buffer: S tiles rotate through three buffers (S of block j + 1 is
    // formed while the softmax of block j runs) and O0, O1 take the last 128 columns.  At d = 128 each
    // tile has one S buffer.
    static constexpr bool kThreeS = D == 64;
    // d = 64 keeps four K/V stages, so a block's V has long landed when its K is waited for: one barrier per
    // stage covers both, which spares the MMA thread one barrier test per block.
    static constexpr bool kOneKVBarrier = D == 64;
    __host__ __device__ static constexpr uint32_t col_s(int t) { return (uint32_t)t * 128; }
    __host__ __device__ static constexpr uint32_t col_o(int t) { return (kThreeS ? 384 : 256) + (uint32_t)t * D; }
    // Buffer of the S tile with issue index k = 2 j + t (block j, tile t) when there are three.
    __host__ __device__ static constexpr uint32_t col_s3(int k) { return (uint32_t)(k % 3) * 128; }
    static constexpr uint32_t kTmemCols = 512;
};

template <int D>
__device__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint8_t* smem,
                         FwdBarriers* bars, int head, int q0, int kv0, int T, int starve) {
    using C = FwdCfg<D>;
    WaitCtl* wc = &bars->wait;
    const uint64_t pol_kv = policy_evict_last();
    const uint64_t pol_q = policy_evict_first();
    // starve != 0 withholds the Q loads so that the MMA warp's first wait runs out: the failure path
    // of the bounded waits, exercised by the tests with a short budget.
    for (int t = 0; t < 2 && !starve; ++t) {
        mbar_expect_tx(&bars->q_full[t], C::kQBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffQ + t * C::kQBytes + c * C::kChunkQ, tm_q, &bars->q_full[t], c * 64,
                        q0 + t * BM, head, pol_q);
    }
    int issued = 0;
    for (int j = 0; j < T; ++j) {
        const int s = j % C::kStages;
        if (j >= C::kStages && !mbar_wait(&bars->kv_empty[s], ((j / C::kStages) - 1) & 1, wc)) break;
        // With one K/V barrier (d = 64) both tiles complete on k_full.
        uint64_t* v_bar = C::kOneKVBarrier ? &bars->k_full[s] : &bars->v_full[s];
        mbar_expect_tx(&bars->k_full[s], C::kOneKVBarrier ? 2 * C::kKVBytes : C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffK + s * C::kKVBytes + c * C::kChunkKV, tm_k, &bars->k_full[s], c * 64,
                        (kv0 + j) * BN, head, pol_kv);
        if (!C::kOneKVBarrier) mbar_expect_tx(v_bar, C::kKVBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(smem + C::kOffV + s * C::kKVBytes + c * C::kChunkKV, tm_v, v_bar, c * 64,
                        (kv0 + j) * BN, head, pol_kv);
        issued = j + 1;
    }
    // Every load issued must have landed before the CTA may exit (only matters after an abort).
    drain_wait(&bars->q_full[0], 0, wc);
    drain_wait(&bars->q_full[1], 0, wc);
    for (int j = (issued > C::kStages ? issued - C::kStages : 0); j < issued; ++j) {
        drain_wait(&bars->k_full[j % C::kStages], (j / C::kStages) & 1, wc);
        if (!C::kOneKVBarrier) drain_wait(&bars->v_full[j % C::kStages], (j / C::kStages) & 1, wc);
    }
}

template <int D, bool kStepNorm>
__device__ void mma_issuer(uint8_t* smem, FwdBarriers* bars, uint32_t tmem, int T) {
    using C = FwdCfg<D>;
    WaitCtl* wc = &bars->wait;
    constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0, 0);
    constexpr uint32_t idPV = idesc_bf16_f32(BM, D, 0, 1);
    // Operand descriptors are built once; each k-step only adds a constant byte offset.
    const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::kOffQ), 16, 1024);
    const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::kOffK), 16, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::kOffV), C::kChunkKV, 1024);

    auto issue_s_to = [&](int t, int s, uint32_t col) {
        const uint64_t a0 = sdesc_advance(dQ0, t * C::kQBytes);
        const uint64_t b0 = sdesc_advance(dK0, s * C::kKVBytes);
        const uint32_t d = tmem + col;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            mma_ss(d, sdesc_advance(a0, (kk / 4) * C::kChunkQ + (kk % 4) * 32),
                   sdesc_advance(b0, (kk / 4) * C::kChunkKV + (kk % 4) * 32), idS, kk > 0);
        }
    };
    auto issue_s = [&](int t, int s) { issue_s_to(t, s, C::col_s(t)); };
    auto issue_pv_from = [&](int t, int s, bool accumulate, uint32_t col) {
        const uint64_t b0 = sdesc_advance(dV0, s * C::kKVBytes);
        const uint32_t d = tmem + C::col_o(t);
        const uint32_t a = tmem + col;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(d, a + kk * 8, sdesc_advance(b0, kk * 16 * 128), idPV, (accumulate || kk > 0) ? 1u : 0u);
    };
    auto issue_pv = [&](int t, int s, bool accumulate) { issue_pv_from(t, s, accumulate, C::col_s(t)); };

    bool ok = mbar_wait_poll(&bars->q_full[0], 0, wc) && mbar_wait_poll(&bars->q_full[1], 0, wc);
    if constexpr (C::kThreeS) {
        // S tiles in issue order k = 2 j + t go to buffer k % 3; PV(k) frees that buffer for S(k + 3), so
        // S of the next block is ready when the softmax warps finish the current one.
        auto kwait = [&](int j) {
            return mbar_wait_poll(&bars->k_full[j % C::kStages], (j / C::kStages) & 1, wc);
        };
        if (ok && (ok = kwait(0))) {
            tc_fence_after();
            issue_s_to(0, 0, C::col_s3(0));
            mma_commit(&bars->s_full[0][0]);
            issue_s_to(1, 0, C::col_s3(1));
            mma_commit(&bars->s_full[1][0]);
            if (T > 1 && (ok = kwait(1))) {
                tc_fence_after();
                issue_s_to(0, 1 % C::kStages, C::col_s3(2));
                mma_commit(&bars->s_full[0][1]);
            }
        }
        // V of block j shares K's barrier, which kwait(j) saw before S of block j was issued.
        static_assert(C::kOneKVBarrier, "the three-buffer loop relies on one K/V barrier per stage");
        for (int j = 0; ok && j < T; ++j) {
            const int s = j % C::kStages;
            for (int t = 0; ok && t < 2; ++t) {
                const int k = 2 * j + t;
                if (!(ok = mbar_wait_poll(&bars->p_full[t][j & 1], (j >> 1) & 1, wc))) break;
                const int kn = k + 3, jn = kn / 2, tn = kn % 2;
                // K/V of the block whose S follows this PV, tested right behind P rather than between PV and
                // S: each barrier test by this thread idles the tensor core, two adjacent ones little more
                // than one (0.4-0.7 % faster at N >= 8192).
                if (jn < T && tn == 0 && !(ok = kwait(jn))) break;
                tc_fence_after();
                issue_pv_from(t, s, j > 0, C::col_s3(k));
                // Only the per-step normalisation rescales O on every block; the lazy rescale finds PV(k)
                // complete through a later commit (see prev_pv_done in the softmax warps).
                if (kStepNorm) mma_commit(&bars->pv_done[t]);
                if (j == T - 1) mma_commit(&bars->o_full[t]);
                if (t == 1) mma_commit(&bars->kv_empty[s]);
                if (jn < T) {
                    issue_s_to(tn, jn % C::kStages, C::col_s3(kn));
                    mma_commit(&bars->s_full[tn][jn & 1]);
                }
            }
        }
    }
    for (int j = 0; !C::kThreeS && ok && j < T; ++j) {
        const int s = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        if (j == 0) {
            if (!(ok = mbar_wait_poll(&bars->k_full[s], ph, wc))) break;
            tc_fence_after();
            issue_s(0, s);
            mma_commit(&bars->s_full[0][0]);
            issue_s(1, s);
            mma_commit(&bars->s_full[1][0]);
        }
        const int s2 = (j + 1) % C::kStages;
        const uint32_t ph2 = ((j + 1) / C::kStages) & 1;
        if (!(ok = mbar_wait_poll(&bars->v_full[s], ph, wc))) break;
        if (!(ok = mbar_wait_poll(&bars->p_full[0][j & 1], (j >> 1) & 1, wc))) break;
        tc_fence_after();
        issue_pv(0, s, j > 0);
        if (j == T - 1) mma_commit(&bars->o_full[0]);
        if (j + 1 < T) {
            if (!(ok = mbar_wait_poll(&bars->k_full[s2], ph2, wc))) break;
            tc_fence_after();
            issue_s(0, s2);
            mma_commit(&bars->s_full[0][(j + 1) & 1]);
        }
        if (!(ok = mbar_wait_poll(&bars->p_full[1][j & 1], (j >> 1) & 1, wc))) break;
        tc_fence_after();
        issue_pv(1, s, j > 0);
        mma_commit(&bars->kv_empty[s]);
        if (j == T - 1) mma_commit(&bars->o_full[1]);
        if (j + 1 < T) {
            issue_s(1, s2);
            mma_commit(&bars->s_full[1][(j + 1) & 1]);
        }
    }
    // Tensor memory is freed after this: every MMA issued must have completed.
    mma_commit(&bars->mma_done);
    drain_wait(&bars->mma_done, 0, wc);
}

// Three S buffers, lazy rescale: before tile t rescales O at block j > 0, PV of its previous block (issue
// index k - 2, with k = 2 j + t) must have completed.  The MMA thread issues S(k + 1) right after PV(k - 2), so
// S(k + 1)'s commit covers it; in the one step with no S(k + 1) (tile 1 of the last block) the commit that
// frees the K/V stage of block j - 1, also issued right after PV(k - 2), does.  Neither barrier can complete
// a later phase before this warpgroup hands over P of block j, so the parity identifies the phase.
template <int D>
__device__ bool prev_pv_done(FwdBarriers* bars, int t, int j, int T, WaitCtl* wc) {
    using C = FwdCfg<D>;
    const int k1 = 2 * j + t + 1;
    if (k1 < 2 * T) {
        const int t1 = k1 & 1, j1 = k1 >> 1;
        return warp_wait(&bars->s_full[t1][j1 & 1], (j1 >> 1) & 1, wc);
    }
    const int jp = j - 1;
    return warp_wait(&bars->kv_empty[jp % C::kStages], (jp / C::kStages) & 1, wc);
}

template <int D, bool kStepNorm>
__device__ void softmax_wg(FwdBarriers* bars, uint32_t tmem, int t, __nv_bfloat16* __restrict__ o,
                           float* __restrict__ lse, int head, int q0, int N, int kv0, int T, int T_all,
                           float scale_log2, float* ml_out) {
    using C = FwdCfg<D>;
    WaitCtl* wc = &bars->wait;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS1 = tmem + C::col_s(t) + lane_off;
    const uint32_t tO = tmem + C::col_o(t) + lane_off;
    const int tail = N - (T_all - 1) * BN;  // valid keys in the head's last block (1..BN)

    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
        if (!(ok = warp_wait(&bars->s_full[t][j & 1], (j >> 1) & 1, wc))) break;
        tc_fence_after();
        const uint32_t tS = C::kThreeS ? tmem + C::col_s3(2 * j + t) + lane_off : tS1;
        uint32_t r[4][32];
        // Four 32-column loads: one 128-column load measured 0.3-2 % slower here (unlike the backward).
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, r[q]);
        tmem_ld_wait();
        if (kv0 + j == T_all - 1 && tail < BN) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (q * 32 + c >= tail) r[q][c] = __float_as_uint(-INFINITY);
        }
        // Row max as eight independent chains of 3-input maxima: with two warps per scheduler there is
        // nothing else to hide a 128-long dependent chain behind.
        float mc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mc[k] = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int c = 0; c < 32; c += 2)
                mc[(c / 2) % 8] = max3(mc[(c / 2) % 8], __uint_as_float(r[q][c]), __uint_as_float(r[q][c + 1]));
        const float mx = max3(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
        if constexpr (kStepNorm) {
            const float m_new = fmaxf(m_run, mx * scale_log2);
            const float alpha = ex2(m_run - m_new);  // 0 on the first block (m_run = -inf)
            m_run = m_new;
            const uint64_t sl2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_run, -m_run);
            uint64_t s2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float x0, x1;
                    f2_unpack(ffma2(f2_pack(__uint_as_float(r[q][e]), __uint_as_float(r[q][e + 1])), sl2, nm2), x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    s2[(e / 2) % 4] = fadd2(s2[(e / 2) % 4], f2_pack(p0, p1));
                    r[q][e] = __float_as_uint(p0);
                    r[q][e + 1] = __float_as_uint(p1);
                }
            float sc[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) f2_unpack(s2[k], sc[2 * k], sc[2 * k + 1]);
            const float l_new = alpha * l_run + (((sc[0] + sc[1]) + (sc[2] + sc[3])) + ((sc[4] + sc[5]) + (sc[6] + sc[7])));
            const float inv = 1.f / l_new;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int q = 2 * h + c / 16, e = (2 * c) % 32;
                    pk[c] = pack_bf16(__uint_as_float(r[q][e]) * inv, __uint_as_float(r[q][e + 1]) * inv);
                }
                tmem_st32(tS + h * 32, pk);
            }
            // With three S buffers, PV of the previous block may still be accumulating into O.
            if (C::kThreeS && j > 0 && !(ok = warp_wait(&bars->pv_done[t], (j - 1) & 1, wc))) break;
            if (j > 0) {
                const float c_old = alpha * l_run * inv;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t x[32];
                    tmem_ld32(tO + q * 32, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * c_old);
                    tmem_st32(tO + q * 32, x);
                }
            }
            l_run = l_new;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->p_full[t][j & 1]);
        } else {
            const float m_new = fmaxf(m_run, mx * scale_log2);
            const bool rescale = m_new - m_run > kRescaleThreshold;  // always true for the first block
            float alpha = 1.f;
            if (rescale) {
                alpha = ex2(m_run - m_new);
                m_run = m_new;
            }
            const float neg_m = -m_run;
            // s * scale*log2e - m and the row sum run on packed pairs (f32x2): two results per instruction.
            const uint64_t sl2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(neg_m, neg_m);
            uint64_t s2[4] = {0, 0, 0, 0};
            // P of keys [64 h, 64 h + 64) as 32 bf16 pairs.
            auto exp_half = [&](int h, uint32_t (&pk)[32]) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int q = 2 * h + c / 16, e = (2 * c) % 32;
                    const uint64_t x2 = ffma2(f2_pack(__uint_as_float(r[q][e]), __uint_as_float(r[q][e + 1])), sl2, nm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    s2[c % 4] = fadd2(s2[c % 4], f2_pack(p0, p1));
                    pk[c] = pack_bf16(p0, p1);
                }
            };
            if constexpr (D == 128) {
                // One 64-column store: 0.5-0.8 % faster here, 0.7 % slower at d = 64 (measured).
                uint32_t pk[2][32];
                exp_half(0, pk[0]);
                exp_half(1, pk[1]);
                tmem_st64(tS, pk);
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
                    exp_half(h, pk);
                    tmem_st32(tS + h * 32, pk);
                }
            }
            float sc[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) f2_unpack(s2[k], sc[2 * k], sc[2 * k + 1]);
            const float sum = ((sc[0] + sc[1]) + (sc[2] + sc[3])) + ((sc[4] + sc[5]) + (sc[6] + sc[7]));
            l_run = l_run * alpha + sum;
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                // With three S buffers, PV of the previous block may still be accumulating into O.
                if (C::kThreeS && !(ok = prev_pv_done<D>(bars, t, j, T, wc))) break;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t x[32];
                    tmem_ld32(tO + q * 32, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * alpha);
                    tmem_st32(tO + q * 32, x);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->p_full[t][j & 1]);
        }
    }
    if (!ok) return;
    if (!warp_wait(&bars->o_full[t], 0, wc)) return;
    tc_fence_after();
    if (ml_out) {  // one half of a split pair: O stays in TMEM, m and l go to shared memory for the merge
        ml_out[t * BM + quarter * 32 + lane] = m_run;
        ml_out[2 * BM + t * BM + quarter * 32 + lane] = l_run;
        return;
    }

    const int row = q0 + t * BM + quarter * 32 + lane;
    const float inv_l = kStepNorm ? 1.f : 1.f / l_run;
    const size_t base = ((size_t)head * N + row) * D;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t x[32];
        tmem_ld32(tO + q * 32, x);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
            pk[c] = pack_bf16(__uint_as_float(x[2 * c]) * inv_l, __uint_as_float(x[2 * c + 1]) * inv_l);
        if (row < N) {
            uint4* dst = reinterpret_cast<uint4*>(o + base + q * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
    }
    if (row < N) lse[(size_t)head * N + row] = (m_run + log2f(l_run)) * 0.69314718055994531f;
}

// Rank 1 of a split pair: this thread's row of O (from TMEM), m and l into rank 0's shared memory
// (O column-major by row so that a warp's stores land in consecutive words).
template <int D>
__device__ void split_send(uint8_t* smem, uint32_t tmem, int t) {
    using C = FwdCfg<D>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t o_peer = mapa_shared(smem_u32(smem + C::kOffK), 0);
    const uint32_t ml_peer = mapa_shared(smem_u32(smem + C::kOffQ), 0);
    const float* ml_own = reinterpret_cast<const float*>(smem + C::kOffQ + 4096);
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t x[32];
        tmem_ld32(tmem + C::col_o(t) + lane_off + q * 32, x);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c)
            st_cluster_f32(o_peer + (uint32_t)(((t * D + q * 32 + c) * BM + r) * 4), __uint_as_float(x[c]));
    }
    st_cluster_f32(ml_peer + (uint32_t)((t * BM + r) * 4), ml_own[t * BM + r]);
    st_cluster_f32(ml_peer + (uint32_t)((2 * BM + t * BM + r) * 4), ml_own[2 * BM + t * BM + r]);
}

// Rank 0 of a split pair: merges its own half (TMEM, m and l in shared memory) with the received one and
// writes this thread's row of O and LSE.
template <int D>
__device__ void split_merge(uint8_t* smem, uint32_t tmem, int t, __nv_bfloat16* __restrict__ o,
                            float* __restrict__ lse, int head, int q0, int N) {
    using C = FwdCfg<D>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float* opart = reinterpret_cast<const float*>(smem + C::kOffK);
    const float* ml_peer = reinterpret_cast<const float*>(smem + C::kOffQ);
    const float* ml_own = reinterpret_cast<const float*>(smem + C::kOffQ + 4096);
    const float m0 = ml_own[t * BM + r], l0 = ml_own[2 * BM + t * BM + r];
    const float m1 = ml_peer[t * BM + r], l1 = ml_peer[2 * BM + t * BM + r];
    const float m = fmaxf(m0, m1);
    const float a0 = ex2(m0 - m), a1 = ex2(m1 - m);
    const float l = a0 * l0 + a1 * l1;
    const float inv = 1.f / l;
    const int row = q0 + t * BM + r;
    const size_t base = ((size_t)head * N + row) * D;
#pragma unroll
    for (int q = 0; q < D / 32; ++q) {
        uint32_t x[32];
        tmem_ld32(tmem + C::col_o(t) + lane_off + q * 32, x);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int col = q * 32 + 2 * c;
            const float v0 = (a0 * __uint_as_float(x[2 * c]) + a1 * opart[(t * D + col) * BM + r]) * inv;
            const float v1 = (a0 * __uint_as_float(x[2 * c + 1]) + a1 * opart[(t * D + col + 1) * BM + r]) * inv;
            pk[c] = pack_bf16(v0, v1);
        }
        if (row < N) {
            uint4* dst = reinterpret_cast<uint4*>(o + base + q * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
    }
    if (row < N) lse[(size_t)head * N + row] = (m + log2f(l)) * 0.69314718055994531f;
}

template <int D, bool kStepNorm>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
              int N, int blocks_per_head, int pair_base, int split, float scale_log2, long long wait_budget,
              int starve) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    FwdBarriers* bars = reinterpret_cast<FwdBarriers*>(smem + C::kOffBar);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // 1-D grid, head-major: the CTAs of one head run together and share its K/V through L2.  With
    // split != 0 two consecutive CTAs (one cluster) share pair pair_base + blockIdx.x / 2.
    const int pair = pair_base + (split ? (int)blockIdx.x / 2 : (int)blockIdx.x);
    const int head = pair / blocks_per_head;
    const int q0 = (pair % blocks_per_head) * 2 * BM;
    const int T_all = (N + BN - 1) / BN;
    const uint32_t rank = split ? cluster_ctarank() : 0;
    const int kv0 = split ? (int)rank * (T_all / 2) : 0;
    const int T = split ? (rank ? T_all - T_all / 2 : T_all / 2) : T_all;
    // The split tail's launch may start on SMs that the full waves have left; it reads only the call's
    // inputs and writes other rows than they do.
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        bars->wait.budget = wait_budget;
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars->q_full[t], 1);
            for (int b = 0; b < 2; ++b) {
                mbar_init(&bars->s_full[t][b], 1);
                mbar_init(&bars->p_full[t][b], BM);
            }
            mbar_init(&bars->o_full[t], 1);
            mbar_init(&bars->pv_done[t], 1);
        }
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->kv_empty[s], 1);
        }
        mbar_init(&bars->mma_done, 1);
        bars->wait.abort = 0;
        fence_mbar_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
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
        if (lane == 0) producer<D>(&tm_q, &tm_k, &tm_v, smem, bars, head, q0, kv0, T, starve);
    } else if (warp == kMmaWarp) {
        if (lane == 0) mma_issuer<D, kStepNorm>(smem, bars, tmem, T);
    } else {
        softmax_wg<D, kStepNorm>(bars, tmem, warp / 4, o, lse, head, q0, N, kv0, T, T_all, scale_log2,
                                 split ? reinterpret_cast<float*>(smem + C::kOffQ + 4096) : nullptr);
    }

    tc_fence_before();
    __syncthreads();
    if (split) {
        // Every thread of both CTAs reaches both cluster barriers: all waits before them are bounded.
        cluster_sync();  // both halves done: rank 0's K/V and Q buffers are free to receive
        tc_fence_after();
        const bool both_ok = !bars->wait.abort;
        if (rank == 1 && warp < 8 && both_ok) split_send<D>(smem, tmem, warp / 4);
        cluster_sync();  // rank 1's stores are visible to rank 0
        if (rank == 0 && warp < 8 && both_ok) split_merge<D>(smem, tmem, warp / 4, o, lse, head, q0, N);
        tc_fence_before();
        __syncthreads();
    }
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (threadIdx.x == 0 && bars->wait.abort) atomicCAS(&g_fwd_status, 0, (int)FA_ERR_TIMEOUT);
    // A split-tail CTA does not finish before the full waves have: what follows on the stream sees both.
    if (threadIdx.x == 0) griddep_wait();
}

template <int D, bool kStepNorm>
cudaError_t launch(const void* q, const void* k, const void* v, void* o, float* lse, const Shape& s, float scale,
                   cudaStream_t st) {
    using C = FwdCfg<D>;
    CUtensorMap tq, tk, tv;
    cudaError_t e;
    if ((e = make_tmap_bf16_3d(&tq, q, s.d, s.N, s.heads(), BM)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tk, k, s.d, s.N, s.heads(), BN)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16_3d(&tv, v, s.d, s.N, s.heads(), BN)) != cudaSuccess) return e;
    e = set_max_dynamic_smem((const void*)fwd_tc_kernel<D, kStepNorm>, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int bph = (s.N + 2 * BM - 1) / (2 * BM);
    if ((long long)bph * s.heads() > INT32_MAX) return cudaErrorInvalidConfiguration;
    const long long pairs = (long long)bph * s.heads();
    // Whole waves of pair CTAs; a last partial wave runs as split pairs (2-CTA clusters) when it fits.
    const long long sms = device_sm_count();
    const long long full = (pairs / sms) * sms, rest = pairs - full;
    const int T_all = (s.N + BN - 1) / BN;
    const bool split_tail = !kStepNorm && T_all >= 2 && rest > 0 && 2 * rest <= sms;
    const unsigned grid = (unsigned)(split_tail ? full : pairs);
    const float scale_log2 = scale * 1.4426950408889634f;
    const WaitPolicy wp = wait_policy();
    auto* out = (__nv_bfloat16*)o;
    if (grid > 0) {
        fwd_tc_kernel<D, kStepNorm><<<grid, kThreads, C::kSmemBytes, st>>>(tq, tk, tv, out, lse, s.N, bph, 0, 0,
                                                                           scale_log2, wp.budget_cycles, wp.starve);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        count_launches(1);
    }
    if (split_tail) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(2 * rest));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = grid > 0 ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, fwd_tc_kernel<D, kStepNorm>, tq, tk, tv, out, lse, s.N, bph, (int)full, 2,
                               scale_log2, wp.budget_cycles, wp.starve);
        if (e != cudaSuccess) return e;
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const void* q, const void* k, const void* v, void* o, float* lse, const Shape& s,
                          float scale, cudaStream_t st, bool stepnorm) {
    if (stepnorm)
        return s.d == 128 ? launch<128, true>(q, k, v, o, lse, s, scale, st)
                          : launch<64, true>(q, k, v, o, lse, s, scale, st);
    return s.d == 128 ? launch<128, false>(q, k, v, o, lse, s, scale, st)
                      : launch<64, false>(q, k, v, o, lse, s, scale, st);
}

int fwd_tc_read_and_clear_status(cudaStream_t st) {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_fwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_fwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    return v;
}

}  // namespace fa
