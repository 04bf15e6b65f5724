/*
 * fa.h — C ABI of libfa.so: exact scaled dot-product attention, forward and backward, on one
 * NVIDIA GB300 (sm_103a), computed tile by tile without ever storing the N x N score matrix.
 *
 * The operation.  For every batch b and head h independently,
 *     O = softmax(scale * Q K^T) V,        LSE_i = log(sum_j exp(scale * q_i . k_j))   (natural log)
 * which is Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V of the FlashAttention fable on
 * ckw19810413.github.io (section 概念揭曉), computed the way "账房先生的奔命：Flash Attention 与内存
 * I/O 革命" §六 describes (Tiling + Online Softmax: Q cut into row blocks, K and V streamed in blocks,
 * a running max, a running exp-sum and an output accumulator rescaled by exp(m_old - m_new)), writing
 * only O and the softmax statistic back to device memory (that page's §六 closing remark; the
 * 技术解读 section of "算珠楼的掌簿人").  LSE is the single statistic saved for the backward pass,
 * which recomputes P from it instead of storing P (the same page's §七 重计算).
 *
 * Conventions shared by every entry point:
 *   - Layout: q, k, v, o, dout, dq, dk, dv are contiguous row-major [B, H, N, d] arrays; lse is a
 *     contiguous [B, H, N] fp32 array.  All pointers are DEVICE pointers, 16-byte aligned.
 *   - Ownership: the caller allocates and frees every buffer (including the backward workspace).
 *     The library allocates no device memory of its own and never anything of N x N size; its only
 *     fixed device buffers are the static scratch array of fa_bwd_noalloc and one status word per
 *     kernel source file (read by fa_check_status).
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every
 *     call is asynchronous on that stream; results are valid once the stream has completed.  No call
 *     synchronises the device.
 *   - Scale: applied to the scores; 1/sqrt(d) gives the pages' definition.  Must be finite and > 0.
 *   - No mask, no dropout, no causal option (the pages define none).
 *   - Errors: arguments are checked on the host before anything is launched.  On FA_ERR_INVALID_ARG or
 *     FA_ERR_UNSUPPORTED nothing was launched and no output was written.  FA_ERR_CUDA means a CUDA call
 *     failed (the launch may have been partial).  fa_last_error_string() gives the message of the last
 *     failing call made on the calling thread.
 *   - Device-side waits in the kernels are bounded.  A wait that runs out of its budget stops the
 *     kernel and records FA_ERR_TIMEOUT in a device status word, read by fa_check_status().
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, B/H/N < 1, bad scale, workspace too small */
    FA_ERR_UNSUPPORTED = 2,   /* a head size or shape this build has no kernel for */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or a launch failed */
    FA_ERR_TIMEOUT = 4        /* a bounded device-side wait expired (reported by fa_check_status) */
} fa_status;

/*
 * fa_fwd — bf16 forward on the tensor cores (tcgen05, fp32 accumulation in tensor memory).
 *   q, k, v : const bf16 [B,H,N,d]        (inputs)
 *   o       : bf16 [B,H,N,d]              (output, O = softmax(scale Q K^T) V rounded to bf16)
 *   lse     : float [B,H,N]               (output, natural-log log-sum-exp of each scaled score row)
 *   d       : 64 or 128 (FA_ERR_UNSUPPORTED otherwise).  N may be any value >= 1 (ragged tails are masked).
 *   Product B*H must fit in 2^31 - 1; N*d in 2^31 - 1.
 *   Repeatability: the same inputs give the same bits on every call (no atomics; fixed block order).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, void* stream);

/*
 * fa_fwd_stepnorm — fa_fwd with the per-step normalised accumulator, an ablation of the update rule.
 *   Same arguments, layouts, results (up to rounding) and errors as fa_fwd.  After every K/V block the
 *   output is kept normalised, O_new = exp(m_old - m_new) (l_old / l_new) O_old + exp(S - m_new) V / l_new,
 *   the update rule printed in "账房先生的奔命：Flash Attention 与内存 I/O 革命" §六 (which that page calls a
 *   simplified form); fa_fwd instead keeps the output unnormalised and divides once at the end (the
 *   rescale of the FlashAttention fable on ckw19810413.github.io, 兩大核心魔法).  This entry point exists to
 *   measure that difference: it rescales O in tensor memory on every block.
 */
fa_status fa_fwd_stepnorm(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int N, int d, float scale, void* stream);

/*
 * fa_fwd_f32 — fp32 forward on the CUDA cores (no tensor-core rounding of any operand).
 *   q, k, v, o : float [B,H,N,d];  lse : float [B,H,N].
 *   d          : 1 .. 128 and a multiple of 4 (FA_ERR_UNSUPPORTED otherwise).
 *   Same tiled, online-softmax method as fa_fwd, for callers that need fp32 results.
 */
fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                     int B, int H, int N, int d, float scale, void* stream);

/*
 * fa_bwd_workspace_size — bytes of device scratch fa_bwd needs for this shape: an fp32 dQ accumulator
 * [B,H,N,d] and two fp32 per-row arrays [B,H,Np] with Np = N rounded up to a multiple of 128 (the
 * negated row term -D_i = -dO_i . O_i and the negated log2-domain LSE), each section rounded up to 256
 * bytes.  Returns 0 for invalid shapes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * fa_bwd — bf16 backward: gradients of O(Q,K,V) contracted with dout.
 *   q, k, v    : const bf16 [B,H,N,d]  (the forward's inputs)
 *   o          : const bf16 [B,H,N,d]  (the forward's output)
 *   dout       : const bf16 [B,H,N,d]  (upstream gradient dO)
 *   lse        : const float [B,H,N]   (the forward's LSE output)
 *   dq, dk, dv : bf16 [B,H,N,d]        (outputs)
 *   workspace  : device scratch of at least fa_bwd_workspace_size(B,H,N,d) bytes, 256-byte aligned;
 *                its contents on entry do not matter and are overwritten.
 *   d          : 64 or 128.
 * P is recomputed tile by tile from q, k and lse (it is never stored); dV = P^T dO, dP = dO V^T,
 * dS = P o (dP - D), dK = scale dS^T Q, dQ = scale dS K with D_i = dO_i . O_i.
 * Repeatability: dk and dv are the same bits on every call with the same inputs; dq sums per-key-block
 * contributions whose order varies between calls, so its last bits may differ (within rounding).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_noalloc — fa_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for callers that receive only their input and output buffers
 * (for example an operator plugin whose host framework owns all device memory) or that must not call
 * cudaMalloc because it can synchronise the device.
 *   Arguments: as fa_bwd, without the workspace.  The call allocates nothing: it uses a scratch array
 *   of FA_BWD_NOALLOC_MAX_SCRATCH_BYTES (32 MiB) compiled into the library, which every GPU that loads
 *   the library holds until the process exits.
 *   Checks: shape, scale and head size are checked first, exactly as fa_bwd checks them (a d other than
 *   64 or 128 gives FA_ERR_UNSUPPORTED), then the size of the scratch, then the pointers.
 *   Limit: shapes with fa_bwd_workspace_size(B,H,N,d) > FA_BWD_NOALLOC_MAX_SCRATCH_BYTES are rejected
 *   with FA_ERR_INVALID_ARG before anything is launched: for d = 128 (about 520 bytes per row) B*H*N
 *   above 64528 rows, for d = 64 (about 264 bytes per row) above 127100 rows.  So B=4, H=16, N=2048,
 *   d=64 (131072 rows) does not fit, nor B=1, H=16, N=8192, d=128; use fa_bwd for those.
 *   Set-up: the first call on a device (made with that device current, like every call) looks up the
 *   array's device address with cudaGetSymbolAddress, and so does the first call after the device's
 *   context has changed (for example after cudaDeviceReset); make those calls before any stream capture.
 *   Under CUDA's lazy module loading (the default) that first call is also when the driver loads the
 *   library's device code and with it the array, so the device's free memory drops by the array's size
 *   then, and never again; a caller that must not see that happen later makes the set-up call early.
 *   Sharing: all calls on a device share the one array, which keeps the last call's contents (the
 *   kernels clear whatever must start at zero).  Calls whose executions overlap on the GPU (on
 *   different streams, or from different threads) race on the array and give wrong results: order
 *   them on one stream or with events.
 */
#define FA_BWD_NOALLOC_MAX_SCRATCH_BYTES (32u << 20)
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, void* stream);

/*
 * fa_debug_time_bwd_main — a timing diagnostic; the pages have no counterpart.  The next fa_bwd or
 * fa_bwd_noalloc call made on the calling thread records `start_event` on its stream right before the
 * backward's main kernel (the one that forms P, dS, dV, dK and dQ) and `stop_event` right after it, so that
 * cudaEventElapsedTime gives that kernel's time alone (the call's other two kernels, the row terms before it
 * and the dQ conversion after it, are outside).  Both are cudaEvent_t passed as void*, created by the
 * caller on the call's device.  The setting is used once: the next backward call takes it even if that
 * call then fails its argument checks (and so records nothing).  NULL, NULL clears it.
 */
void fa_debug_time_bwd_main(void* start_event, void* stop_event);

/*
 * fa_test_force_wait_timeout — a switch for testing the failure path of the bounded device waits; the
 * pages have no counterpart.  With enable != 0, every later launch of the tensor-core kernels (fa_fwd,
 * fa_fwd_stepnorm, fa_bwd, fa_bwd_noalloc, from any thread) withholds its Q tile loads and gives its waits
 * a budget of about 10 ms instead of about 2 s, so that the first wait on Q runs out: the kernel winds down
 * by itself (no fault, no trap), fa_check_status() then reports FA_ERR_TIMEOUT, and the outputs of those
 * calls are not valid.  enable = 0 restores normal operation.  Off by default; nothing but an explicit call
 * (no environment variable) turns it on.
 */
void fa_test_force_wait_timeout(int enable);

/* Message of the last failing call on the calling thread ("" if none).  Valid until the next call. */
const char* fa_last_error_string(void);

/*
 * fa_kernel_launches — number of kernels this library has launched in this process so far, over all
 * threads and devices; every entry point adds each kernel it enqueues (fa_fwd: one or two, the second for
 * the last partial wave of tiles; fa_bwd: three; fa_fwd_f32: one).  Never reset.  A diagnostic: the
 * difference across a region counts the launches made in it.
 */
unsigned long long fa_kernel_launches(void);

/*
 * fa_check_status — synchronises `stream`, then reports and clears the device status word:
 * FA_ERR_TIMEOUT if a kernel gave up a bounded wait since the last check, FA_ERR_CUDA if the stream
 * reported an error, else FA_OK.  A debugging and test helper; the fast path never calls it.
 */
fa_status fa_check_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
