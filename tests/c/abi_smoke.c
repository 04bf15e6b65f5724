/*
 * Plain-C use of libfa.so through include/fa.h only: device buffers from the CUDA runtime, the bf16
 * forward (fa_fwd) checked against the fp32 forward (fa_fwd_f32) on the same bf16-rounded inputs, the
 * backward run once, and the host-side argument checks.  Exit code 0 on success.
 * Build: gcc -std=c11 -Iinclude -I<cuda>/include tests/c/abi_smoke.c -L<lib dir> -lfa -lcudart -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "fa.h"

#define CHECK_CUDA(x)                                                          \
    do {                                                                       \
        cudaError_t e_ = (x);                                                  \
        if (e_ != cudaSuccess) {                                               \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));           \
            return 2;                                                          \
        }                                                                      \
    } while (0)

static uint16_t to_bf16(float f) { /* round to nearest even */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}
static uint64_t rng = 88172645463325252ull;
static float uniform_pm1(void) { /* xorshift64 */
    rng ^= rng << 13;
    rng ^= rng >> 7;
    rng ^= rng << 17;
    return (float)((rng >> 11) * (1.0 / 9007199254740992.0)) * 2.f - 1.f;
}

int main(void) {
    const int B = 2, H = 3, N = 333, d = 128;
    const size_t n = (size_t)B * H * N * d, rows = (size_t)B * H * N;
    const float scale = 1.f / sqrtf((float)d);
    uint16_t* hb[4];
    float* hf[4];
    for (int t = 0; t < 4; ++t) {
        hb[t] = malloc(n * 2);
        hf[t] = malloc(n * 4);
        for (size_t i = 0; i < n; ++i) {
            hb[t][i] = to_bf16(2.f * uniform_pm1());
            hf[t][i] = from_bf16(hb[t][i]);
        }
    }
    void *q, *k, *v, *dout, *o, *dq, *dk, *dv, *ws;
    float *qf, *kf, *vf, *of, *lse, *lsef;
    CHECK_CUDA(cudaMalloc(&q, n * 2));
    CHECK_CUDA(cudaMalloc(&k, n * 2));
    CHECK_CUDA(cudaMalloc(&v, n * 2));
    CHECK_CUDA(cudaMalloc(&dout, n * 2));
    CHECK_CUDA(cudaMalloc(&o, n * 2));
    CHECK_CUDA(cudaMalloc(&dq, n * 2));
    CHECK_CUDA(cudaMalloc(&dk, n * 2));
    CHECK_CUDA(cudaMalloc(&dv, n * 2));
    CHECK_CUDA(cudaMalloc((void**)&qf, n * 4));
    CHECK_CUDA(cudaMalloc((void**)&kf, n * 4));
    CHECK_CUDA(cudaMalloc((void**)&vf, n * 4));
    CHECK_CUDA(cudaMalloc((void**)&of, n * 4));
    CHECK_CUDA(cudaMalloc((void**)&lse, rows * 4));
    CHECK_CUDA(cudaMalloc((void**)&lsef, rows * 4));
    void* dev_b[4] = {q, k, v, dout};
    float* dev_f[3] = {qf, kf, vf};
    for (int t = 0; t < 4; ++t) CHECK_CUDA(cudaMemcpy(dev_b[t], hb[t], n * 2, cudaMemcpyHostToDevice));
    for (int t = 0; t < 3; ++t) CHECK_CUDA(cudaMemcpy(dev_f[t], hf[t], n * 4, cudaMemcpyHostToDevice));

    const unsigned long long launches0 = fa_kernel_launches();
    if (fa_fwd(q, k, v, o, lse, B, H, N, d, scale, NULL) != FA_OK) { fprintf(stderr, "fa_fwd: %s\n", fa_last_error_string()); return 1; }
    if (fa_fwd_f32(qf, kf, vf, of, lsef, B, H, N, d, scale, NULL) != FA_OK) { fprintf(stderr, "fa_fwd_f32: %s\n", fa_last_error_string()); return 1; }
    const size_t wsb = fa_bwd_workspace_size(B, H, N, d);
    CHECK_CUDA(cudaMalloc(&ws, wsb));
    if (fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, ws, wsb, NULL) != FA_OK) { fprintf(stderr, "fa_bwd: %s\n", fa_last_error_string()); return 1; }
    if (fa_check_status(NULL) != FA_OK) { fprintf(stderr, "status: %s\n", fa_last_error_string()); return 1; }
    /* fa_fwd: one or two kernels, fa_fwd_f32: one, fa_bwd: three. */
    const unsigned long long launches = fa_kernel_launches() - launches0;
    if (launches < 5 || launches > 6) { fprintf(stderr, "kernel launches: %llu\n", launches); return 1; }

    uint16_t* ho = malloc(n * 2);
    float *hof = malloc(n * 4), *hl = malloc(rows * 4), *hlf = malloc(rows * 4);
    uint16_t* hdq = malloc(n * 2);
    CHECK_CUDA(cudaMemcpy(ho, o, n * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hof, of, n * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hl, lse, rows * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hlf, lsef, rows * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hdq, dq, n * 2, cudaMemcpyDeviceToHost));
    double eo = 0, el = 0;
    int finite = 1;
    for (size_t i = 0; i < n; ++i) {
        eo = fmax(eo, fabs((double)from_bf16(ho[i]) - hof[i]));
        if (!isfinite(from_bf16(hdq[i]))) finite = 0;
    }
    for (size_t i = 0; i < rows; ++i) el = fmax(el, fabs((double)hl[i] - hlf[i]));
    printf("bf16 vs fp32 forward: O max-abs %.3e, LSE max-abs %.3e; dQ finite: %d\n", eo, el, finite);
    if (!(eo <= 2e-2 && el <= 1e-3 && finite)) return 1;

    /* host-side checks: nothing is launched for these */
    if (fa_fwd(NULL, k, v, o, lse, B, H, N, d, scale, NULL) != FA_ERR_INVALID_ARG) return 1;
    if (strstr(fa_last_error_string(), "q is NULL") == NULL) return 1;
    if (fa_fwd(q, k, v, o, lse, B, H, N, 96, scale, NULL) != FA_ERR_UNSUPPORTED) return 1;
    if (fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, ws, wsb - 1, NULL) != FA_ERR_INVALID_ARG) return 1;
    printf("C ABI smoke: ok\n");
    return 0;
}
