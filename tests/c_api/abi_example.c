/* Using libgemm_f32 from plain C (C99): device buffers, one product on a
 * stream, the status check, and an exact check of the result on small
 * integers (every partial sum is exact in fp32 and TF32, so all modes must
 * match a host triple loop bit for bit).  Prints "ok <kernel>" per mode and
 * returns 0, or prints the first mismatch and returns 1. */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "gemm_f32.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 1;                                                              \
        }                                                                          \
    } while (0)

int main(int argc, char** argv) {
    const int M = argc > 1 ? atoi(argv[1]) : 300;
    const int K = argc > 2 ? atoi(argv[2]) : 200;
    const int N = argc > 3 ? atoi(argv[3]) : 260;
    float* hA = (float*)malloc(sizeof(float) * M * K);
    float* hB = (float*)malloc(sizeof(float) * K * N);
    float* hC = (float*)malloc(sizeof(float) * M * N);
    if (!hA || !hB || !hC) return 1;
    for (int i = 0; i < M * K; ++i) hA[i] = (float)((i * 7 + 3) % 17 - 8);
    for (int i = 0; i < K * N; ++i) hB[i] = (float)((i * 5 + 1) % 13 - 6);

    float *dA, *dB, *dC;
    cudaStream_t s;
    CHECK_CUDA(cudaMalloc((void**)&dA, sizeof(float) * M * K));
    CHECK_CUDA(cudaMalloc((void**)&dB, sizeof(float) * K * N));
    CHECK_CUDA(cudaMalloc((void**)&dC, sizeof(float) * M * N));
    CHECK_CUDA(cudaStreamCreate(&s));
    CHECK_CUDA(cudaMemcpy(dA, hA, sizeof(float) * M * K, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dB, hB, sizeof(float) * K * N, cudaMemcpyHostToDevice));

    printf("%s\n", gemm_f32_version());
    const int modes[3] = {GEMM_F32_MODE_TC3X, GEMM_F32_MODE_FFMA, GEMM_F32_MODE_TC1X};
    for (int m = 0; m < 3; ++m) {
        /* flag SINGLE_CTA keeps the mode's own kernels even for small sizes */
        int rc = gemm_f32_ex(dA, dB, dC, M, N, K, modes[m], GEMM_F32_FLAG_SINGLE_CTA,
                             (gemm_f32_stream_t)s);
        if (rc != GEMM_F32_OK) {
            fprintf(stderr, "gemm_f32_ex: %d\n", rc);
            return 1;
        }
        unsigned site = 0;
        rc = gemm_f32_status((gemm_f32_stream_t)s, &site);
        if (rc != GEMM_F32_OK) {
            fprintf(stderr, "gemm_f32_status: %d (site %u)\n", rc, site);
            return 1;
        }
        const char* kernel = gemm_f32_last_kernel();
        CHECK_CUDA(cudaMemcpy(hC, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost));
        for (int i = 0; i < M; ++i)
            for (int j = 0; j < N; ++j) {
                long long acc = 0;
                for (int k = 0; k < K; ++k) acc += (long long)hA[i * K + k] * (long long)hB[k * N + j];
                if (hC[i * N + j] != (float)acc) {
                    fprintf(stderr, "mode %d: C[%d][%d] = %g, want %lld\n", modes[m], i, j,
                            hC[i * N + j], acc);
                    return 1;
                }
            }
        printf("ok %s\n", kernel);
    }
    /* the default entry point with the legacy default stream */
    if (gemm_f32(dA, dB, dC, M, N, K, 0) != GEMM_F32_OK) return 1;
    if (gemm_f32_status(0, NULL) != GEMM_F32_OK) return 1;
    printf("ok gemm_f32\n");
    gemm_f32_release();
    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dC);
    cudaStreamDestroy(s);
    free(hA);
    free(hB);
    free(hC);
    return 0;
}
