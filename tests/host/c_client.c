/*
 * c_client.c -- a plain C11 caller of librepops through include/repops.h: no
 * Python, no PyTorch, device memory from the CUDA runtime.  Test helper.
 *
 * Integer-valued operands keep every partial sum exact in binary32, so the
 * expected results are closed forms computed here:
 *   - GEMM ("Verde与RepOps" §3.2): C[i][j] = sum_k A[i][k] * B[k][j] over a
 *     ragged 300 x 200 x 777 problem, |sum| < 2^24, with B row-major and
 *     stored transposed, and a 1100 x 1000 x 600 one whose scratch (the
 *     transposed B copied) comes from a caller workspace;
 *   - mean + SGD ("Zoo Per-LLM Chain Soundness" §5): four contributors (the
 *     divide by 4 is exact), eta = 1/16, in the order repops_sort_ids gives
 *     for four DIDs of different lengths;
 *   - the host-buffer GEMM on buffers from repops_host_alloc;
 *   - the Merkle root of C's bytes (4096-byte leaves, a short last leaf) is
 *     printed for the caller to compare with the oracle's.
 * Prints "ok <root hex>" and exits 0, else the first mismatch and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "repops.h"

#define CUDA_OK(x)                                                             \
    do {                                                                       \
        cudaError_t e_ = (x);                                                  \
        if (e_ != cudaSuccess) {                                               \
            printf("CUDA error %d in %s\n", (int)e_, #x);                      \
            return 1;                                                          \
        }                                                                      \
    } while (0)

#define REPOPS_OK_(x)                                                          \
    do {                                                                       \
        int r_ = (x);                                                          \
        if (r_ != REPOPS_OK) {                                                 \
            printf("%s returned %d (%s)\n", #x, r_, repops_status_string(r_)); \
            return 1;                                                          \
        }                                                                      \
    } while (0)

/* small integers in [-4, 4] */
static float val(int64_t i, int64_t j, unsigned salt) {
    return (float)((int)((uint64_t)(i * 7 + j * 13 + salt) % 9u) - 4);
}

static int check_gemm(const float *C, int64_t M, int64_t N, int64_t K, const char *what) {
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)val(i, k, 1) * (int64_t)val(k, j, 2);
            if (C[i * N + j] != (float)s) {
                printf("%s: C[%lld][%lld] = %.9g, want %lld\n", what, (long long)i, (long long)j,
                       (double)C[i * N + j], (long long)s);
                return 1;
            }
        }
    return 0;
}

int main(void) {
    const int64_t M = 300, N = 200, K = 777;
    float *hA = malloc(sizeof(float) * M * K), *hB = malloc(sizeof(float) * K * N);
    float *hBt = malloc(sizeof(float) * N * K), *hC = malloc(sizeof(float) * M * N);
    if (!hA || !hB || !hBt || !hC) return 1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) hA[i * K + k] = val(i, k, 1);
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) hB[k * N + j] = hBt[j * K + k] = val(k, j, 2);

    cudaStream_t s;
    CUDA_OK(cudaStreamCreate(&s));
    float *dA, *dB, *dBt, *dC;
    CUDA_OK(cudaMalloc((void **)&dA, sizeof(float) * M * K));
    CUDA_OK(cudaMalloc((void **)&dB, sizeof(float) * K * N));
    CUDA_OK(cudaMalloc((void **)&dBt, sizeof(float) * N * K));
    CUDA_OK(cudaMalloc((void **)&dC, sizeof(float) * M * N));
    CUDA_OK(cudaMemcpy(dA, hA, sizeof(float) * M * K, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dB, hB, sizeof(float) * K * N, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dBt, hBt, sizeof(float) * N * K, cudaMemcpyHostToDevice));

    /* GEMM, B row-major, then B stored transposed */
    REPOPS_OK_(repops_gemm_f32(M, N, K, dA, K, dB, N, dC, N, s));
    CUDA_OK(cudaMemcpyAsync(hC, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    if (check_gemm(hC, M, N, K, "repops_gemm_f32")) return 1;
    CUDA_OK(cudaMemset(dC, 0xff, sizeof(float) * M * N));
    REPOPS_OK_(repops_gemm_f32_ex(0, 1, M, N, K, dA, K, dBt, K, dC, N, s));
    CUDA_OK(cudaMemcpyAsync(hC, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    if (check_gemm(hC, M, N, K, "repops_gemm_f32_ex (B transposed)")) return 1;

    /* a larger product with B stored transposed: its scratch (B copied into the
     * kernels' row-major layout) from a workspace of the caller's */
    {
        const int64_t M2 = 1100, N2 = 1000, K2 = 600;
        float *hA2 = malloc(sizeof(float) * M2 * K2), *hBt2 = malloc(sizeof(float) * N2 * K2);
        float *hC2 = malloc(sizeof(float) * M2 * N2);
        if (!hA2 || !hBt2 || !hC2) return 1;
        for (int64_t i = 0; i < M2; ++i)
            for (int64_t k = 0; k < K2; ++k) hA2[i * K2 + k] = val(i, k, 1);
        for (int64_t j = 0; j < N2; ++j)
            for (int64_t k = 0; k < K2; ++k) hBt2[j * K2 + k] = val(k, j, 2);
        float *dA2, *dBt2, *dC2;
        void *ws;
        CUDA_OK(cudaMalloc((void **)&dA2, sizeof(float) * M2 * K2));
        CUDA_OK(cudaMalloc((void **)&dBt2, sizeof(float) * N2 * K2));
        CUDA_OK(cudaMalloc((void **)&dC2, sizeof(float) * M2 * N2));
        CUDA_OK(cudaMemcpy(dA2, hA2, sizeof(float) * M2 * K2, cudaMemcpyHostToDevice));
        CUDA_OK(cudaMemcpy(dBt2, hBt2, sizeof(float) * N2 * K2, cudaMemcpyHostToDevice));
        const uint64_t need = repops_gemm_workspace_bytes(0, 1, M2, N2, K2, dA2, K2, dBt2, K2);
        if (need == 0) {
            printf("repops_gemm_workspace_bytes: 0 for a transposed B of %lld GFLOP\n",
                   (long long)(2 * M2 * N2 * K2 / 1000000000));
            return 1;
        }
        CUDA_OK(cudaMalloc(&ws, need));
        REPOPS_OK_(repops_gemm_f32_ws(0, 1, M2, N2, K2, dA2, K2, dBt2, K2, dC2, N2, ws, need, s));
        CUDA_OK(cudaMemcpyAsync(hC2, dC2, sizeof(float) * M2 * N2, cudaMemcpyDeviceToHost, s));
        CUDA_OK(cudaStreamSynchronize(s));
        if (check_gemm(hC2, M2, N2, K2, "repops_gemm_f32_ws (B transposed)")) return 1;
        cudaFree(dA2); cudaFree(dBt2); cudaFree(dC2); cudaFree(ws);
        free(hA2); free(hBt2); free(hC2);
    }

    /* the host-buffer GEMM on buffers from the library's host allocator */
    {
        float *pA = NULL, *pB = NULL, *pC = NULL;
        REPOPS_OK_(repops_host_alloc(sizeof(float) * M * K, (void **)&pA));
        REPOPS_OK_(repops_host_alloc(sizeof(float) * K * N, (void **)&pB));
        REPOPS_OK_(repops_host_alloc(sizeof(float) * M * N, (void **)&pC));
        memcpy(pA, hA, sizeof(float) * M * K);
        memcpy(pB, hB, sizeof(float) * K * N);
        REPOPS_OK_(repops_gemm_f32_host(M, N, K, pA, K, pB, N, pC, N, s));
        CUDA_OK(cudaStreamSynchronize(s));
        if (check_gemm(pC, M, N, K, "repops_gemm_f32_host (repops_host_alloc buffers)")) return 1;
        REPOPS_OK_(repops_host_free(pA));
        REPOPS_OK_(repops_host_free(pB));
        REPOPS_OK_(repops_host_free(pC));
        if (repops_host_free(pC) != REPOPS_ERR_INVALID_ARG) {
            printf("repops_host_free accepted a pointer freed already\n");
            return 1;
        }
    }

    /* contributor order: DIDs compared as unsigned bytes, a proper prefix first */
    const uint8_t ids[] = {0xb0, 0x01, /* 0: b0 01 */ 0x7f, /* 1: 7f */ 0xb0, /* 2: b0 */ 0x80, 0x00 /* 3: 80 00 */};
    const int64_t offsets[4] = {0, 2, 3, 4}, lengths[4] = {2, 1, 1, 2};
    int order[4];
    REPOPS_OK_(repops_sort_ids(4, ids, offsets, lengths, order));
    const int want_order[4] = {1, 3, 2, 0};
    for (int r = 0; r < 4; ++r)
        if (order[r] != want_order[r]) {
            printf("repops_sort_ids: position %d holds %d, want %d\n", r, order[r], want_order[r]);
            return 1;
        }

    /* mean + SGD over four contributors */
    const int64_t len = 1001;
    float *hg = malloc(sizeof(float) * 4 * len), *ht = malloc(sizeof(float) * len);
    if (!hg || !ht) return 1;
    for (int r = 0; r < 4; ++r)
        for (int64_t e = 0; e < len; ++e) hg[r * len + e] = val(e, r, 3);
    for (int64_t e = 0; e < len; ++e) ht[e] = val(e, 5, 4);
    float *dg, *dt;
    CUDA_OK(cudaMalloc((void **)&dg, sizeof(float) * 4 * len));
    CUDA_OK(cudaMalloc((void **)&dt, sizeof(float) * len));
    CUDA_OK(cudaMemcpy(dg, hg, sizeof(float) * 4 * len, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dt, ht, sizeof(float) * len, cudaMemcpyHostToDevice));
    const float *ptrs[4] = {dg, dg + len, dg + 2 * len, dg + 3 * len};
    REPOPS_OK_(repops_fixed_order_mean_sgd(4, len, ptrs, order, 0.0625f, dt, s));
    float *got = malloc(sizeof(float) * len);
    if (!got) return 1;
    CUDA_OK(cudaMemcpyAsync(got, dt, sizeof(float) * len, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    for (int64_t e = 0; e < len; ++e) {
        /* every step exact: integer sums, a divide by 4 and a multiply by 1/16 */
        float S = hg[order[0] * len + e];
        for (int r = 1; r < 4; ++r) S += hg[order[r] * len + e];
        const float want = ht[e] - 0.0625f * (S / 4.0f);
        if (got[e] != want) {
            printf("mean + SGD: theta[%lld] = %.9g, want %.9g\n", (long long)e, (double)got[e], (double)want);
            return 1;
        }
    }

    /* Merkle root of C's bytes */
    uint8_t *droot, root[32];
    CUDA_OK(cudaMalloc((void **)&droot, 32));
    REPOPS_OK_(repops_merkle_sha256(dC, (uint64_t)(sizeof(float) * M * N), 4096, droot, s));
    CUDA_OK(cudaMemcpyAsync(root, droot, 32, cudaMemcpyDeviceToHost, s));
    int status = 0;
    REPOPS_OK_(repops_device_status(s, &status));
    if (status != REPOPS_OK) {
        printf("device status %d (%s)\n", status, repops_status_string(status));
        return 1;
    }
    printf("ok ");
    for (int b = 0; b < 32; ++b) printf("%02x", root[b]);
    printf("\n");

    cudaFree(dA); cudaFree(dB); cudaFree(dBt); cudaFree(dC);
    cudaFree(dg); cudaFree(dt); cudaFree(droot);
    cudaStreamDestroy(s);
    free(hA); free(hB); free(hBt); free(hC); free(hg); free(ht); free(got);
    return 0;
}
