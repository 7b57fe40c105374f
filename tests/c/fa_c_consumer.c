/*
 * fa_c_consumer.c -- a plain C program that uses the library through include/fa.h
 * only (no Python, no PyTorch): it draws seeded bf16 inputs, runs fa_fwd and
 * fa_bwd on device buffers it allocates itself, and writes inputs and results to
 * a file that tests/test_c_consumer.py checks against the fp64 oracle.
 *
 * Usage: fa_c_consumer OUT_FILE B H H_KV S_Q S_K D CAUSAL
 * Output file: int32 header {B, H, H_kv, S_q, S_k, d, causal}, then the bf16 arrays
 * Q, K, V, dO, O, dQ, dK, dV and the float32 LSE, each in the library layout.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fa.h"

/* float -> bf16 bits, round to nearest even (inputs are finite) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* xorshift64* stream, then a Box-Muller pair per two draws */
static uint64_t g_state = 0x9e3779b97f4a7c15ull;
static double uniform01(void) {
    g_state ^= g_state >> 12;
    g_state ^= g_state << 25;
    g_state ^= g_state >> 27;
    return ((g_state * 0x2545f4914f6cdd1dull) >> 11) * (1.0 / 9007199254740992.0);
}
static float normal(void) {
    double u1 = uniform01(), u2 = uniform01();
    if (u1 < 1e-300) u1 = 1e-300;
    const double two_pi = 6.283185307179586;
    double r = -2.0 * __builtin_log(u1);
    return (float)(__builtin_sqrt(r) * __builtin_cos(two_pi * u2));
}

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 2;                                                              \
        }                                                                          \
    } while (0)
#define CHECK_FA(x)                                                                \
    do {                                                                           \
        int s_ = (x);                                                              \
        if (s_ != FA_OK) {                                                         \
            fprintf(stderr, "%s: status %d: %s\n", #x, s_, fa_last_error());       \
            return 3;                                                              \
        }                                                                          \
    } while (0)

int main(int argc, char** argv) {
    if (argc != 9) {
        fprintf(stderr, "usage: %s OUT B H H_KV S_Q S_K D CAUSAL\n", argv[0]);
        return 1;
    }
    const int B = atoi(argv[2]), H = atoi(argv[3]), H_kv = atoi(argv[4]);
    const int S_q = atoi(argv[5]), S_k = atoi(argv[6]), d = atoi(argv[7]), causal = atoi(argv[8]);
    const size_t nq = (size_t)B * H * S_q * d, nk = (size_t)B * H_kv * S_k * d, nr = (size_t)B * H * S_q;
    uint16_t* hbuf = (uint16_t*)malloc(sizeof(uint16_t) * (4 * nq + 4 * nk));
    float* hlse = (float*)malloc(sizeof(float) * nr);
    if (!hbuf || !hlse) return 1;
    uint16_t *hQ = hbuf, *hK = hQ + nq, *hV = hK + nk, *hdO = hV + nk, *hO = hdO + nq, *hdQ = hO + nq,
             *hdK = hdQ + nq, *hdV = hdK + nk;
    for (size_t i = 0; i < nq; ++i) hQ[i] = to_bf16(normal());
    for (size_t i = 0; i < nk; ++i) hK[i] = to_bf16(normal());
    for (size_t i = 0; i < nk; ++i) hV[i] = to_bf16(normal());
    for (size_t i = 0; i < nq; ++i) hdO[i] = to_bf16(normal());

    void *Q, *K, *V, *dO, *O, *dQ, *dK, *dV;
    float* LSE;
    CHECK_CUDA(cudaMalloc(&Q, 2 * nq));
    CHECK_CUDA(cudaMalloc(&K, 2 * nk));
    CHECK_CUDA(cudaMalloc(&V, 2 * nk));
    CHECK_CUDA(cudaMalloc(&dO, 2 * nq));
    CHECK_CUDA(cudaMalloc(&O, 2 * nq));
    CHECK_CUDA(cudaMalloc(&dQ, 2 * nq));
    CHECK_CUDA(cudaMalloc(&dK, 2 * nk));
    CHECK_CUDA(cudaMalloc(&dV, 2 * nk));
    CHECK_CUDA(cudaMalloc((void**)&LSE, 4 * nr));
    CHECK_CUDA(cudaMemcpy(Q, hQ, 2 * nq, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(K, hK, 2 * nk, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(V, hV, 2 * nk, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dO, hdO, 2 * nq, cudaMemcpyHostToDevice));

    cudaStream_t st;
    CHECK_CUDA(cudaStreamCreate(&st));
    const float scale = 1.0f / __builtin_sqrtf((float)d);
    CHECK_FA(fa_fwd(Q, K, V, O, LSE, B, H, H_kv, S_q, S_k, d, scale, causal, FA_BF16, st));
    CHECK_FA(fa_bwd(dO, Q, K, V, O, LSE, dQ, dK, dV, B, H, H_kv, S_q, S_k, d, scale, causal, FA_BF16, st));
    CHECK_CUDA(cudaStreamSynchronize(st));
    CHECK_FA(fa_check_device(st));
    /* a bad argument is reported, not run */
    if (fa_bwd(dO, Q, K, V, O, LSE, dQ, dK, dV, B, H, H_kv, S_q, S_k, 80, scale, causal, FA_BF16, st) !=
            FA_ERR_UNSUPPORTED ||
        strncmp(fa_last_error(), "d:", 2) != 0) {
        fprintf(stderr, "unsupported head dim not reported\n");
        return 4;
    }

    CHECK_CUDA(cudaMemcpy(hO, O, 2 * nq, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hdQ, dQ, 2 * nq, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hdK, dK, 2 * nk, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hdV, dV, 2 * nk, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hlse, LSE, 4 * nr, cudaMemcpyDeviceToHost));

    FILE* f = fopen(argv[1], "wb");
    if (!f) return 1;
    const int32_t hdr[7] = {B, H, H_kv, S_q, S_k, d, causal};
    fwrite(hdr, sizeof(hdr), 1, f);
    fwrite(hbuf, sizeof(uint16_t), 4 * nq + 4 * nk, f);
    fwrite(hlse, sizeof(float), nr, f);
    fclose(f);

    cudaFree(Q); cudaFree(K); cudaFree(V); cudaFree(dO); cudaFree(O);
    cudaFree(dQ); cudaFree(dK); cudaFree(dV); cudaFree(LSE);
    cudaStreamDestroy(st);
    fa_shutdown();
    free(hbuf);
    free(hlse);
    printf("ok\n");
    return 0;
}
