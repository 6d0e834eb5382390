/*
 * A caller of librsa written in plain C: only include/rsa.h and the CUDA
 * runtime's C API, no Python and no C++.  It draws seeded bf16 inputs, runs
 * the whole ring (rsa_ring_attn_fwd) on device buffers and the host-to-host
 * call (rsa_ring_attn_fwd_host) on the same inputs, checks an argument error
 * and its message, and writes inputs and results as raw files for the test
 * that compares them with the oracle.
 *
 * usage: c_abi_ring OUTDIR     exit status 0 on success
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "rsa.h"

enum { B = 1, H = 2, T = 1024, D = 128, N = 4, CAUSAL = 1 };
#define ELEMS ((size_t)B * H * T * D)
#define ROWS ((size_t)B * H * T)

static uint32_t lcg_state = 12345u;

/* uniform in [-1, 1) from a 32-bit linear congruential generator */
static float next_uniform(void)
{
    lcg_state = lcg_state * 1664525u + 1013904223u;
    return (float)(lcg_state >> 8) / 8388608.0f - 1.0f;
}

/* fp32 -> bf16 bits, round to nearest even (inputs are finite) */
static uint16_t to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static int write_file(const char *dir, const char *name, const void *p, size_t bytes)
{
    char path[1024];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot write %s\n", path);
        if (f)
            fclose(f);
        return 1;
    }
    fclose(f);
    return 0;
}

#define CUDA_OK(x)                                                               \
    do {                                                                         \
        cudaError_t e_ = (x);                                                    \
        if (e_ != cudaSuccess) {                                                 \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));             \
            return 1;                                                            \
        }                                                                        \
    } while (0)

#define RSA_OK_(x)                                                               \
    do {                                                                         \
        rsa_status s_ = (x);                                                     \
        if (s_ != RSA_OK) {                                                      \
            fprintf(stderr, "%s: %s (%s)\n", #x, rsa_status_string(s_), rsa_last_error_string()); \
            return 1;                                                            \
        }                                                                        \
    } while (0)

int main(int argc, char **argv)
{
    if (argc != 2) {
        fprintf(stderr, "usage: %s OUTDIR\n", argv[0]);
        return 2;
    }
    const char *dir = argv[1];
    uint16_t *hq = malloc(ELEMS * 2), *hk = malloc(ELEMS * 2), *hv = malloc(ELEMS * 2);
    uint16_t *hout = malloc(ELEMS * 2);
    float *hlse = malloc(ROWS * 4);
    if (!hq || !hk || !hv || !hout || !hlse)
        return 1;
    for (size_t i = 0; i < ELEMS; ++i)
        hq[i] = to_bf16(2.0f * next_uniform());
    for (size_t i = 0; i < ELEMS; ++i)
        hk[i] = to_bf16(2.0f * next_uniform());
    for (size_t i = 0; i < ELEMS; ++i)
        hv[i] = to_bf16(next_uniform());

    /* an argument error: N must divide T; nothing is launched and a message is set */
    if (rsa_ring_attn_fwd(NULL, NULL, NULL, RSA_BF16, B, H, T, D, 3, CAUSAL, NULL, NULL, NULL, 0, NULL) !=
            RSA_ERR_INVALID_ARG ||
        strlen(rsa_last_error_string()) == 0) {
        fprintf(stderr, "expected RSA_ERR_INVALID_ARG with a message for N = 3\n");
        return 1;
    }

    void *dq, *dk, *dv, *dout, *dws;
    float *dlse;
    size_t ws_bytes = 0;
    RSA_OK_(rsa_ring_attn_workspace_size(RSA_BF16, B, H, T, D, N, CAUSAL, &ws_bytes));
    CUDA_OK(cudaMalloc(&dq, ELEMS * 2));
    CUDA_OK(cudaMalloc(&dk, ELEMS * 2));
    CUDA_OK(cudaMalloc(&dv, ELEMS * 2));
    CUDA_OK(cudaMalloc(&dout, ELEMS * 2));
    CUDA_OK(cudaMalloc((void **)&dlse, ROWS * 4));
    CUDA_OK(cudaMalloc(&dws, ws_bytes > 0 ? ws_bytes : 1));
    CUDA_OK(cudaMemcpy(dq, hq, ELEMS * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dk, hk, ELEMS * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dv, hv, ELEMS * 2, cudaMemcpyHostToDevice));

    RSA_OK_(rsa_ring_attn_fwd(dq, dk, dv, RSA_BF16, B, H, T, D, N, CAUSAL, dout, dlse, dws, ws_bytes, NULL));
    RSA_OK_(rsa_check_device_error(NULL));
    CUDA_OK(cudaMemcpy(hout, dout, ELEMS * 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hlse, dlse, ROWS * 4, cudaMemcpyDeviceToHost));

    /* the host-to-host call on the same inputs, from page-locked library blocks */
    void *pq, *pk, *pv, *pout, *plse, *dhws;
    size_t hws_bytes = 0;
    RSA_OK_(rsa_host_alloc(ELEMS * 2, &pq));
    RSA_OK_(rsa_host_alloc(ELEMS * 2, &pk));
    RSA_OK_(rsa_host_alloc(ELEMS * 2, &pv));
    RSA_OK_(rsa_host_alloc(ELEMS * 2, &pout));
    RSA_OK_(rsa_host_alloc(ROWS * 4, &plse));
    memcpy(pq, hq, ELEMS * 2);
    memcpy(pk, hk, ELEMS * 2);
    memcpy(pv, hv, ELEMS * 2);
    RSA_OK_(rsa_ring_attn_host_workspace_size(RSA_BF16, B, H, T, D, N, CAUSAL, &hws_bytes));
    CUDA_OK(cudaMalloc(&dhws, hws_bytes)); /* cudaMalloc returns 256-byte-aligned memory */
    RSA_OK_(rsa_ring_attn_fwd_host(pq, pk, pv, RSA_BF16, B, H, T, D, N, CAUSAL, pout, (float *)plse, dhws,
                                   hws_bytes, NULL));
    CUDA_OK(cudaDeviceSynchronize());
    RSA_OK_(rsa_check_device_error(NULL));
    const int host_equal = memcmp(pout, hout, ELEMS * 2) == 0 && memcmp(plse, hlse, ROWS * 4) == 0;

    if (write_file(dir, "q.bin", hq, ELEMS * 2) || write_file(dir, "k.bin", hk, ELEMS * 2) ||
        write_file(dir, "v.bin", hv, ELEMS * 2) || write_file(dir, "out.bin", hout, ELEMS * 2) ||
        write_file(dir, "lse.bin", hlse, ROWS * 4))
        return 1;
    printf("rsa_version %d host_call_bit_exact %d\n", rsa_version(), host_equal);

    RSA_OK_(rsa_host_free(pq));
    RSA_OK_(rsa_host_free(pk));
    RSA_OK_(rsa_host_free(pv));
    RSA_OK_(rsa_host_free(pout));
    RSA_OK_(rsa_host_free(plse));
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dout);
    cudaFree(dlse);
    cudaFree(dws);
    cudaFree(dhws);
    free(hq);
    free(hk);
    free(hv);
    free(hout);
    free(hlse);
    return host_equal ? 0 : 1;
}
