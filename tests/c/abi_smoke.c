/*
 * abi_smoke.c -- liblse called from plain C, with no Python and no torch:
 * device buffers from the CUDA runtime, one lse_forward call and one
 * lse_forward16 call.
 *
 * Usage: abi_smoke <dtype 0=f32|1=bf16|2=f16> <B> <N> <seed> <x_out_path>
 * Writes the raw input elements it generated to x_out_path and prints, per
 * row, the lse_forward and the lse_forward16 results (%.9g %.9g), so a test
 * can check them against the oracle.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "lse.h"

static uint32_t lcg(uint64_t *s)
{
    *s = *s * 6364136223846793005ULL + 1442695040888963407ULL;
    return (uint32_t)(*s >> 33);
}

int main(int argc, char **argv)
{
    if (argc != 6) {
        fprintf(stderr, "usage: %s dtype B N seed x_out_path\n", argv[0]);
        return 2;
    }
    const int dt = atoi(argv[1]);
    const int64_t B = atoll(argv[2]), N = atoll(argv[3]);
    uint64_t s = (uint64_t)atoll(argv[4]);
    const size_t eb = dt == 0 ? 4 : 2, n = (size_t)(B * N);
    unsigned char *h = malloc(n * eb + 1);
    float *out = malloc((size_t)B * sizeof(float) + 1);
    float *out16 = malloc((size_t)B * sizeof(float) + 1);
    if (!h || !out || !out16)
        return 3;
    for (size_t i = 0; i < n; ++i) {
        const uint32_t r = lcg(&s);
        if (dt == 0) {
            const float v = ((float)(r % 65536u) - 32768.0f) / 2048.0f; /* [-16, 16) */
            memcpy(h + 4 * i, &v, 4);
        } else {
            /* sign, exponent field and mantissa of a moderate finite value */
            uint16_t bits;
            if (dt == 1)
                bits = (uint16_t)(((r & 1u) << 15) | ((117u + (r >> 1) % 14u) << 7) | ((r >> 8) & 0x7fu));
            else
                bits = (uint16_t)(((r & 1u) << 15) | ((5u + (r >> 1) % 14u) << 10) | ((r >> 8) & 0x3ffu));
            memcpy(h + 2 * i, &bits, 2);
        }
    }
    FILE *f = fopen(argv[5], "wb");
    if (!f || fwrite(h, eb, n, f) != n)
        return 4;
    fclose(f);

    void *dx = NULL;
    float *dout = NULL;
    if (cudaMalloc(&dx, n * eb) != cudaSuccess || cudaMalloc((void **)&dout, (size_t)B * 4) != cudaSuccess)
        return 5;
    if (cudaMemcpy(dx, h, n * eb, cudaMemcpyHostToDevice) != cudaSuccess)
        return 6;
    const lse_status st = lse_forward(dx, (lse_dtype)dt, B, N, N, dout, NULL);
    if (st != LSE_OK) {
        fprintf(stderr, "lse_forward: %s\n", lse_status_string(st));
        return 7;
    }
    if (cudaMemcpy(out, dout, (size_t)B * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 8;
    const lse_status st16 = lse_forward16(dx, (lse_dtype)dt, B, N, N, dout, NULL, NULL);
    if (st16 != LSE_OK) {
        fprintf(stderr, "lse_forward16: %s\n", lse_status_string(st16));
        return 9;
    }
    if (cudaMemcpy(out16, dout, (size_t)B * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 10;
    for (int64_t b = 0; b < B; ++b)
        printf("%.9g %.9g\n", out[b], out16[b]);
    cudaFree(dx);
    cudaFree(dout);
    free(h);
    free(out);
    free(out16);
    return 0;
}
