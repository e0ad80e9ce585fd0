/* abi_demo.c -- the C ABI used from plain C99 (no C++, no Python): allocate
 * device buffers with the CUDA runtime, rotate a slice forward and a
 * gradient backward with rope_partial_inplace_fwd / _bwd on a stream, and
 * write inputs and outputs to a file for the test that checks them against
 * the CPU oracle.  Also exercises the status codes of two invalid calls.
 *
 * Usage: abi_demo OUTPUT_FILE
 * File layout (little-endian): int64 B, S, N, D, start, end; then float32
 * x[B*S*N*D], r1[S*L], r2[S*L], g[B*S*N*D] (inputs), then y, dx (outputs). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "rope_partial.h"

#define CHECK_CUDA(call)                                                     \
    do {                                                                     \
        cudaError_t e_ = (call);                                             \
        if (e_ != cudaSuccess) {                                             \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));      \
            return 2;                                                        \
        }                                                                    \
    } while (0)

/* a deterministic value in (-2, 2) that is exact in fp32 */
static float value(int64_t i, int64_t salt) {
    return (float)((i * 7919 + salt * 104729) % 4001 - 2000) / 1000.0f;
}

int main(int argc, char** argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s OUTPUT_FILE\n", argv[0]);
        return 1;
    }
    const int64_t B = 2, S = 5, N = 3, D = 40, start = 6, end = 38, L = end - start;
    const int64_t nx = B * S * N * D, nr = S * L;
    float* h = (float*)malloc(sizeof(float) * (size_t)(4 * nx + 2 * nr));
    if (!h) return 2;
    float *x = h, *g = h + nx, *r1 = h + 2 * nx, *r2 = h + 2 * nx + nr, *y = h + 2 * nx + 2 * nr,
          *dx = y + nx;
    for (int64_t i = 0; i < nx; ++i) {
        x[i] = value(i, 1);
        g[i] = value(i, 2);
    }
    for (int64_t i = 0; i < nr; ++i) {
        r1[i] = value(i, 3);
        r2[i] = value(i, 4);
    }

    float *dx_d, *dg_d, *dr1, *dr2;
    CHECK_CUDA(cudaMalloc((void**)&dx_d, sizeof(float) * (size_t)nx));
    CHECK_CUDA(cudaMalloc((void**)&dg_d, sizeof(float) * (size_t)nx));
    CHECK_CUDA(cudaMalloc((void**)&dr1, sizeof(float) * (size_t)nr));
    CHECK_CUDA(cudaMalloc((void**)&dr2, sizeof(float) * (size_t)nr));
    CHECK_CUDA(cudaMemcpy(dx_d, x, sizeof(float) * (size_t)nx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dg_d, g, sizeof(float) * (size_t)nx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dr1, r1, sizeof(float) * (size_t)nr, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dr2, r2, sizeof(float) * (size_t)nr, cudaMemcpyHostToDevice));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));

    /* cos/sin of shape (1, S, 1, L): one row per position, broadcast over
       batches and heads (element strides; the stride of a size-1 dim is
       ignored) */
    const int64_t r_shape[4] = {1, S, 1, L};
    const int64_t r_stride[4] = {0, L, 0, 1};
    rope_status_t st = rope_partial_inplace_fwd(dx_d, dr1, dr2, ROPE_FP32, B, S, N, D, r_shape,
                                                r_stride, r_shape, r_stride, start, end,
                                                (rope_stream_t)stream);
    if (st != ROPE_OK) {
        fprintf(stderr, "fwd: %s: %s\n", rope_status_str(st), rope_last_error_message());
        return 3;
    }
    st = rope_partial_inplace_bwd(dg_d, dr1, dr2, ROPE_FP32, B, S, N, D, r_shape, r_stride,
                                  r_shape, r_stride, start, end, (rope_stream_t)stream);
    if (st != ROPE_OK) {
        fprintf(stderr, "bwd: %s: %s\n", rope_status_str(st), rope_last_error_message());
        return 3;
    }
    /* invalid calls change nothing and say why */
    if (rope_partial_inplace_fwd(dx_d, dr1, dr2, ROPE_FP32, B, S, N, D, r_shape, r_stride,
                                 r_shape, r_stride, 5, 38, (rope_stream_t)stream) !=
            ROPE_ERR_INVALID ||
        strstr(rope_last_error_message(), "even") == NULL)
        return 4;
    if (rope_partial_inplace_fwd(NULL, dr1, dr2, ROPE_FP32, B, S, N, D, r_shape, r_stride,
                                 r_shape, r_stride, start, end, (rope_stream_t)stream) !=
        ROPE_ERR_NULLPTR)
        return 4;
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(y, dx_d, sizeof(float) * (size_t)nx, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dx, dg_d, sizeof(float) * (size_t)nx, cudaMemcpyDeviceToHost));

    FILE* f = fopen(argv[1], "wb");
    if (!f) return 2;
    const int64_t hdr[6] = {B, S, N, D, start, end};
    fwrite(hdr, sizeof(int64_t), 6, f);
    fwrite(x, sizeof(float), (size_t)nx, f);
    fwrite(r1, sizeof(float), (size_t)nr, f);
    fwrite(r2, sizeof(float), (size_t)nr, f);
    fwrite(g, sizeof(float), (size_t)nx, f);
    fwrite(y, sizeof(float), (size_t)nx, f);
    fwrite(dx, sizeof(float), (size_t)nx, f);
    fclose(f);
    cudaStreamDestroy(stream);
    cudaFree(dx_d);
    cudaFree(dg_d);
    cudaFree(dr1);
    cudaFree(dr2);
    free(h);
    printf("abi_demo ok\n");
    return 0;
}
