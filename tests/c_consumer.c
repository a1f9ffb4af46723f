/*
 * A plain C11 consumer of libcamp's C ABI (include/camp.h): device buffers come from the
 * CUDA runtime, a stream from cudaStreamCreate, and nothing else is involved (no Python,
 * no torch). It reads its inputs from a file, runs camp_rmsnorm (fp32) and camp_rope
 * (bf16 bit patterns) on a stream of its own, checks a few argument errors, and writes the
 * outputs to a file; tests/test_c_abi_gpu.py compares them with the oracle.
 *
 * Usage: c_consumer IN OUT
 *   IN:  int64 rows, cols, B, S, H, D; float x[rows*cols]; float w[cols];
 *        uint16 q[B*S*H*D] (bf16); float sin[S*D/2]; float cos[S*D/2]
 *   OUT: float y[rows*cols]; uint16 yq[B*S*H*D]
 * Exit status 0 on success; 2 for a file or CUDA error; 3 for an unexpected status.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "camp.h"

static int cuda_ok(cudaError_t e, const char* what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 0;
    }
    return 1;
}

static int expect(camp_status_t got, camp_status_t want, const char* what) {
    if (got != want) {
        fprintf(stderr, "%s: status %d (%s), expected %d\n", what, (int)got,
                camp_status_string(got), (int)want);
        return 0;
    }
    return 1;
}

static void* read_block(FILE* f, size_t bytes) {
    void* p = malloc(bytes ? bytes : 1);
    if (p != NULL && bytes > 0 && fread(p, 1, bytes, f) != bytes) {
        free(p);
        return NULL;
    }
    return p;
}

int main(int argc, char** argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s IN OUT\n", argv[0]);
        return 2;
    }
    FILE* in = fopen(argv[1], "rb");
    if (in == NULL) return 2;
    int64_t dims[6];
    if (fread(dims, sizeof(int64_t), 6, in) != 6) return 2;
    const int64_t rows = dims[0], cols = dims[1], B = dims[2], S = dims[3], H = dims[4],
                  D = dims[5];
    const size_t nx = (size_t)(rows * cols), nq = (size_t)(B * S * H * D),
                 nt = (size_t)(S * (D / 2));
    float* x = read_block(in, nx * sizeof(float));
    float* w = read_block(in, (size_t)cols * sizeof(float));
    uint16_t* q = read_block(in, nq * sizeof(uint16_t));
    float* sn = read_block(in, nt * sizeof(float));
    float* cs = read_block(in, nt * sizeof(float));
    fclose(in);
    if (x == NULL || w == NULL || q == NULL || sn == NULL || cs == NULL) return 2;

    void *dx, *dw, *dy, *dq, *dyq, *dsn, *dcs;
    if (!cuda_ok(cudaMalloc(&dx, nx * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dw, (size_t)cols * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dy, nx * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dq, nq * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dyq, nq * sizeof(uint16_t)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dsn, nt * sizeof(float)), "cudaMalloc") ||
        !cuda_ok(cudaMalloc(&dcs, nt * sizeof(float)), "cudaMalloc"))
        return 2;
    cudaStream_t stream;
    if (!cuda_ok(cudaStreamCreate(&stream), "cudaStreamCreate")) return 2;
    if (!cuda_ok(cudaMemcpyAsync(dx, x, nx * sizeof(float), cudaMemcpyHostToDevice, stream), "copy") ||
        !cuda_ok(cudaMemcpyAsync(dw, w, (size_t)cols * sizeof(float), cudaMemcpyHostToDevice, stream), "copy") ||
        !cuda_ok(cudaMemcpyAsync(dq, q, nq * sizeof(uint16_t), cudaMemcpyHostToDevice, stream), "copy") ||
        !cuda_ok(cudaMemcpyAsync(dsn, sn, nt * sizeof(float), cudaMemcpyHostToDevice, stream), "copy") ||
        !cuda_ok(cudaMemcpyAsync(dcs, cs, nt * sizeof(float), cudaMemcpyHostToDevice, stream), "copy"))
        return 2;

    int ok = 1;
    /* argument errors, reported before any launch */
    ok &= expect(camp_rmsnorm(NULL, dw, dy, rows, cols, 1e-5f, CAMP_DTYPE_F32, (void*)stream),
                 CAMP_ERR_INVALID_ARG, "null x");
    ok &= expect(camp_rmsnorm(dx, dw, dy, rows, cols, -1.0f, CAMP_DTYPE_F32, (void*)stream),
                 CAMP_ERR_INVALID_ARG, "negative eps");
    ok &= expect(camp_rmsnorm(dx, dw, dy, rows, cols, 1e-5f, (camp_dtype_t)7, (void*)stream),
                 CAMP_ERR_UNSUPPORTED_DTYPE, "unknown dtype");
    ok &= expect(camp_rope(dq, dsn, dcs, dyq, B, S, H, D + 1, CAMP_DTYPE_BF16, (void*)stream),
                 CAMP_ERR_INVALID_ARG, "odd head_dim");
    ok &= expect(camp_rmsnorm(NULL, NULL, NULL, 0, cols, 1e-5f, CAMP_DTYPE_F32, (void*)stream),
                 CAMP_SUCCESS, "empty input");
    if (camp_status_string(CAMP_SUCCESS) == NULL) ok = 0;

    /* the two operators, on the caller's stream */
    ok &= expect(camp_rmsnorm(dx, dw, dy, rows, cols, 1e-5f, CAMP_DTYPE_F32, (void*)stream),
                 CAMP_SUCCESS, "camp_rmsnorm");
    ok &= expect(camp_rope(dq, dsn, dcs, dyq, B, S, H, D, CAMP_DTYPE_BF16, (void*)stream),
                 CAMP_SUCCESS, "camp_rope");
    if (!cuda_ok(cudaMemcpyAsync(x, dy, nx * sizeof(float), cudaMemcpyDeviceToHost, stream), "copy") ||
        !cuda_ok(cudaMemcpyAsync(q, dyq, nq * sizeof(uint16_t), cudaMemcpyDeviceToHost, stream), "copy") ||
        !cuda_ok(cudaStreamSynchronize(stream), "cudaStreamSynchronize"))
        return 2;
    uint32_t flags = 1;
    ok &= expect(camp_device_errors(&flags, 0), CAMP_SUCCESS, "camp_device_errors");
    if (flags != 0) ok = 0;

    FILE* out = fopen(argv[2], "wb");
    if (out == NULL || fwrite(x, sizeof(float), nx, out) != nx ||
        fwrite(q, sizeof(uint16_t), nq, out) != nq)
        return 2;
    fclose(out);
    cudaFree(dx);
    cudaFree(dw);
    cudaFree(dy);
    cudaFree(dq);
    cudaFree(dyq);
    cudaFree(dsn);
    cudaFree(dcs);
    cudaStreamDestroy(stream);
    free(x);
    free(w);
    free(q);
    free(sn);
    free(cs);
    return ok ? 0 : 3;
}
