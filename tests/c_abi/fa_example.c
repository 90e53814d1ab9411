/*
 * A C99 caller of the library: reads q, k, v (16-bit bit patterns) from a
 * file, runs fa_fwd on the GPU and writes O and LSE to another file.
 *   fa_example <in> <out>
 * <in>:  int32 B, H, N, d, causal, dtype; float32 scale; then q, k, v as
 *        uint16 [B, H, N, d] each.
 * <out>: O as uint16 [B, H, N, d], then LSE as float32 [B, H, N].
 * Exit status: 0 on success, 2 on bad input, 3 on a CUDA error, 4 on a
 * library error (the status is printed).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "fa.h"

static int read_all(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n; }

int main(int argc, char** argv) {
    if (argc != 3) return 2;
    FILE* in = fopen(argv[1], "rb");
    if (!in) return 2;
    int32_t hdr[6];
    float scale;
    if (!read_all(in, hdr, sizeof hdr) || !read_all(in, &scale, sizeof scale)) return 2;
    const int B = hdr[0], H = hdr[1], N = hdr[2], d = hdr[3], causal = hdr[4], dtype = hdr[5];
    if (B < 1 || H < 1 || N < 1 || d < 1) return 2;
    const size_t n = (size_t)B * H * N * d, rows = (size_t)B * H * N;
    uint16_t* host = malloc(3 * n * sizeof(uint16_t));
    uint16_t* o_host = malloc(n * sizeof(uint16_t));
    float* lse_host = malloc(rows * sizeof(float));
    if (!host || !o_host || !lse_host || !read_all(in, host, 3 * n * sizeof(uint16_t))) return 2;
    fclose(in);

    void *q, *k, *v, *o;
    float* lse;
    if (cudaMalloc(&q, n * 2) != cudaSuccess || cudaMalloc(&k, n * 2) != cudaSuccess ||
        cudaMalloc(&v, n * 2) != cudaSuccess || cudaMalloc(&o, n * 2) != cudaSuccess ||
        cudaMalloc((void**)&lse, rows * 4) != cudaSuccess)
        return 3;
    if (cudaMemcpy(q, host, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(k, host + n, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(v, host + 2 * n, n * 2, cudaMemcpyHostToDevice) != cudaSuccess)
        return 3;

    int st = fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, NULL);
    if (st == FA_OK) st = fa_check_device_status(NULL);
    if (st != FA_OK) {
        fprintf(stderr, "fa_fwd: %s\n", fa_status_string(st));
        return 4;
    }
    if (cudaMemcpy(o_host, o, n * 2, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(lse_host, lse, rows * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 3;
    FILE* out = fopen(argv[2], "wb");
    if (!out || fwrite(o_host, 2, n, out) != n || fwrite(lse_host, 4, rows, out) != rows) return 3;
    fclose(out);
    printf("fa_example: version %d, %s\n", fa_version(), fa_status_string(st));
    cudaFree(q); cudaFree(k); cudaFree(v); cudaFree(o); cudaFree(lse);
    free(host); free(o_host); free(lse_host);
    return 0;
}
