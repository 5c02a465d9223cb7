/*
 * Plain-C caller of libattn.so: no Python, no PyTorch.  It reads bf16 Q, K, V
 * (raw bit patterns) from a file, runs attn_fwd through the C ABI on device
 * buffers from cudaMalloc, and writes O and LSE (fp32) to a file.  It also
 * checks that a call with an invalid argument returns ATTN_ERR_INVALID_ARG.
 *
 *   attn_abi_demo <in.bin> <out.bin> B Hq Hkv Sq Sk D causal scale
 *
 * Exit status 0 on success; 1 on a usage or I/O error; 2 on a library or
 * CUDA error.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "attn.h"

static int check_cuda(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 0;
    }
    return 1;
}

int main(int argc, char **argv)
{
    if (argc != 11) {
        fprintf(stderr, "usage: %s in.bin out.bin B Hq Hkv Sq Sk D causal scale\n", argv[0]);
        return 1;
    }
    const int B = atoi(argv[3]), Hq = atoi(argv[4]), Hkv = atoi(argv[5]);
    const int Sq = atoi(argv[6]), Sk = atoi(argv[7]), D = atoi(argv[8]);
    const int causal = atoi(argv[9]);
    const float scale = (float)atof(argv[10]);
    const size_t nq = (size_t)B * Hq * Sq * D, nk = (size_t)B * Hkv * Sk * D;
    const size_t nl = (size_t)B * Hq * Sq;

    unsigned short *h_in = (unsigned short *)malloc(sizeof(unsigned short) * (nq + 2 * nk));
    float *h_out = (float *)malloc(sizeof(float) * (nq + nl));
    if (h_in == NULL || h_out == NULL) return 1;
    FILE *f = fopen(argv[1], "rb");
    if (f == NULL || fread(h_in, sizeof(unsigned short), nq + 2 * nk, f) != nq + 2 * nk) return 1;
    fclose(f);

    void *q = NULL, *k = NULL, *v = NULL;
    float *o = NULL, *lse = NULL;
    if (!check_cuda(cudaMalloc(&q, nq * 2), "cudaMalloc q") ||
        !check_cuda(cudaMalloc(&k, nk * 2), "cudaMalloc k") ||
        !check_cuda(cudaMalloc(&v, nk * 2), "cudaMalloc v") ||
        !check_cuda(cudaMalloc((void **)&o, nq * 4), "cudaMalloc o") ||
        !check_cuda(cudaMalloc((void **)&lse, nl * 4), "cudaMalloc lse"))
        return 2;
    if (!check_cuda(cudaMemcpy(q, h_in, nq * 2, cudaMemcpyHostToDevice), "copy q") ||
        !check_cuda(cudaMemcpy(k, h_in + nq, nk * 2, cudaMemcpyHostToDevice), "copy k") ||
        !check_cuda(cudaMemcpy(v, h_in + nq + nk, nk * 2, cudaMemcpyHostToDevice), "copy v"))
        return 2;

    /* A rejected call launches nothing and reports its status. */
    if (attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, -1.0f, NULL) !=
        ATTN_ERR_INVALID_ARG) {
        fprintf(stderr, "negative scale was not rejected\n");
        return 2;
    }
    const int st = attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, NULL);
    if (st != ATTN_OK) {
        fprintf(stderr, "attn_fwd: %s\n", attn_status_string(st));
        return 2;
    }
    if (!check_cuda(cudaDeviceSynchronize(), "synchronize")) return 2;
    const int dev_status = attn_debug_status(NULL);
    if (dev_status != ATTN_OK) {
        fprintf(stderr, "device status: %s\n", attn_status_string(dev_status));
        return 2;
    }
    if (!check_cuda(cudaMemcpy(h_out, o, nq * 4, cudaMemcpyDeviceToHost), "copy o") ||
        !check_cuda(cudaMemcpy(h_out + nq, lse, nl * 4, cudaMemcpyDeviceToHost), "copy lse"))
        return 2;
    f = fopen(argv[2], "wb");
    if (f == NULL || fwrite(h_out, sizeof(float), nq + nl, f) != nq + nl) return 1;
    fclose(f);
    cudaFree(q);
    cudaFree(k);
    cudaFree(v);
    cudaFree(o);
    cudaFree(lse);
    free(h_in);
    free(h_out);
    printf("attn_abi_demo ok (library version %d.%d)\n", attn_version() >> 16,
           attn_version() & 0xffff);
    return 0;
}
