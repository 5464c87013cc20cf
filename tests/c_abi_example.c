/*
 * c_abi_example.c -- the library used from plain C (no Python, no torch):
 * certify and run the fused forward on inputs read from files, write O, lse2
 * and the certificates back.  Built and run by tests/test_gpu_c_abi.py, which
 * writes the inputs and compares the outputs with the oracle.
 *
 *   c_abi_example <dir> B H N d causal
 *   reads  <dir>/q.bin k.bin v.bin   (bf16 bits, [B, H, N, d] contiguous)
 *   writes <dir>/o.bin (bf16), lse2.bin (fp32), certs.bin (clis_head_cert_t)
 * Exit status 0 on success; any CUDA or library error prints a message and
 * exits 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "clis.h"

static int fail(const char *what, const char *msg)
{
    fprintf(stderr, "%s: %s\n", what, msg);
    return 1;
}

static int read_file(const char *dir, const char *name, void *dst, size_t bytes)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return 0;
    size_t n = fread(dst, 1, bytes, f);
    fclose(f);
    return n == bytes;
}

static int write_file(const char *dir, const char *name, const void *src, size_t bytes)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return 0;
    size_t n = fwrite(src, 1, bytes, f);
    fclose(f);
    return n == bytes;
}

#define CUDA_OK(call)                                                   \
    do {                                                                \
        cudaError_t e_ = (call);                                        \
        if (e_ != cudaSuccess) return fail(#call, cudaGetErrorString(e_)); \
    } while (0)

#define CLIS_OK_(call)                                                  \
    do {                                                                \
        clis_status_t s_ = (call);                                      \
        if (s_ != CLIS_OK) return fail(#call, clis_status_string(s_));  \
    } while (0)

int main(int argc, char **argv)
{
    if (argc != 7) return fail("usage", "c_abi_example <dir> B H N d causal");
    const char *dir = argv[1];
    const int64_t B = atol(argv[2]), H = atol(argv[3]), N = atol(argv[4]), d = atol(argv[5]);
    const int causal = atoi(argv[6]);
    const size_t elems = (size_t)(B * H * N * d), bytes = elems * 2, rows = (size_t)(B * H * N);

    clis_shape_t s;
    s.B = B; s.H = H; s.Nq = N; s.Nk = N; s.d = d; s.dtype = CLIS_DT_BF16;
    s.q_sn = s.k_sn = s.v_sn = s.o_sn = d;
    s.q_sh = s.k_sh = s.v_sh = s.o_sh = N * d;
    s.q_sb = s.k_sb = s.v_sb = s.o_sb = H * N * d;

    uint16_t *h_in = (uint16_t *)malloc(bytes);
    if (!h_in) return fail("malloc", "host buffer");
    void *q, *k, *v, *o, *ws;
    float *kbar, *mu, *lse2;
    clis_head_cert_t *certs;
    size_t ws_bytes = 0;
    CLIS_OK_(clis_certify_workspace_size(&s, &ws_bytes));
    CUDA_OK(cudaMalloc(&q, bytes));
    CUDA_OK(cudaMalloc(&k, bytes));
    CUDA_OK(cudaMalloc(&v, bytes));
    CUDA_OK(cudaMalloc(&o, bytes));
    CUDA_OK(cudaMalloc(&ws, ws_bytes ? ws_bytes : 256));
    CUDA_OK(cudaMalloc((void **)&kbar, (size_t)(B * H * d) * sizeof(float)));
    CUDA_OK(cudaMalloc((void **)&mu, rows * sizeof(float)));
    CUDA_OK(cudaMalloc((void **)&lse2, rows * sizeof(float)));
    CUDA_OK(cudaMalloc((void **)&certs, (size_t)(B * H) * sizeof(clis_head_cert_t)));
    const char *names[3] = {"q.bin", "k.bin", "v.bin"};
    void *dev[3] = {q, k, v};
    for (int t = 0; t < 3; t++) {
        if (!read_file(dir, names[t], h_in, bytes)) return fail("read", names[t]);
        CUDA_OK(cudaMemcpy(dev[t], h_in, bytes, cudaMemcpyHostToDevice));
    }

    cudaStream_t stream;
    CUDA_OK(cudaStreamCreate(&stream));
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)d);  /* log2(e) / sqrt(d) */
    CLIS_OK_(clis_certify(&s, q, k, v, scale_log2, CLIS_FMT_BF16, CLIS_FMT_FP32, kbar, certs, mu, ws, ws_bytes,
                          (clis_stream_t)stream));
    CLIS_OK_(clis_attn_fwd(&s, q, k, v, o, lse2, kbar, certs, mu, scale_log2, causal, CLIS_AUTO,
                           (clis_stream_t)stream));
    CUDA_OK(cudaStreamSynchronize(stream));
    uint32_t code = 0;
    if (clis_get_device_error(&code) != CLIS_OK || code != 0) return fail("device error word", "set");

    float *h_lse = (float *)malloc(rows * sizeof(float));
    clis_head_cert_t *h_certs = (clis_head_cert_t *)malloc((size_t)(B * H) * sizeof(clis_head_cert_t));
    if (!h_lse || !h_certs) return fail("malloc", "host outputs");
    CUDA_OK(cudaMemcpy(h_in, o, bytes, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(h_lse, lse2, rows * sizeof(float), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(h_certs, certs, (size_t)(B * H) * sizeof(clis_head_cert_t), cudaMemcpyDeviceToHost));
    if (!write_file(dir, "o.bin", h_in, bytes) || !write_file(dir, "lse2.bin", h_lse, rows * sizeof(float)) ||
        !write_file(dir, "certs.bin", h_certs, (size_t)(B * H) * sizeof(clis_head_cert_t)))
        return fail("write", "outputs");
    int n_cert = 0;
    for (int64_t h = 0; h < B * H; h++) n_cert += h_certs[h].certified;
    printf("ok: %d of %lld heads certified\n", n_cert, (long long)(B * H));
    cudaStreamDestroy(stream);
    return 0;
}
