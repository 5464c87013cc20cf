/*
 * c_abi_example.c -- the library used from plain C (no Python, no torch):
 * certify and run the forward on inputs read from files, write O, lse2 and
 * the certificates back.  Built and run by tests/test_gpu_c_abi.py, which
 * writes the inputs and compares the outputs with the oracle.
 *
 *   c_abi_example <dir> B H N d causal [mode]
 *   reads  <dir>/q.bin k.bin v.bin   (bf16 bits, [B, H, N, d] contiguous)
 *   writes <dir>/o.bin (bf16), lse2.bin (fp32), certs.bin (clis_head_cert_t)
 *   mode   fused    clis_certify + clis_attn_fwd (default)
 *          noalloc  clis_certify_noalloc + clis_attn_fwd
 *          chunks   clis_certify, then K/V in three chunks merged by
 *                   clis_attn_fwd_chunk (causal: clis_attn_fwd_chunk_causal,
 *                   chunk offsets as key_offset), then clis_attn_chunk_finalize
 *          fp8      clis_certify + clis_v_to_e4m3 + clis_attn_fwd_fp8pv with
 *                   every head forced onto E4M3 P.V (no mask, d = 128)
 *          host     clis_attention_host on page-locked host buffers with a
 *                   plan of three head groups; the certificates come from the workspace
 *                   (k-bar first, certificates at the next multiple of 256
 *                   bytes) and lse2.bin holds NaN (this path has no lse2)
 * Exit status 0 on success; any CUDA or library error prints a message and
 * exits 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

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
    if (argc != 7 && argc != 8) return fail("usage", "c_abi_example <dir> B H N d causal [mode]");
    const char *dir = argv[1];
    const int64_t B = atol(argv[2]), H = atol(argv[3]), N = atol(argv[4]), d = atol(argv[5]);
    const int causal = atoi(argv[6]);
    const char *mode = argc == 8 ? argv[7] : "fused";
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
    const clis_stream_t cs = (clis_stream_t)stream;
    if (strcmp(mode, "noalloc") == 0)
        CLIS_OK_(clis_certify_noalloc(&s, q, k, v, scale_log2, CLIS_FMT_BF16, CLIS_FMT_FP32, kbar, certs, mu, cs));
    else if (strcmp(mode, "host") != 0)
        CLIS_OK_(clis_certify(&s, q, k, v, scale_log2, CLIS_FMT_BF16, CLIS_FMT_FP32, kbar, certs, mu, ws, ws_bytes,
                              cs));
    if (strcmp(mode, "host") == 0) {
        void *hbuf[4], *hws;
        size_t hws_bytes = 0;
        clis_host_plan_t *plan = NULL;
        CLIS_OK_(clis_host_plan_create(&s, causal, 3, &plan));
        CLIS_OK_(clis_host_plan_workspace_size(plan, &hws_bytes));
        CUDA_OK(cudaMalloc(&hws, hws_bytes));
        for (int t = 0; t < 4; t++) CUDA_OK(cudaMallocHost(&hbuf[t], bytes));
        for (int t = 0; t < 3; t++)
            if (!read_file(dir, names[t], hbuf[t], bytes)) return fail("read", names[t]);
        CLIS_OK_(clis_attention_host(plan, hbuf[0], hbuf[1], hbuf[2], hbuf[3], scale_log2, CLIS_AUTO, hws, hws_bytes,
                                     cs));
        CLIS_OK_(clis_host_plan_wait(plan, cs));
        CUDA_OK(cudaStreamSynchronize(stream));
        CLIS_OK_(clis_host_plan_destroy(plan));
        /* Through the device buffers, so the common code below writes the files. */
        const size_t cert_off = ((size_t)(B * H * d) * sizeof(float) + 255) / 256 * 256;
        CUDA_OK(cudaMemcpy(o, hbuf[3], bytes, cudaMemcpyHostToDevice));
        CUDA_OK(cudaMemcpy(certs, (const char *)hws + cert_off, (size_t)(B * H) * sizeof(clis_head_cert_t),
                           cudaMemcpyDeviceToDevice));
        CUDA_OK(cudaMemset(lse2, 0xff, rows * sizeof(float)));
        for (int t = 0; t < 4; t++) cudaFreeHost(hbuf[t]);
        cudaFree(hws);
    } else if (strcmp(mode, "fused") == 0 || strcmp(mode, "noalloc") == 0) {
        CLIS_OK_(clis_attn_fwd(&s, q, k, v, o, lse2, kbar, certs, mu, scale_log2, causal, CLIS_AUTO, cs));
    } else if (strcmp(mode, "chunks") == 0) {
        /* K/V in three chunks (the split points leave ragged tiles); fp32
         * accumulators O [rows, d], l [rows], m [rows]. */
        float *o_acc, *l_acc, *m_acc;
        CUDA_OK(cudaMalloc((void **)&o_acc, rows * (size_t)d * sizeof(float)));
        CUDA_OK(cudaMalloc((void **)&l_acc, rows * sizeof(float)));
        CUDA_OK(cudaMalloc((void **)&m_acc, rows * sizeof(float)));
        const int64_t cut[4] = {0, N / 3 + 1, 2 * N / 3 + 5, N};
        for (int c = 0; c < 3; c++) {
            clis_shape_t sc = s;
            sc.Nk = cut[c + 1] - cut[c];
            const uint16_t *kc = (const uint16_t *)k + cut[c] * d, *vc = (const uint16_t *)v + cut[c] * d;
            if (causal)
                CLIS_OK_(clis_attn_fwd_chunk_causal(&sc, q, kc, vc, o_acc, l_acc, m_acc, kbar, certs, NULL, mu,
                                                    scale_log2, cut[c], c == 0, CLIS_AUTO, cs));
            else
                CLIS_OK_(clis_attn_fwd_chunk(&sc, q, kc, vc, o_acc, l_acc, m_acc, kbar, certs, mu, scale_log2,
                                             c == 0, CLIS_AUTO, cs));
        }
        CLIS_OK_(clis_attn_chunk_finalize(&s, o_acc, l_acc, m_acc, o, lse2, cs));
        CUDA_OK(cudaStreamSynchronize(stream));
        cudaFree(o_acc);
        cudaFree(l_acc);
        cudaFree(m_acc);
    } else if (strcmp(mode, "fp8") == 0) {
        size_t vt_bytes = 0;
        void *vt8;
        CLIS_OK_(clis_v_e4m3_size(&s, &vt_bytes));
        CUDA_OK(cudaMalloc(&vt8, vt_bytes));
        CLIS_OK_(clis_v_to_e4m3(&s, v, vt8, cs));
        CLIS_OK_(clis_attn_fwd_fp8pv(&s, q, k, v, vt8, o, lse2, kbar, certs, mu, scale_log2, CLIS_CERTIFIED_FORCED,
                                     cs));
        CUDA_OK(cudaStreamSynchronize(stream));
        cudaFree(vt8);
    } else {
        return fail("mode", mode);
    }
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
