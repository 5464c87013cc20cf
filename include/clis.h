/*
 * clis.h -- C ABI of the CLiS attention library (libclis.so), sm_103a.
 *
 * CLiS ("CLiS: Plug-and-Play Attention Acceleration for Video Diffusion on
 * TPUs via Certified Stabilization", Tsai et al., 2026) fixes one softmax
 * stabiliser per query row before the KV loop, so the fused attention kernel
 * needs no running row maximum and no accumulator rescaling.  A per-head
 * certificate (Algorithm 1) proves that doing so cannot overflow; heads that
 * fail certification run standard online softmax instead (abstract).
 *
 * Conventions shared by every entry point:
 *  - Tensors are bf16 (or fp16, shape->dtype) in layout [B, H, N, d] with
 *    element strides given in clis_shape_t; the d dimension is contiguous.
 *  - Device pointers must be 16-byte aligned and every stride (n, h, b) a
 *    multiple of 8 elements (16 bytes); otherwise CLIS_ERR_MISALIGNED.
 *  - d must be 64 or 128 (CLIS_ERR_UNSUPPORTED otherwise).
 *  - The caller owns every buffer.  The library allocates no device memory;
 *    scratch space is passed in as `workspace`.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise the host.  The returned status
 *    covers argument checks and launch errors only: on any argument error
 *    nothing is launched.  Faults found inside a kernel (a pipeline wait
 *    that exceeded its time limit) are recorded in a device-side error word
 *    read by clis_get_device_error().
 *  - All results are deterministic: every floating-point sum has a fixed
 *    order.  (The one place that adds through memory, the KV-chunk merge of
 *    certified heads, adds one value per accumulator element per launch, so
 *    the order is the launch order.  The certification combines partial
 *    maxima with atomic max operations, which are exact in any order.)
 */
#ifndef CLIS_H
#define CLIS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CLIS_API __attribute__((visibility("default")))
#else
#define CLIS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle, ABI-compatible with cudaStream_t. */
typedef struct CUstream_st *clis_stream_t;

typedef enum {
    CLIS_OK = 0,
    CLIS_ERR_INVALID_ARG = 1,  /* null pointer, negative/zero size, bad enum or dtype, non-finite or <= 0 scale */
    CLIS_ERR_UNSUPPORTED = 2,  /* head dim not in {64, 128}, causal with Nq != Nk, sizes beyond int32 */
    CLIS_ERR_MISALIGNED = 3,   /* pointer not 16-byte aligned or stride not a multiple of 8 elements */
    CLIS_ERR_WORKSPACE = 4,    /* workspace null or smaller than clis_certify_workspace_size() */
    CLIS_ERR_CUDA = 5,         /* a CUDA runtime/driver call or a kernel launch failed */
    CLIS_ERR_TIMEOUT = 6       /* a kernel pipeline wait exceeded its limit (device error word) */
} clis_status_t;

/* Floating-point formats whose exp2 overflow limits Figure 3 tabulates (FP16,
 * BF16, FP32).  U_exp and U_acc of Algorithm 1 step 7 are those limits for
 * the format holding exp2 outputs and for the accumulator format. */
typedef enum { CLIS_FMT_FP16 = 0, CLIS_FMT_BF16 = 1, CLIS_FMT_FP32 = 2 } clis_fmt_t;

/* Which softmax the attention kernel runs per head:
 *  CLIS_AUTO              certified heads use the fixed stabiliser, the rest
 *                         fall back to online softmax (the fallback the
 *                         abstract describes for heads that fail);
 *  CLIS_ONLINE            every head uses online softmax that rescales the
 *                         accumulator after every KV block (the baseline);
 *  CLIS_CERTIFIED_FORCED  every head uses the fixed stabiliser, ignoring the
 *                         flags (benchmarks and tests only: output of a head
 *                         that did not certify is then unspecified);
 *  CLIS_ONLINE_LAZY       every head uses online softmax that rescales only
 *                         when a row maximum grows by more than 8 (exp2 units),
 *                         the FlashAttention-4-style baseline the paper adapts
 *                         as "FA4-style (row)" (Tables 5 and 8); needs no
 *                         certificate. */
typedef enum {
    CLIS_AUTO = 0,
    CLIS_ONLINE = 1,
    CLIS_CERTIFIED_FORCED = 2,
    CLIS_ONLINE_LAZY = 3
} clis_variant_t;

/* Element type of Q, K, V and O (all four share it).  The attention kernel
 * feeds P to the tensor cores in the same type, so with FP16 data the exp2
 * outputs are FP16 (Figure 3: U_exp = 15.9993): certify FP16 data with
 * exp_fmt = CLIS_FMT_FP16.  As a safeguard, in CLIS_AUTO an FP16 head takes the
 * fixed-stabiliser path only if its certificate also satisfies
 * B_h <= min(15, C); otherwise it runs online softmax. */
typedef enum { CLIS_DT_BF16 = 0, CLIS_DT_FP16 = 1 } clis_dtype_t;

/* Problem shape and element strides (elements, not bytes).  K and V share
 * Nk; Q and O share Nq.  O strides are ignored by clis_certify.  dtype is a
 * clis_dtype_t (0 = BF16, the zero-initialised default).
 *
 * Strides are non-negative, n-strides at least d.  A head or batch stride of
 * 0 on K and V makes the heads (or batches) read one K/V head: grouped-query
 * and multi-query attention map onto it by folding the key/value heads into
 * the batch (B' = B * H_kv, H' = query heads per key/value head, K and V
 * head stride 0, batch stride one K/V head).  Each query head is then
 * certified against the shared keys and values like any other head.  Strides
 * of anything written must not make two elements share an address: an O (or,
 * in the backward, dQ, dK, dV) head stride of 0 with H > 1 or batch stride of
 * 0 with B > 1 is CLIS_ERR_INVALID_ARG, with one exception: the backward
 * writes dK and dV with the K and V strides, and when K and V are broadcast
 * over the heads together (both head strides 0) it sums the gradients of all
 * H query heads into each dK and dV row and writes it once. */
typedef struct {
    int64_t B, H, Nq, Nk, d;
    int64_t q_sb, q_sh, q_sn;
    int64_t k_sb, k_sh, k_sn;
    int64_t v_sb, v_sh, v_sn;
    int64_t o_sb, o_sh, o_sn;
    int64_t dtype;
} clis_shape_t;

/* Per-head certificate, Algorithm 1 (one per (b, h) pair, index b*H + h).
 *  certified  1 if every input of the head is finite and B_h <= C
 *  G          step 5: ceil(log2 max(1, max |V|))
 *  A          step 6: ceil(log2 Nk) + G
 *  C          step 7: min(floor(U_exp), ceil(U_acc - A) - 1)
 *  reason     0 certified, 1 B_h > C, 2 a non-finite value in Q, K or V
 *             (then G = A = C = 0 and B_h = +inf)
 *  B_h        step 4 with BoundUp(q, kappa) = scale_log2 * ||q||_2 * kappa,
 *             rounded upward (exp2-argument units)
 *  kappa      step 3: an upper bound on max_r ||k_r - kbar||_2 computed
 *             with upward rounding about the kbar returned by clis_certify
 *  qmax       an upper bound on max_r ||q_r||_2 */
typedef struct {
    int32_t certified, G, A, C, reason;
    float B_h, kappa, qmax;
} clis_head_cert_t;

/* Bytes of device workspace clis_certify needs for this shape.
 * Host-only; never touches the GPU.  Errors: CLIS_ERR_INVALID_ARG for a
 * null argument or a negative size. */
CLIS_API clis_status_t clis_certify_workspace_size(const clis_shape_t *shape, size_t *bytes);

/* Certification pre-pass, Algorithm 1 steps 1-7 plus the decision, for all
 * B*H heads (Algorithm 1 certifies one dense attention head; here every
 * (b, h) pair is one such head).  The decision after step 7 is lost from the
 * text; it is read here as: every input finite and B_h <= C.
 *   q, k, v     device bf16 [B,H,Nq,d] / [B,H,Nk,d] / [B,H,Nk,d]
 *   scale_log2  softmax scale times log2(e) (> 0, finite); scores enter
 *               exp2 as scale_log2 * q.k
 *   exp_fmt     format that holds exp2 outputs (U_exp); the attention
 *               kernel feeds P to the tensor cores as BF16
 *   acc_fmt     accumulator format (U_acc); the kernel accumulates in FP32
 *   kbar        device fp32 out [B*H, d]: step 1 key mean, round-to-nearest
 *   certs       device out [B*H]
 *   mu          optional device fp32 out [B*H*Nq] (index (b*H + h)*Nq + i):
 *               the per-row stabilisers mu_i = scale_log2 * (q_i . kbar) that
 *               the certified path fixes before the KV loop (Figure 5(a));
 *               pass it to clis_attn_fwd so the kernel need not recompute
 *               them.  NULL = skip.
 *   workspace   device scratch of at least clis_certify_workspace_size()
 *               bytes, 256-byte aligned; contents need no initialisation
 * Launches four kernels on `stream`.  Nk must be >= 1; Nq may be 0. */
CLIS_API clis_status_t clis_certify(const clis_shape_t *shape, const void *q, const void *k,
                           const void *v, float scale_log2, clis_fmt_t exp_fmt,
                           clis_fmt_t acc_fmt, float *kbar, clis_head_cert_t *certs,
                           float *mu, void *workspace, size_t ws_bytes, clis_stream_t stream);

/* Size in bytes of the scratch buffer that clis_certify_noalloc uses instead
 * of a caller workspace (a fixed array inside the library). */
#define CLIS_NOALLOC_SCRATCH_BYTES (4u << 20)

/* clis_certify for callers that must not allocate device memory.  The paper
 * has no counterpart to this entry point: it exists for code that runs where
 * cudaMalloc is off limits -- a plugin or custom operator inside another
 * runtime that owns all device memory and hands out no workspace, a serving
 * loop whose memory was planned up front, or any caller for whom an
 * allocation would synchronise the device or break the host's accounting.
 *
 * Same arguments and results as clis_certify minus the workspace: the
 * scratch lives in one library-owned device array of
 * CLIS_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library keeps
 * until the process exits.  The caller still provides q, k, v, kbar and
 * certs.  Nothing is allocated or freed, by this call or by any routine it
 * uses.
 *   - The first call on a device (with that device current) does the set-up:
 *     it looks up the array's device address with cudaGetSymbolAddress (which
 *     allocates nothing).  Make that first call before any stream capture on
 *     that device.  Later calls made outside capture repeat the lookup in the
 *     current context, so a device reset or another context gets its own
 *     address; a call made while `stream` is being captured does no lookup and
 *     uses the address of the last lookup in the same context (CLIS_ERR_CUDA
 *     if there was none).
 *   - All calls share the one array and it keeps what the last call left in
 *     it.  The kernels overwrite every scratch word they read, so nothing
 *     needs clearing between calls, but calls that overlap on the GPU (two
 *     streams, two host threads) race on it: serialise them.
 *   - Arguments are checked first, with the statuses of clis_certify.  Then
 *     shapes whose clis_certify_workspace_size() exceeds
 *     CLIS_NOALLOC_SCRATCH_BYTES return CLIS_ERR_WORKSPACE before anything
 *     is launched (about B*H*ceil(Nk/1024)*d*4 bytes; B*H = 40 heads of
 *     75,600 keys at d = 128 need 1.6 MB).
 *   - CLIS_ERR_CUDA if the address lookup fails. */
CLIS_API clis_status_t clis_certify_noalloc(const clis_shape_t *shape, const void *q, const void *k,
                                   const void *v, float scale_log2, clis_fmt_t exp_fmt,
                                   clis_fmt_t acc_fmt, float *kbar, clis_head_cert_t *certs,
                                   float *mu, clis_stream_t stream);

/* Fused attention forward O = softmax(scale * Q K^T) V (abstract and
 * Figure 5(a): with mu_i fixed before the KV loop, the loop needs no running
 * maximum and no rescaling).  One persistent kernel; each 256-row query block of a
 * head runs either
 *   - the certified path: mu_i = scale_log2 * (q_i . kbar) fixed before the
 *     KV loop, p_ij = exp2(scale_log2 * s_ij - mu_i), no row maximum, no
 *     rescaling; or
 *   - the online path: running row maximum and accumulator rescaling.
 *   o       device bf16 out [B,H,Nq,d] (strides from shape)
 *   lse2    optional device fp32 out [B*H*Nq] (contiguous, index
 *           (b*H + h)*Nq + i): log2 sum_j exp2(scale_log2 * s_ij); NULL = skip
 *   kbar, certs  outputs of clis_certify (may be NULL for CLIS_ONLINE and
 *           CLIS_ONLINE_LAZY)
 *   mu      optional per-row stabilisers from clis_certify (NULL: the kernel
 *           computes mu_i from q_i and kbar itself)
 *   causal  0 or 1; 1 requires Nq == Nk (key j visible to query i iff j <= i)
 * Nq == 0 or B*H == 0 launches nothing and returns CLIS_OK. */
CLIS_API clis_status_t clis_attn_fwd(const clis_shape_t *shape, const void *q, const void *k,
                            const void *v, void *o, float *lse2, const float *kbar,
                            const clis_head_cert_t *certs, const float *mu, float scale_log2,
                            int causal, clis_variant_t variant, clis_stream_t stream);

/* The forward for Q, K, V and O held in host memory (the abstract's
 * plug-and-play use: the attention call of a model whose tensors live on the
 * host).  Per group of consecutive heads: copy Q, K, V to the device, run
 * clis_certify (variants CLIS_AUTO and CLIS_CERTIFIED_FORCED; exp2 format of
 * the data type, FP32 accumulation) and clis_attn_fwd with its stabilisers,
 * copy O back.  The copies of one group overlap the kernels of others: copies
 * in on one stream of the plan, the kernels of even and odd groups on two
 * more, copies out on a fourth.  Each head is computed alone by the kernels
 * of clis_certify and clis_attn_fwd, so k-bar and the certificates equal
 * theirs on the whole tensors bit for bit; O may differ from their O by
 * rounding, because the attention kernel sweeps the keys of some work tiles
 * in reverse order depending on where the tile falls in its launch.
 *
 * clis_host_plan_create: a plan for one shape on the current device: its
 *   four streams and per-group events.  shape is as for clis_attn_fwd, but
 *   Q, K, V and O must be dense (n-stride d, head stride N*d, batch stride
 *   H*N*d, free when B = 1; CLIS_ERR_UNSUPPORTED otherwise); causal as for
 *   clis_attn_fwd; groups = number of head groups, 0 = about one group per
 *   2 TFLOP of attention work, at least 8 and at most B*H.  Argument errors
 *   as for clis_attn_fwd; CLIS_ERR_CUDA if a stream or event cannot be made.
 * clis_host_plan_workspace_size: bytes of device workspace every call with
 *   the plan needs: staging for Q, K, V and O of every head, k-bar,
 *   certificates and stabilisers, and two certification scratch areas (0 when
 *   B*H = 0 or Nq = 0).
 * clis_attention_host: one forward with the plan.
 *   q, k, v, o  host memory, any alignment; o is written.  Page-locked memory
 *               (cudaHostAlloc, cudaHostRegister) lets the copies run
 *               asynchronously; with pageable memory the CUDA runtime stages
 *               each copy and the call returns only after its copies ran.
 *   scale_log2, variant  as for clis_attn_fwd
 *   workspace   device memory of clis_host_plan_workspace_size() bytes,
 *               256-byte aligned, the same for every call with the plan.  Once
 *               the call is complete, its first B*H*d floats hold k-bar and the
 *               B*H certificates start at the next multiple of 256 bytes
 *               (certified variants).
 *   stream      the copies in follow the work queued on it before the call
 *   The call is queued, not waited for.  Calls with one plan must come from
 *   one host thread at a time (the plan records its events in each call).  Consecutive calls with one plan
 *   overlap: a call's copies of a group start once the previous call's
 *   kernels on that group have run, and its kernels once the previous call's
 *   copy out of that group has.  Must be called on the plan's device
 *   (CLIS_ERR_INVALID_ARG otherwise).  Errors: the argument checks of
 *   clis_attn_fwd, CLIS_ERR_WORKSPACE, CLIS_ERR_MISALIGNED for the
 *   workspace, all before anything is queued; CLIS_ERR_CUDA when a copy or
 *   launch fails, after which clis_host_plan_wait still covers everything the
 *   call queued.  B*H = 0 or Nq = 0 returns CLIS_OK and queues nothing.
 * clis_host_plan_wait: makes `stream` wait for the last copy out of the most
 *   recent call with the plan (nothing if there was none): o of that call and
 *   of every earlier one is complete once `stream` passes this point.
 * clis_host_plan_destroy: releases the plan (NULL is a no-op); work already
 *   queued still runs, and the CUDA runtime frees the streams and events
 *   after it.  The workspace may be reused or freed once that work is done. */
typedef struct clis_host_plan_s clis_host_plan_t;
CLIS_API clis_status_t clis_host_plan_create(const clis_shape_t *shape, int causal, int groups,
                                             clis_host_plan_t **plan);
CLIS_API clis_status_t clis_host_plan_workspace_size(const clis_host_plan_t *plan, size_t *bytes);
CLIS_API clis_status_t clis_attention_host(clis_host_plan_t *plan, const void *q, const void *k,
                                           const void *v, void *o, float scale_log2,
                                           clis_variant_t variant, void *workspace, size_t ws_bytes,
                                           clis_stream_t stream);
CLIS_API clis_status_t clis_host_plan_wait(clis_host_plan_t *plan, clis_stream_t stream);
CLIS_API clis_status_t clis_host_plan_destroy(clis_host_plan_t *plan);

/* FP8 P.V path.  Figure 3 tabulates exp2 limits per format; one step below
 * FP16 is E4M3 (largest finite value 448, so U_exp = log2 448 and the budget
 * is floor(U_exp) = 8).  One tcgen05.mma of kind::f8f6f4 takes both operands
 * in 8 bits, so P in E4M3 needs V in E4M3 too.  A head takes this path when it
 * certifies (clis_certify, BF16/FP32 formats) and also B_h <= min(8, C) and
 * G <= 8 (max |V| <= 256 fits E4M3) -- these make E4M3 safe -- and, for
 * accuracy, Nk >= 4096; every other head runs exactly as in clis_attn_fwd
 * (certified BF16 path or online softmax).  The row sum stays the fp32 sum of
 * the unrounded exp2 outputs.  Accuracy: V's E4M3 rounding (up to 2^-4
 * relative per entry) averages over the keys, so on diffuse heads the mean
 * output error is about 0.033 / sqrt(Nk) (2e-4 at 32,760 keys, 1.4e-3 at 513)
 * and the largest about ten times the BF16 path's; sharp heads (B_h above 8)
 * never qualify.
 *
 * clis_v_e4m3_size: bytes of the E4M3 V^T buffer, B*H*d*pitch with pitch =
 *   Nk rounded up to 16.
 * clis_v_to_e4m3: writes V^T [b*H + h][c][j] = E4M3(V[b, h, j, c]) (round to
 *   nearest even, saturating at +-448; bytes from Nk to the pitch are 0).
 *   BF16 V only (CLIS_ERR_UNSUPPORTED for FP16); vt8 16-byte aligned.
 * clis_attn_fwd_fp8pv: clis_attn_fwd (no mask) for d = 128 and BF16 data
 *   (CLIS_ERR_UNSUPPORTED otherwise) that also takes vt8 from clis_v_to_e4m3
 *   of the same v.  variant: CLIS_AUTO (the rule above) or
 *   CLIS_CERTIFIED_FORCED (every head on the FP8 P.V path whatever its
 *   certificate or length: benchmarks and tests only); other variants
 *   CLIS_ERR_INVALID_ARG. */
CLIS_API clis_status_t clis_v_e4m3_size(const clis_shape_t *shape, size_t *bytes);
CLIS_API clis_status_t clis_v_to_e4m3(const clis_shape_t *shape, const void *v, void *vt8, clis_stream_t stream);
CLIS_API clis_status_t clis_attn_fwd_fp8pv(const clis_shape_t *shape, const void *q, const void *k,
                                           const void *v, const void *vt8, void *o, float *lse2,
                                           const float *kbar, const clis_head_cert_t *certs, const float *mu,
                                           float scale_log2, clis_variant_t variant, clis_stream_t stream);

/* The ring-step form (clis_attn_fwd_chunk, no mask) with the FP8 P.V path:
 * vt8 is clis_v_to_e4m3 of the chunk's v (k and v point at the chunk, shape->Nk
 * its length); a head takes E4M3 by the rule above, with Nk the chunk's
 * length.  Certified heads still merge by plain addition.  Other arguments
 * and errors as clis_attn_fwd_chunk and clis_attn_fwd_fp8pv. */
CLIS_API clis_status_t clis_attn_fwd_chunk_fp8pv(const clis_shape_t *shape, const void *q, const void *k,
                                                 const void *v, const void *vt8, float *o_acc, float *l_acc,
                                                 float *m_acc, const float *kbar, const clis_head_cert_t *certs,
                                                 const float *mu, float scale_log2, int first,
                                                 clis_variant_t variant, clis_stream_t stream);

/* Per-prefix certificates for causal attention: clis_certify plus one flag per
 * block of 256 query rows.  The pages certify causal heads with the head's
 * bound (Table 3) and state no finer rule; this entry point is a finer reading
 * of the same Cauchy-Schwarz bound.  A causal row i sees keys 0..i only, so
 * for query block b (rows 256b .. 256b + 255) every exp2 argument is bounded
 * by B_b = scale_log2 * max_{i in b} ||q_i|| * max_{j <= 256b + 255}
 * ||k_j - kbar|| (rounded upward as B_h is), and the block is safe when the
 * head's inputs are finite and B_b <= C, the head's budget.  A certified head
 * has every block certified; a head that fails can still certify the blocks
 * whose prefixes exclude its large keys.
 *   tile_certs  device uint8 out [B*H][ceil(Nq / 256)]: 1 = the block may take
 *               the fixed stabiliser in clis_attn_fwd_tiles
 *   (other arguments as for clis_certify; Nq must equal Nk)
 * Errors as for clis_certify; CLIS_ERR_INVALID_ARG for a null tile_certs,
 * CLIS_ERR_UNSUPPORTED if Nq != Nk. */
CLIS_API clis_status_t clis_certify_tiles(const clis_shape_t *shape, const void *q, const void *k,
                                          const void *v, float scale_log2, clis_fmt_t exp_fmt,
                                          clis_fmt_t acc_fmt, float *kbar, clis_head_cert_t *certs,
                                          float *mu, uint8_t *tile_certs, void *workspace,
                                          size_t ws_bytes, clis_stream_t stream);

/* clis_attn_fwd for causal attention (causal = 1, variant = CLIS_AUTO) that
 * also takes the per-prefix certificates of clis_certify_tiles: a query block
 * of a head that failed certification as a whole still takes the fixed
 * stabiliser when its block flag is set (for FP16 data only if the head's
 * budget C <= 15).  Errors as for clis_attn_fwd; CLIS_ERR_INVALID_ARG for a
 * null tile_certs, causal = 0 or another variant. */
CLIS_API clis_status_t clis_attn_fwd_tiles(const clis_shape_t *shape, const void *q, const void *k,
                                           const void *v, void *o, float *lse2, const float *kbar,
                                           const clis_head_cert_t *certs, const uint8_t *tile_certs,
                                           const float *mu, float scale_log2, int causal,
                                           clis_variant_t variant, clis_stream_t stream);

/* One KV chunk of a ring / context-parallel attention step (paper: Table 7,
 * the ring and 2D-ring columns, and Figure 6, one ring attention step).  The
 * keys and values of a head are split into chunks that arrive one at a time;
 * each call runs the fused kernel over one chunk (shape->Nk = its length, k and
 * v point at it) and merges the chunk's partial result into fp32 accumulators
 * kept by the caller (contiguous, index (b*H + h)*Nq + i):
 *   o_acc [B*H*Nq*d]  sum_j 2^(x_ij - m_i) v_j over the keys merged so far
 *   l_acc [B*H*Nq]    sum_j 2^(x_ij - m_i)
 *   m_acc [B*H*Nq]    the shift m_i (exp2 units), x_ij = scale_log2 * q_i . k_j
 * first = 1 overwrites the accumulators (first chunk), 0 merges.  A certified
 * head's shift is its fixed stabiliser mu_i in every chunk, so its partials
 * add with no exponentials, no rescaling and no read of the accumulators
 * (in-memory vector adds); other heads read the accumulators and merge by
 * rescaling to the larger maximum.  Calls on one set of accumulators must
 * be ordered (one stream, or events between streams).  kbar, certs (and mu, optional) must come from
 * clis_certify over the whole key sequence (for a ring: the k-bar partials and norm maxima of all
 * chunks reduced before the first step).  Non-causal (clis_attn_fwd_chunk_causal is the causal
 * form); shape->o_* ignored.
 * Errors as clis_attn_fwd. */
CLIS_API clis_status_t clis_attn_fwd_chunk(const clis_shape_t *shape, const void *q, const void *k,
                                  const void *v, float *o_acc, float *l_acc, float *m_acc,
                                  const float *kbar, const clis_head_cert_t *certs,
                                  const float *mu, float scale_log2, int first,
                                  clis_variant_t variant, clis_stream_t stream);

/* Causal form of clis_attn_fwd_chunk (Table 7's ring columns and Figure 6's
 * ring step, for the causal training setting of Table 3): the chunk holds keys
 * key_offset .. key_offset + shape->Nk - 1 of the head (k and v point at the
 * chunk's first key), q all shape->Nq query rows, and query i sees chunk key j
 * iff key_offset + j <= i.  Rows before key_offset see none of the chunk's
 * keys and their accumulators are left untouched; query blocks of 256 rows that
 * end before key_offset are not computed at all.  The partials merge as in
 * clis_attn_fwd_chunk: a certified row's shift is its fixed mu_i in every chunk,
 * so its partial is added with no rescaling, in any chunk order.
 *   key_offset  >= 0, with key_offset + shape->Nk <= shape->Nq
 *               (CLIS_ERR_UNSUPPORTED otherwise)
 *   first       1 overwrites the accumulators of every row: only the chunk
 *               with key_offset = 0 may be first (CLIS_ERR_INVALID_ARG
 *               otherwise); the other chunks follow in any order
 *   tile_certs  optional per-prefix certificates from clis_certify_tiles over
 *               the whole sequence (NULL: per-head flags only); a query block
 *               whose flag is set takes the fixed stabiliser in every chunk
 *               (CLIS_AUTO only; CLIS_ERR_INVALID_ARG with another variant)
 *   kbar, certs, mu  from clis_certify (or clis_certify_tiles) over the whole
 *               sequence
 * Other arguments and errors as clis_attn_fwd_chunk. */
CLIS_API clis_status_t clis_attn_fwd_chunk_causal(const clis_shape_t *shape, const void *q, const void *k,
                                                  const void *v, float *o_acc, float *l_acc, float *m_acc,
                                                  const float *kbar, const clis_head_cert_t *certs,
                                                  const uint8_t *tile_certs, const float *mu, float scale_log2,
                                                  int64_t key_offset, int first, clis_variant_t variant,
                                                  clis_stream_t stream);

/* After the last chunk: o = o_acc / l_acc (bf16, strides shape->o_*) and, if
 * lse2 is not NULL, lse2 = m_acc + log2(l_acc). */
CLIS_API clis_status_t clis_attn_chunk_finalize(const clis_shape_t *shape, const float *o_acc,
                                       const float *l_acc, const float *m_acc, void *o,
                                       float *lse2, clis_stream_t stream);

/* Workspace bytes for clis_attn_bwd: one fp32 per query row (B*H*Nq, the
 * row dots D_i), rounded up to 256.  CLIS_ERR_INVALID_ARG for a NULL or
 * invalid shape. */
CLIS_API clis_status_t clis_attn_bwd_workspace_size(const clis_shape_t *shape, size_t *bytes);

/* Attention backward: dQ, dK, dV of L = sum(dout * O) for O = softmax(scale *
 * Q K^T) V, scale = scale_log2 * ln 2.  The paper's causal LLM training
 * results (Table 3) run a backward pass but the paper gives none; this is the
 * plain chain rule through softmax, driven by the forward's row statistic:
 *   P_ij = exp2(scale_log2 * s_ij - lse2_i),  D_i = dout_i . o_i,
 *   dS_ij = P_ij (dout_i . v_j - D_i),
 *   dV_j = sum_i P_ij dout_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
 * lse2 is fixed per row, whichever forward path produced it, so the
 * backward has no running maximum and no rescaling.
 *   q, k, v   the forward's inputs (device, shape->dtype)
 *   o         the forward's output and dout its gradient, both with strides
 *             shape->o_*
 *   lse2      device fp32 [B*H*Nq], from clis_attn_fwd (or
 *             clis_attn_chunk_finalize) with the same q, k, scale_log2, causal
 *   dq, dk, dv  device outputs, same dtype; dq has strides shape->q_*, dk
 *             shape->k_*, dv shape->v_*.  Every element is written once
 *             (deterministic: no atomics).
 *   workspace device buffer of at least clis_attn_bwd_workspace_size() bytes,
 *             16-byte aligned (CLIS_ERR_WORKSPACE otherwise)
 *   causal    0 or 1; 1 requires Nq == Nk
 * Nq == 0 writes dK = dV = 0.  Errors as clis_attn_fwd. */
CLIS_API clis_status_t clis_attn_bwd(const clis_shape_t *shape, const void *q, const void *k,
                                     const void *v, const void *o, const void *dout,
                                     const float *lse2, void *dq, void *dk, void *dv,
                                     float scale_log2, int causal, void *workspace,
                                     size_t ws_bytes, clis_stream_t stream);

/* Static description of a status code (never NULL). */
CLIS_API const char *clis_status_string(clis_status_t status);

/* Reads the device error word of the current device (synchronises the
 * device).  *code = 0 when no kernel recorded a fault; otherwise bit flags of
 * the pipeline waits that timed out.  Returns CLIS_ERR_TIMEOUT if *code != 0,
 * CLIS_ERR_CUDA if the read failed. */
CLIS_API clis_status_t clis_get_device_error(uint32_t *code);

/* Resets the device error word of the current device to 0 (synchronous). */
CLIS_API clis_status_t clis_clear_device_error(void);

/* Self-test of the kernels' bounded waits (no counterpart in the paper).
 * Launches one small kernel whose single wait is on a barrier that nothing
 * ever arrives on, with a limit of limit_us microseconds (1..1,000,000): the
 * wait gives up, records CLIS_WAIT_SELFTEST_BIT in the device error word and
 * the kernel returns, leaving the context usable.  Read the word with
 * clis_get_device_error() and reset it with clis_clear_device_error(). */
#define CLIS_WAIT_SELFTEST_BIT (1u << 8)
CLIS_API clis_status_t clis_debug_wait_selftest(uint32_t limit_us, clis_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CLIS_H */
