// clis_internal.h -- declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/clis.h"

namespace clis {

// ----------------------------------------------------------- certification

constexpr int kCertChunkRows = 1024;  // rows per partial-reduction chunk
constexpr int kCertNormSplit = 4;     // norms-kernel blocks per chunk
constexpr int kCertThreads = 256;

// Query rows per work tile of the attention kernel, which is also the block
// of the per-prefix certificates: the norms pass keeps one maximum per block
// of kCertChunkRows / kCertNormSplit rows, and the certificate of query block
// b is read by the attention work tile with the same rows.
constexpr int kQueryBlockRows = 256;
static_assert(kCertChunkRows % kCertNormSplit == 0 && kCertChunkRows / kCertNormSplit == kQueryBlockRows,
              "per-prefix certificates need one norms block per attention work tile");

struct CertWorkspace {
    float *ksum;       // [BH][nck][d]  per-chunk column sums of K
    uint32_t *knorm2;  // [BH][nck]     per-chunk max of ||k - kbar||^2 (fp32 bits, rounded up)
    uint32_t *qnorm2;  // [BH][ncq]     per-chunk max of ||q||^2 (fp32 bits, rounded up)
    uint32_t *kabs;    // [BH][nck]     per-chunk max of |k| as bf16 bits (& 0x7FFF)
    uint32_t *qabs;    // [BH][ncq]
    uint32_t *vabs;    // [BH][nck]
    // Per 256-row block (kCertChunkRows / kCertNormSplit rows) maxima of the
    // norms pass, for the per-prefix certificates of causal heads.
    uint32_t *knorm2s;  // [BH][kCertNormSplit * nck]
    uint32_t *qnorm2s;  // [BH][kCertNormSplit * ncq]
};

struct CertArgs {
    const uint16_t *q, *k, *v;  // bf16 bits
    int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn, v_sb, v_sh, v_sn;
    int B, H, Nq, Nk, d;
    int dtype;  // clis_dtype_t
    int nck, ncq;
    float scale_log2;
    int emax_exp, emax_acc;  // floor(U) of the exp2-output and accumulator formats
    float *kbar;
    clis_head_cert_t *certs;
    float *mu;  // optional per-row stabilisers [B*H*Nq]
    uint8_t *tile_certs = nullptr;  // optional per-prefix certificates [B*H][nqb] (causal, Nq == Nk)
    int nqb = 0;                    // 256-row query blocks per head
};

// Carves the workspace for the given sizes; returns the bytes needed.
size_t cert_workspace_layout(int64_t BH, int64_t nck, int64_t ncq, int64_t d, void *base,
                             CertWorkspace *ws);

cudaError_t launch_certify(const CertArgs &a, const CertWorkspace &ws, cudaStream_t stream);

// Device address of the library-owned certification scratch array in the
// current context: looked up on every call outside stream capture, taken from
// the last such lookup in the same (device, context) while `stream` is being
// captured; nullptr on failure or when no lookup was made before the capture.
void *certify_static_scratch(cudaStream_t stream);

// ---------------------------------------------------------------- attention

struct AttnArgs {
    const uint16_t *q, *k, *v;
    uint16_t *o;
    float *lse2;
    const float *kbar;
    const clis_head_cert_t *certs;
    const float *mu = nullptr;  // optional per-row stabilisers from clis_certify
    const uint8_t *tile_certs = nullptr;  // optional per-prefix certificates (causal AUTO)
    int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn, v_sb, v_sh, v_sn, o_sb, o_sh, o_sn;
    int B, H, Nq, Nk, d;
    int dtype = CLIS_DT_BF16;
    float scale_log2;
    int causal;
    int variant;
    int chunk_mode = 0;  // 0 off, 1 merge into the accumulators, 2 first chunk
    float *o_acc = nullptr, *l_acc = nullptr, *m_acc = nullptr;
    int k_off = 0;  // causal KV chunk: index of the chunk's first key in the head
    // FP8 P.V path: V^T in E4M3 [B*H][d][vt8_pitch] (nullptr: BF16 P.V only).
    const uint8_t *vt8 = nullptr;
    int64_t vt8_pitch = 0;
};

// Conversion of V to its E4M3 transpose for the FP8 P.V path.
struct VtArgs {
    const uint16_t *v;  // bf16 [B, H, Nk, d]
    int64_t v_sb, v_sh, v_sn;
    int B, H, Nk, d;
    uint8_t *vt;        // E4M3 [B*H][d][pitch]
    int64_t pitch;      // bytes per row of V^T: Nk rounded up to 16
};

clis_status_t launch_v_to_e4m3t(const VtArgs &a, cudaStream_t stream);

struct ChunkFinalizeArgs {
    const float *o_acc, *l_acc, *m_acc;
    uint16_t *o;
    float *lse2;
    int64_t o_sb, o_sh, o_sn;
    int B, H, Nq, d;
    int dtype;
};

clis_status_t launch_chunk_finalize(const ChunkFinalizeArgs &a, cudaStream_t stream);

// Builds the tensor maps and launches the persistent attention kernel.
// Returns CLIS_OK, CLIS_ERR_CUDA (tensor-map encode or launch failure).
clis_status_t launch_attn_fwd(const AttnArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- backward

struct AttnBwdArgs {
    const uint16_t *q, *k, *v, *o, *dout;
    const float *lse2;
    float *dvec;  // workspace: D_i = dO_i . O_i, [B*H*Nq]
    uint16_t *dq, *dk, *dv;
    // dq shares q's strides, dk k's, dv v's, dout o's.
    int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn, v_sb, v_sh, v_sn, o_sb, o_sh, o_sn;
    int B, H, Nq, Nk, d;
    int dtype;
    float scale_log2;
    int causal;
};

// Launches the row-dot, dK/dV and dQ kernels (or zero-fills dK and dV when
// Nq = 0).  Returns CLIS_OK or CLIS_ERR_CUDA.
clis_status_t launch_attn_bwd(const AttnBwdArgs &a, cudaStream_t stream);
clis_status_t read_bwd_error(uint32_t *code);
clis_status_t clear_bwd_error();

clis_status_t launch_wait_selftest(uint32_t limit_us, cudaStream_t stream);
clis_status_t read_device_error(uint32_t *code);
clis_status_t clear_device_error();

}  // namespace clis
