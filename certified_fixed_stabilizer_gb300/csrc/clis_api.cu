// clis_api.cu -- the extern "C" boundary declared in include/clis.h.
//
// Every entry point validates its arguments on the host before touching the
// GPU; on any argument error it returns a status and launches nothing.
#include <cmath>
#include <cstdint>

#include "clis_internal.h"

namespace {

constexpr int64_t kMaxN = (int64_t(1) << 31) - 1024;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

clis_status_t check_strides(int64_t sb, int64_t sh, int64_t sn, int64_t d)
{
    if (sb < 0 || sh < 0 || sn < d) return CLIS_ERR_INVALID_ARG;
    if ((sb | sh | sn) & 7) return CLIS_ERR_MISALIGNED;
    if (sb >= (int64_t(1) << 38) || sh >= (int64_t(1) << 38) || sn >= (int64_t(1) << 38))
        return CLIS_ERR_UNSUPPORTED;
    return CLIS_OK;
}

// Strides of a written tensor must give every (b, h) its own elements: a zero
// head (batch) stride with more than one head (batch) would make them share
// (a tensor of N = 0 rows has no elements to share).
bool aliasing(int64_t B, int64_t H, int64_t N, int64_t sb, int64_t sh)
{
    return N > 0 && ((H > 1 && sh == 0) || (B > 1 && sb == 0));
}

clis_status_t check_shape(const clis_shape_t *s, bool with_o)
{
    if (!s) return CLIS_ERR_INVALID_ARG;
    if (s->B < 0 || s->H < 0 || s->Nq < 0 || s->Nk < 1 || s->d < 1) return CLIS_ERR_INVALID_ARG;
    if (s->d != 64 && s->d != 128) return CLIS_ERR_UNSUPPORTED;
    if (s->dtype != CLIS_DT_BF16 && s->dtype != CLIS_DT_FP16) return CLIS_ERR_INVALID_ARG;
    if (s->Nq > kMaxN || s->Nk > kMaxN || s->B * s->H > kMaxN || s->B > kMaxN || s->H > kMaxN)
        return CLIS_ERR_UNSUPPORTED;
    clis_status_t st;
    if ((st = check_strides(s->q_sb, s->q_sh, s->q_sn, s->d)) != CLIS_OK) return st;
    if ((st = check_strides(s->k_sb, s->k_sh, s->k_sn, s->d)) != CLIS_OK) return st;
    if ((st = check_strides(s->v_sb, s->v_sh, s->v_sn, s->d)) != CLIS_OK) return st;
    if (with_o && (st = check_strides(s->o_sb, s->o_sh, s->o_sn, s->d)) != CLIS_OK) return st;
    if (with_o && aliasing(s->B, s->H, s->Nq, s->o_sb, s->o_sh)) return CLIS_ERR_INVALID_ARG;
    return CLIS_OK;
}

bool valid_fmt(int f) { return f == CLIS_FMT_FP16 || f == CLIS_FMT_BF16 || f == CLIS_FMT_FP32; }

// floor(log2 of the largest finite value) = the format's maximum exponent.
int fmt_emax(int f) { return f == CLIS_FMT_FP16 ? 15 : 127; }

int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Bytes per row of the E4M3 V^T buffer: Nk rounded up to 16 (TMA strides are
// multiples of 16 bytes).
int64_t vt8_pitch(int64_t Nk) { return div_up(Nk, 16) * 16; }

}  // namespace

extern "C" {

clis_status_t clis_certify_workspace_size(const clis_shape_t *shape, size_t *bytes)
{
    if (!shape || !bytes) return CLIS_ERR_INVALID_ARG;
    if (shape->B < 0 || shape->H < 0 || shape->Nq < 0 || shape->Nk < 1 || shape->d < 1)
        return CLIS_ERR_INVALID_ARG;
    const int64_t BH = shape->B * shape->H;
    const int64_t nck = div_up(shape->Nk, clis::kCertChunkRows);
    const int64_t ncq = div_up(shape->Nq, clis::kCertChunkRows);
    *bytes = clis::cert_workspace_layout(BH, nck, ncq, shape->d, nullptr, nullptr);
    return CLIS_OK;
}

}  // extern "C"

namespace {

// Every check of the certification arguments except the workspace.
clis_status_t check_certify_args(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                 float scale_log2, clis_fmt_t exp_fmt, clis_fmt_t acc_fmt, const float *kbar,
                                 const clis_head_cert_t *certs, const float *mu)
{
    clis_status_t st = check_shape(shape, false);
    if (st != CLIS_OK) return st;
    // q is never read when Nq == 0 and may then be NULL.
    if ((!q && shape->Nq > 0) || !k || !v || !kbar || !certs) return CLIS_ERR_INVALID_ARG;
    if (!std::isfinite(scale_log2) || !(scale_log2 > 0.f)) return CLIS_ERR_INVALID_ARG;
    if (!valid_fmt(exp_fmt) || !valid_fmt(acc_fmt)) return CLIS_ERR_INVALID_ARG;
    if ((q && !aligned16(q)) || !aligned16(k) || !aligned16(v) || !aligned16(kbar) || !aligned16(certs) ||
        (mu && (reinterpret_cast<uintptr_t>(mu) & 3u)))
        return CLIS_ERR_MISALIGNED;
    return CLIS_OK;
}

clis_status_t certify_impl(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                           float scale_log2, clis_fmt_t exp_fmt, clis_fmt_t acc_fmt, float *kbar,
                           clis_head_cert_t *certs, float *mu, uint8_t *tile_certs, void *workspace,
                           size_t ws_bytes, clis_stream_t stream)
{
    const clis_status_t st = check_certify_args(shape, q, k, v, scale_log2, exp_fmt, acc_fmt, kbar, certs, mu);
    if (st != CLIS_OK) return st;
    size_t need = 0;
    clis_certify_workspace_size(shape, &need);
    if (need > 0 && (!workspace || ws_bytes < need)) return CLIS_ERR_WORKSPACE;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return CLIS_ERR_MISALIGNED;
    const int64_t BH = shape->B * shape->H;
    if (BH == 0) return CLIS_OK;

    clis::CertArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.q_sb = shape->q_sb;
    a.q_sh = shape->q_sh;
    a.q_sn = shape->q_sn;
    a.k_sb = shape->k_sb;
    a.k_sh = shape->k_sh;
    a.k_sn = shape->k_sn;
    a.v_sb = shape->v_sb;
    a.v_sh = shape->v_sh;
    a.v_sn = shape->v_sn;
    a.B = static_cast<int>(shape->B);
    a.H = static_cast<int>(shape->H);
    a.Nq = static_cast<int>(shape->Nq);
    a.Nk = static_cast<int>(shape->Nk);
    a.d = static_cast<int>(shape->d);
    a.dtype = static_cast<int>(shape->dtype);
    a.nck = static_cast<int>(div_up(shape->Nk, clis::kCertChunkRows));
    a.ncq = static_cast<int>(div_up(shape->Nq, clis::kCertChunkRows));
    a.scale_log2 = scale_log2;
    a.emax_exp = fmt_emax(exp_fmt);
    a.emax_acc = fmt_emax(acc_fmt);
    a.kbar = kbar;
    a.certs = certs;
    a.mu = mu;
    a.tile_certs = tile_certs;
    a.nqb = static_cast<int>(div_up(shape->Nq, clis::kQueryBlockRows));
    if (clis::kCertNormSplit * BH * (2 * a.nck + a.ncq) > kMaxN) return CLIS_ERR_UNSUPPORTED;
    clis::CertWorkspace ws;
    clis::cert_workspace_layout(BH, a.nck, a.ncq, a.d, workspace, &ws);
    return clis::launch_certify(a, ws, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? CLIS_OK
                                                                                              : CLIS_ERR_CUDA;
}

}  // namespace

extern "C" {

clis_status_t clis_certify(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                           float scale_log2, clis_fmt_t exp_fmt, clis_fmt_t acc_fmt, float *kbar,
                           clis_head_cert_t *certs, float *mu, void *workspace, size_t ws_bytes,
                           clis_stream_t stream)
{
    return certify_impl(shape, q, k, v, scale_log2, exp_fmt, acc_fmt, kbar, certs, mu, nullptr, workspace,
                        ws_bytes, stream);
}

clis_status_t clis_certify_tiles(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                 float scale_log2, clis_fmt_t exp_fmt, clis_fmt_t acc_fmt, float *kbar,
                                 clis_head_cert_t *certs, float *mu, uint8_t *tile_certs, void *workspace,
                                 size_t ws_bytes, clis_stream_t stream)
{
    if (!shape || !tile_certs) return CLIS_ERR_INVALID_ARG;
    if (shape->Nq != shape->Nk) return CLIS_ERR_UNSUPPORTED;  // per-prefix: causal heads only
    return certify_impl(shape, q, k, v, scale_log2, exp_fmt, acc_fmt, kbar, certs, mu, tile_certs, workspace,
                        ws_bytes, stream);
}

}  // extern "C"

namespace {

clis_status_t attn_fwd_impl(const clis_shape_t *shape, const void *q, const void *k, const void *v, void *o,
                            float *lse2, const float *kbar, const clis_head_cert_t *certs,
                            const uint8_t *tile_certs, const float *mu, float scale_log2, int causal,
                            clis_variant_t variant, clis_stream_t stream, const void *vt8 = nullptr)
{
    clis_status_t st = check_shape(shape, true);
    if (st != CLIS_OK) return st;
    if (shape->B * shape->H == 0 || shape->Nq == 0) return CLIS_OK;  // nothing to compute
    if (!q || !k || !v || !o) return CLIS_ERR_INVALID_ARG;
    if (!std::isfinite(scale_log2) || !(scale_log2 > 0.f)) return CLIS_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return CLIS_ERR_INVALID_ARG;
    if (variant != CLIS_AUTO && variant != CLIS_ONLINE && variant != CLIS_CERTIFIED_FORCED &&
        variant != CLIS_ONLINE_LAZY)
        return CLIS_ERR_INVALID_ARG;
    if ((variant == CLIS_AUTO || variant == CLIS_CERTIFIED_FORCED) && !kbar) return CLIS_ERR_INVALID_ARG;
    if (variant == CLIS_AUTO && !certs) return CLIS_ERR_INVALID_ARG;
    if (causal && shape->Nq != shape->Nk) return CLIS_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return CLIS_ERR_MISALIGNED;
    if ((kbar && !aligned16(kbar)) || (certs && !aligned16(certs)) ||
        (lse2 && (reinterpret_cast<uintptr_t>(lse2) & 3u)) || (mu && (reinterpret_cast<uintptr_t>(mu) & 3u)))
        return CLIS_ERR_MISALIGNED;

    clis::AttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.o = static_cast<uint16_t *>(o);
    a.lse2 = lse2;
    a.kbar = kbar;
    a.certs = certs;
    a.mu = mu;
    a.q_sb = shape->q_sb;
    a.q_sh = shape->q_sh;
    a.q_sn = shape->q_sn;
    a.k_sb = shape->k_sb;
    a.k_sh = shape->k_sh;
    a.k_sn = shape->k_sn;
    a.v_sb = shape->v_sb;
    a.v_sh = shape->v_sh;
    a.v_sn = shape->v_sn;
    a.o_sb = shape->o_sb;
    a.o_sh = shape->o_sh;
    a.o_sn = shape->o_sn;
    a.B = static_cast<int>(shape->B);
    a.H = static_cast<int>(shape->H);
    a.Nq = static_cast<int>(shape->Nq);
    a.Nk = static_cast<int>(shape->Nk);
    a.d = static_cast<int>(shape->d);
    a.dtype = static_cast<int>(shape->dtype);
    a.scale_log2 = scale_log2;
    a.causal = causal;
    a.variant = variant;
    a.tile_certs = tile_certs;
    a.vt8 = static_cast<const uint8_t *>(vt8);
    a.vt8_pitch = vt8_pitch(shape->Nk);
    const int64_t tiles = shape->B * shape->H * div_up(shape->Nq, clis::kQueryBlockRows);
    if (tiles > kMaxN) return CLIS_ERR_UNSUPPORTED;
    return clis::launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

clis_status_t clis_attn_fwd(const clis_shape_t *shape, const void *q, const void *k, const void *v, void *o,
                            float *lse2, const float *kbar, const clis_head_cert_t *certs, const float *mu,
                            float scale_log2, int causal, clis_variant_t variant, clis_stream_t stream)
{
    return attn_fwd_impl(shape, q, k, v, o, lse2, kbar, certs, nullptr, mu, scale_log2, causal, variant, stream);
}

clis_status_t clis_attn_fwd_tiles(const clis_shape_t *shape, const void *q, const void *k, const void *v, void *o,
                                  float *lse2, const float *kbar, const clis_head_cert_t *certs,
                                  const uint8_t *tile_certs, const float *mu, float scale_log2, int causal,
                                  clis_variant_t variant, clis_stream_t stream)
{
    if (!shape || !tile_certs) return CLIS_ERR_INVALID_ARG;
    if (!causal || variant != CLIS_AUTO) return CLIS_ERR_INVALID_ARG;  // per-prefix: causal AUTO only
    return attn_fwd_impl(shape, q, k, v, o, lse2, kbar, certs, tile_certs, mu, scale_log2, causal, variant,
                         stream);
}

clis_status_t clis_v_e4m3_size(const clis_shape_t *shape, size_t *bytes)
{
    if (!shape || !bytes) return CLIS_ERR_INVALID_ARG;
    if (shape->B < 0 || shape->H < 0 || shape->Nk < 1 || shape->d < 1) return CLIS_ERR_INVALID_ARG;
    *bytes = static_cast<size_t>(shape->B * shape->H * shape->d * vt8_pitch(shape->Nk));
    return CLIS_OK;
}

clis_status_t clis_v_to_e4m3(const clis_shape_t *shape, const void *v, void *vt8, clis_stream_t stream)
{
    clis_status_t st = check_shape(shape, false);
    if (st != CLIS_OK) return st;
    if (shape->dtype != CLIS_DT_BF16) return CLIS_ERR_UNSUPPORTED;
    if (shape->B * shape->H == 0) return CLIS_OK;
    if (!v || !vt8) return CLIS_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(vt8)) return CLIS_ERR_MISALIGNED;
    if (shape->B * shape->H > 65535) return CLIS_ERR_UNSUPPORTED;  // grid.y
    clis::VtArgs a;
    a.v = static_cast<const uint16_t *>(v);
    a.v_sb = shape->v_sb;
    a.v_sh = shape->v_sh;
    a.v_sn = shape->v_sn;
    a.B = static_cast<int>(shape->B);
    a.H = static_cast<int>(shape->H);
    a.Nk = static_cast<int>(shape->Nk);
    a.d = static_cast<int>(shape->d);
    a.vt = static_cast<uint8_t *>(vt8);
    a.pitch = vt8_pitch(shape->Nk);
    return clis::launch_v_to_e4m3t(a, reinterpret_cast<cudaStream_t>(stream));
}

clis_status_t clis_attn_fwd_fp8pv(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                  const void *vt8, void *o, float *lse2, const float *kbar,
                                  const clis_head_cert_t *certs, const float *mu, float scale_log2,
                                  clis_variant_t variant, clis_stream_t stream)
{
    clis_status_t st = check_shape(shape, true);
    if (st != CLIS_OK) return st;
    if (shape->d != 128 || shape->dtype != CLIS_DT_BF16) return CLIS_ERR_UNSUPPORTED;
    if (variant != CLIS_AUTO && variant != CLIS_CERTIFIED_FORCED) return CLIS_ERR_INVALID_ARG;
    if (shape->B * shape->H == 0 || shape->Nq == 0) return CLIS_OK;
    if (!vt8) return CLIS_ERR_INVALID_ARG;
    if (!aligned16(vt8)) return CLIS_ERR_MISALIGNED;
    return attn_fwd_impl(shape, q, k, v, o, lse2, kbar, certs, nullptr, mu, scale_log2, 0, variant, stream, vt8);
}

clis_status_t clis_certify_noalloc(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                   float scale_log2, clis_fmt_t exp_fmt, clis_fmt_t acc_fmt, float *kbar,
                                   clis_head_cert_t *certs, float *mu, clis_stream_t stream)
{
    // Argument errors first, so a shape that is invalid or unsupported reports
    // that rather than its scratch size.
    clis_status_t st = check_certify_args(shape, q, k, v, scale_log2, exp_fmt, acc_fmt, kbar, certs, mu);
    if (st != CLIS_OK) return st;
    size_t need = 0;
    if ((st = clis_certify_workspace_size(shape, &need)) != CLIS_OK) return st;
    if (need > CLIS_NOALLOC_SCRATCH_BYTES) return CLIS_ERR_WORKSPACE;
    if (shape->B * shape->H == 0) return CLIS_OK;
    void *scratch = clis::certify_static_scratch(reinterpret_cast<cudaStream_t>(stream));
    if (!scratch) return CLIS_ERR_CUDA;
    return clis_certify(shape, q, k, v, scale_log2, exp_fmt, acc_fmt, kbar, certs, mu, scratch,
                        CLIS_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"

namespace {

clis_status_t attn_chunk_impl(const clis_shape_t *shape, const void *q, const void *k, const void *v, float *o_acc,
                              float *l_acc, float *m_acc, const float *kbar, const clis_head_cert_t *certs,
                              const uint8_t *tile_certs, const float *mu, float scale_log2, int causal,
                              int64_t key_offset, int first, clis_variant_t variant, clis_stream_t stream,
                              const void *vt8 = nullptr)
{
    clis_status_t st = check_shape(shape, false);
    if (st != CLIS_OK) return st;
    if (shape->B * shape->H == 0 || shape->Nq == 0) return CLIS_OK;
    if (!q || !k || !v || !o_acc || !l_acc || !m_acc) return CLIS_ERR_INVALID_ARG;
    if (!std::isfinite(scale_log2) || !(scale_log2 > 0.f)) return CLIS_ERR_INVALID_ARG;
    if (first != 0 && first != 1) return CLIS_ERR_INVALID_ARG;
    if (variant != CLIS_AUTO && variant != CLIS_ONLINE && variant != CLIS_CERTIFIED_FORCED &&
        variant != CLIS_ONLINE_LAZY)
        return CLIS_ERR_INVALID_ARG;
    if ((variant == CLIS_AUTO || variant == CLIS_CERTIFIED_FORCED) && !kbar) return CLIS_ERR_INVALID_ARG;
    if (variant == CLIS_AUTO && !certs) return CLIS_ERR_INVALID_ARG;
    if (tile_certs && variant != CLIS_AUTO) return CLIS_ERR_INVALID_ARG;
    if (causal) {
        if (key_offset < 0) return CLIS_ERR_INVALID_ARG;
        // The first chunk initialises every row's accumulators, so it must be
        // the one holding key 0 (the only chunk every query row sees).
        if (first && key_offset != 0) return CLIS_ERR_INVALID_ARG;
        if (key_offset + shape->Nk > shape->Nq) return CLIS_ERR_UNSUPPORTED;
    }
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_acc)) return CLIS_ERR_MISALIGNED;
    if ((kbar && !aligned16(kbar)) || (certs && !aligned16(certs)) ||
        (reinterpret_cast<uintptr_t>(l_acc) & 3u) || (reinterpret_cast<uintptr_t>(m_acc) & 3u) ||
        (mu && (reinterpret_cast<uintptr_t>(mu) & 3u)))
        return CLIS_ERR_MISALIGNED;
    const int64_t tiles = shape->B * shape->H * div_up(shape->Nq, clis::kQueryBlockRows);
    if (tiles > kMaxN) return CLIS_ERR_UNSUPPORTED;

    clis::AttnArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.o = nullptr;
    a.lse2 = nullptr;
    a.kbar = kbar;
    a.certs = certs;
    a.mu = mu;
    a.tile_certs = tile_certs;
    a.q_sb = shape->q_sb;
    a.q_sh = shape->q_sh;
    a.q_sn = shape->q_sn;
    a.k_sb = shape->k_sb;
    a.k_sh = shape->k_sh;
    a.k_sn = shape->k_sn;
    a.v_sb = shape->v_sb;
    a.v_sh = shape->v_sh;
    a.v_sn = shape->v_sn;
    a.o_sb = a.o_sh = a.o_sn = 0;
    a.B = static_cast<int>(shape->B);
    a.H = static_cast<int>(shape->H);
    a.Nq = static_cast<int>(shape->Nq);
    a.Nk = static_cast<int>(shape->Nk);
    a.d = static_cast<int>(shape->d);
    a.dtype = static_cast<int>(shape->dtype);
    a.scale_log2 = scale_log2;
    a.causal = causal;
    a.k_off = causal ? static_cast<int>(key_offset) : 0;
    a.variant = variant;
    a.chunk_mode = first ? 2 : 1;
    a.o_acc = o_acc;
    a.l_acc = l_acc;
    a.m_acc = m_acc;
    a.vt8 = static_cast<const uint8_t *>(vt8);
    a.vt8_pitch = vt8_pitch(shape->Nk);
    return clis::launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

clis_status_t clis_attn_fwd_chunk(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                  float *o_acc, float *l_acc, float *m_acc, const float *kbar,
                                  const clis_head_cert_t *certs, const float *mu, float scale_log2, int first,
                                  clis_variant_t variant, clis_stream_t stream)
{
    return attn_chunk_impl(shape, q, k, v, o_acc, l_acc, m_acc, kbar, certs, nullptr, mu, scale_log2, 0, 0, first,
                           variant, stream);
}

clis_status_t clis_attn_fwd_chunk_fp8pv(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                        const void *vt8, float *o_acc, float *l_acc, float *m_acc,
                                        const float *kbar, const clis_head_cert_t *certs, const float *mu,
                                        float scale_log2, int first, clis_variant_t variant, clis_stream_t stream)
{
    if (!shape) return CLIS_ERR_INVALID_ARG;
    if (shape->d != 128 || shape->dtype != CLIS_DT_BF16) return CLIS_ERR_UNSUPPORTED;
    if (variant != CLIS_AUTO && variant != CLIS_CERTIFIED_FORCED) return CLIS_ERR_INVALID_ARG;
    if (shape->B * shape->H != 0 && shape->Nq != 0) {
        if (!vt8) return CLIS_ERR_INVALID_ARG;
        if (!aligned16(vt8)) return CLIS_ERR_MISALIGNED;
    }
    return attn_chunk_impl(shape, q, k, v, o_acc, l_acc, m_acc, kbar, certs, nullptr, mu, scale_log2, 0, 0, first,
                           variant, stream, vt8);
}

clis_status_t clis_attn_fwd_chunk_causal(const clis_shape_t *shape, const void *q, const void *k, const void *v,
                                         float *o_acc, float *l_acc, float *m_acc, const float *kbar,
                                         const clis_head_cert_t *certs, const uint8_t *tile_certs, const float *mu,
                                         float scale_log2, int64_t key_offset, int first, clis_variant_t variant,
                                         clis_stream_t stream)
{
    return attn_chunk_impl(shape, q, k, v, o_acc, l_acc, m_acc, kbar, certs, tile_certs, mu, scale_log2, 1,
                           key_offset, first, variant, stream);
}

clis_status_t clis_attn_chunk_finalize(const clis_shape_t *shape, const float *o_acc, const float *l_acc,
                                       const float *m_acc, void *o, float *lse2, clis_stream_t stream)
{
    if (!shape) return CLIS_ERR_INVALID_ARG;
    if (shape->B < 0 || shape->H < 0 || shape->Nq < 0) return CLIS_ERR_INVALID_ARG;
    if (shape->d != 64 && shape->d != 128) return CLIS_ERR_UNSUPPORTED;
    if (shape->dtype != CLIS_DT_BF16 && shape->dtype != CLIS_DT_FP16) return CLIS_ERR_INVALID_ARG;
    if (shape->Nq > kMaxN || shape->B * shape->H > kMaxN) return CLIS_ERR_UNSUPPORTED;
    if (shape->B * shape->H == 0 || shape->Nq == 0) return CLIS_OK;
    if (!o_acc || !l_acc || !m_acc || !o) return CLIS_ERR_INVALID_ARG;
    clis_status_t st = check_strides(shape->o_sb, shape->o_sh, shape->o_sn, shape->d);
    if (st != CLIS_OK) return st;
    if (aliasing(shape->B, shape->H, shape->Nq, shape->o_sb, shape->o_sh)) return CLIS_ERR_INVALID_ARG;
    if (!aligned16(o_acc) || !aligned16(o) || (reinterpret_cast<uintptr_t>(l_acc) & 3u) ||
        (reinterpret_cast<uintptr_t>(m_acc) & 3u) || (lse2 && (reinterpret_cast<uintptr_t>(lse2) & 3u)))
        return CLIS_ERR_MISALIGNED;
    clis::ChunkFinalizeArgs a;
    a.o_acc = o_acc;
    a.l_acc = l_acc;
    a.m_acc = m_acc;
    a.o = static_cast<uint16_t *>(o);
    a.lse2 = lse2;
    a.o_sb = shape->o_sb;
    a.o_sh = shape->o_sh;
    a.o_sn = shape->o_sn;
    a.B = static_cast<int>(shape->B);
    a.H = static_cast<int>(shape->H);
    a.Nq = static_cast<int>(shape->Nq);
    a.d = static_cast<int>(shape->d);
    a.dtype = static_cast<int>(shape->dtype);
    return clis::launch_chunk_finalize(a, reinterpret_cast<cudaStream_t>(stream));
}

const char *clis_status_string(clis_status_t s)
{
    switch (s) {
    case CLIS_OK: return "ok";
    case CLIS_ERR_INVALID_ARG: return "invalid argument";
    case CLIS_ERR_UNSUPPORTED: return "unsupported shape or option";
    case CLIS_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case CLIS_ERR_WORKSPACE: return "workspace missing or too small";
    case CLIS_ERR_CUDA: return "CUDA call or kernel launch failed";
    case CLIS_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
    }
    return "unknown status";
}

clis_status_t clis_attn_bwd_workspace_size(const clis_shape_t *shape, size_t *bytes)
{
    if (!bytes) return CLIS_ERR_INVALID_ARG;
    clis_status_t st = check_shape(shape, true);
    if (st != CLIS_OK) return st;
    const int64_t rows = shape->B * shape->H * shape->Nq;
    *bytes = static_cast<size_t>(div_up(rows * 4, 256) * 256);
    return CLIS_OK;
}

clis_status_t clis_attn_bwd(const clis_shape_t *shape, const void *q, const void *k, const void *v, const void *o,
                            const void *dout, const float *lse2, void *dq, void *dk, void *dv, float scale_log2,
                            int causal, void *workspace, size_t ws_bytes, clis_stream_t stream)
{
    clis_status_t st = check_shape(shape, true);
    if (st != CLIS_OK) return st;
    // dQ, dK and dV are written with the Q, K and V strides.  K and V broadcast
    // over the heads together (both head strides 0: grouped-query attention
    // folded into the batch) are the one sharing allowed: the kernel then sums
    // the group's gradients and writes each dK, dV row once.
    const bool kv_bcast = shape->H > 1 && shape->k_sh == 0 && shape->v_sh == 0;
    if (aliasing(shape->B, shape->H, shape->Nq, shape->q_sb, shape->q_sh) ||
        aliasing(shape->B, kv_bcast ? 1 : shape->H, shape->Nk, shape->k_sb, shape->k_sh) ||
        aliasing(shape->B, kv_bcast ? 1 : shape->H, shape->Nk, shape->v_sb, shape->v_sh))
        return CLIS_ERR_INVALID_ARG;
    if (shape->B * shape->H == 0) return CLIS_OK;
    if (!std::isfinite(scale_log2) || !(scale_log2 > 0.f)) return CLIS_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return CLIS_ERR_INVALID_ARG;
    if (causal && shape->Nq != shape->Nk) return CLIS_ERR_UNSUPPORTED;
    if (!k || !v || !dk || !dv) return CLIS_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)) return CLIS_ERR_MISALIGNED;
    if (shape->Nq > 0) {
        if (!q || !o || !dout || !lse2 || !dq) return CLIS_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
            (reinterpret_cast<uintptr_t>(lse2) & 3u))
            return CLIS_ERR_MISALIGNED;
        size_t need = 0;
        clis_attn_bwd_workspace_size(shape, &need);
        if (!workspace || ws_bytes < need || !aligned16(workspace)) return CLIS_ERR_WORKSPACE;
    }
    const int64_t tiles = shape->B * shape->H * div_up(shape->Nk > shape->Nq ? shape->Nk : shape->Nq, 128);
    if (tiles > kMaxN) return CLIS_ERR_UNSUPPORTED;

    clis::AttnBwdArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.o = static_cast<const uint16_t *>(o);
    a.dout = static_cast<const uint16_t *>(dout);
    a.lse2 = lse2;
    a.dvec = static_cast<float *>(workspace);
    a.dq = static_cast<uint16_t *>(dq);
    a.dk = static_cast<uint16_t *>(dk);
    a.dv = static_cast<uint16_t *>(dv);
    a.q_sb = shape->q_sb;
    a.q_sh = shape->q_sh;
    a.q_sn = shape->q_sn;
    a.k_sb = shape->k_sb;
    a.k_sh = shape->k_sh;
    a.k_sn = shape->k_sn;
    a.v_sb = shape->v_sb;
    a.v_sh = shape->v_sh;
    a.v_sn = shape->v_sn;
    a.o_sb = shape->o_sb;
    a.o_sh = shape->o_sh;
    a.o_sn = shape->o_sn;
    a.B = static_cast<int>(shape->B);
    a.H = static_cast<int>(shape->H);
    a.Nq = static_cast<int>(shape->Nq);
    a.Nk = static_cast<int>(shape->Nk);
    a.d = static_cast<int>(shape->d);
    a.dtype = static_cast<int>(shape->dtype);
    a.scale_log2 = scale_log2;
    a.causal = causal;
    return clis::launch_attn_bwd(a, reinterpret_cast<cudaStream_t>(stream));
}

clis_status_t clis_get_device_error(uint32_t *code)
{
    if (!code) return CLIS_ERR_INVALID_ARG;
    uint32_t fwd = 0, bwd = 0;
    clis_status_t st = clis::read_device_error(&fwd);
    if (st == CLIS_ERR_CUDA) return st;
    if (clis::read_bwd_error(&bwd) != CLIS_OK) return CLIS_ERR_CUDA;
    *code = fwd | bwd;
    return *code ? CLIS_ERR_TIMEOUT : CLIS_OK;
}

clis_status_t clis_clear_device_error(void)
{
    clis_status_t st = clis::clear_device_error();
    return st != CLIS_OK ? st : clis::clear_bwd_error();
}

clis_status_t clis_debug_wait_selftest(uint32_t limit_us, clis_stream_t stream)
{
    if (limit_us < 1 || limit_us > 1000000) return CLIS_ERR_INVALID_ARG;
    return clis::launch_wait_selftest(limit_us, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
