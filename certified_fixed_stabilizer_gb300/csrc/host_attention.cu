// host_attention.cu -- the attention forward for Q, K, V and O held in host
// memory: each group of heads is copied in, certified and attended on the
// device, and copied out, with the copies of one group overlapping the
// kernels of others.  Host code only; the kernels are the ones behind
// clis_certify and clis_attn_fwd.
//
// A plan (one shape, one device) owns four streams and the events below:
// s_in carries every copy to the device, s_run[0] and s_run[1] the kernels of
// even and odd groups (so that one group's launch can take the SMs the
// previous group's tail leaves idle; heads are independent), s_out every copy
// back.  Per call and group g:
//   s_in:       wait ev_run[g] of the previous call (its kernels have read
//               the staging of g); copy Q, K, V of g -> record ev_in
//   s_run[g%2]: wait ev_in; wait ev_out[g] of the previous call (the O
//               staging of g has been copied out); certify g; attention g
//               -> record ev_run[g]
//   s_out:      wait ev_run[g]; copy O of g back -> record ev_out[g]
// so consecutive calls overlap: a call's copies of a group start as soon as
// the previous call's kernels on that group are done.  ev_in is re-recorded
// for the next group only after the wait on its previous recording is queued
// (a wait takes the event's state when it is queued).  ev_done follows the
// last copy out; clis_host_plan_wait queues a wait for it.
#include <cmath>
#include <cstdint>
#include <new>

#include "clis_internal.h"

namespace {

constexpr int64_t kMaxN = (int64_t(1) << 31) - 1024;
constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Dense [B, H, N, d]: n-stride d, head stride N*d, batch stride H*N*d (the
// batch stride is free when B == 1).
bool dense(int64_t B, int64_t H, int64_t N, int64_t d, int64_t sb, int64_t sh, int64_t sn)
{
    return sn == d && sh == N * d && (B <= 1 || sb == H * N * d);
}

struct Plan {
    int64_t heads = 0, per = 0, groups = 0;
    size_t q_head = 0, kv_head = 0;  // bytes of one head of Q (or O) and of K (or V)
    size_t off_kbar = 0, off_certs = 0, off_mu = 0, off_q = 0, off_k = 0, off_v = 0, off_o = 0;
    size_t off_ws[2] = {0, 0}, ws_each = 0, total = 0;
};

// The shape of heads [f0, f0 + n) of the dense staging buffers as one batch entry.
clis_shape_t group_shape(const clis_shape_t &s, int64_t n)
{
    clis_shape_t g = s;
    g.B = 1;
    g.H = n;
    g.q_sn = g.k_sn = g.v_sn = g.o_sn = s.d;
    g.q_sh = g.o_sh = s.Nq * s.d;
    g.k_sh = g.v_sh = s.Nk * s.d;
    // B == 1: the batch stride is never multiplied by a non-zero index.
    g.q_sb = g.q_sh;
    g.o_sb = g.o_sh;
    g.k_sb = g.k_sh;
    g.v_sb = g.v_sh;
    return g;
}

// Argument checks shared by both entry points (no pointers); fills the plan.
clis_status_t make_plan(const clis_shape_t *s, int causal, int groups, Plan *P)
{
    if (!s) return CLIS_ERR_INVALID_ARG;
    if (s->B < 0 || s->H < 0 || s->Nq < 0 || s->Nk < 1 || s->d < 1) return CLIS_ERR_INVALID_ARG;
    if (s->dtype != CLIS_DT_BF16 && s->dtype != CLIS_DT_FP16) return CLIS_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return CLIS_ERR_INVALID_ARG;
    if (groups < 0) return CLIS_ERR_INVALID_ARG;
    if (s->d != 64 && s->d != 128) return CLIS_ERR_UNSUPPORTED;
    if (causal && s->Nq != s->Nk) return CLIS_ERR_UNSUPPORTED;
    if (s->Nq > kMaxN || s->Nk > kMaxN || s->B > kMaxN || s->H > kMaxN || s->B * s->H > kMaxN)
        return CLIS_ERR_UNSUPPORTED;
    if (!dense(s->B, s->H, s->Nq, s->d, s->q_sb, s->q_sh, s->q_sn) ||
        !dense(s->B, s->H, s->Nk, s->d, s->k_sb, s->k_sh, s->k_sn) ||
        !dense(s->B, s->H, s->Nk, s->d, s->v_sb, s->v_sh, s->v_sn) ||
        !dense(s->B, s->H, s->Nq, s->d, s->o_sb, s->o_sh, s->o_sn))
        return CLIS_ERR_UNSUPPORTED;
    // Sizes the kernels behind clis_certify and clis_attn_fwd index with int32
    // (checked here for all heads at once, so that no group fails later).
    const int64_t heads = s->B * s->H;
    const int64_t nck = div_up(s->Nk, clis::kCertChunkRows), ncq = div_up(s->Nq, clis::kCertChunkRows);
    if (clis::kCertNormSplit * heads * (2 * nck + ncq) > kMaxN ||
        heads * div_up(s->Nq, clis::kQueryBlockRows) > kMaxN)
        return CLIS_ERR_UNSUPPORTED;

    P->heads = heads;
    if (heads == 0 || s->Nq == 0) return CLIS_OK;  // nothing to compute, no workspace
    if (groups == 0) {
        // About one group per 2 TFLOP of attention work (~1.2 ms): only the first
        // group's copies in and the last group's copy out are left exposed.
        const double work = 4.0 * static_cast<double>(heads) * static_cast<double>(s->Nq) *
                            static_cast<double>(s->Nk) * static_cast<double>(s->d) / (causal ? 2.0 : 1.0);
        const double g = work / 2e12;
        groups = static_cast<int>(g < 8.0 ? 8.0 : (g > static_cast<double>(heads) ? static_cast<double>(heads) : g));
    }
    if (groups > heads) groups = static_cast<int>(heads);
    P->per = div_up(heads, groups);
    P->groups = div_up(heads, P->per);
    const size_t es = 2;
    P->q_head = static_cast<size_t>(s->Nq) * static_cast<size_t>(s->d) * es;
    P->kv_head = static_cast<size_t>(s->Nk) * static_cast<size_t>(s->d) * es;
    const clis_shape_t gs = group_shape(*s, P->per);
    size_t ws = 0;
    const clis_status_t st = clis_certify_workspace_size(&gs, &ws);
    if (st != CLIS_OK) return st;
    const size_t h = static_cast<size_t>(heads);
    size_t off = 0;
    P->off_kbar = off;
    off += up(h * static_cast<size_t>(s->d) * sizeof(float));
    P->off_certs = off;
    off += up(h * sizeof(clis_head_cert_t));
    P->off_mu = off;
    off += up(h * static_cast<size_t>(s->Nq) * sizeof(float));
    P->off_q = off;
    off += up(h * P->q_head);
    P->off_k = off;
    off += up(h * P->kv_head);
    P->off_v = off;
    off += up(h * P->kv_head);
    P->off_o = off;
    off += up(h * P->q_head);
    P->ws_each = up(ws);
    P->off_ws[0] = off;
    off += P->ws_each;
    P->off_ws[1] = off;
    off += P->ws_each;
    P->total = off;
    return CLIS_OK;
}

}  // namespace

struct clis_host_plan_s {
    clis_shape_t shape;
    int causal = 0;
    int device = 0;
    Plan P;
    bool used = false;  // a call has queued work (the per-group events are recorded)
    cudaStream_t s_in = nullptr, s_out = nullptr, s_run[2] = {nullptr, nullptr};
    cudaEvent_t ev_entry = nullptr, ev_in = nullptr, ev_done = nullptr;
    cudaEvent_t *ev_run = nullptr, *ev_out = nullptr;  // [groups] each
};

namespace {

void release(clis_host_plan_t *h)
{
    for (cudaEvent_t e : {h->ev_entry, h->ev_in, h->ev_done})
        if (e) cudaEventDestroy(e);
    for (int64_t g = 0; g < h->P.groups; g++) {
        if (h->ev_run && h->ev_run[g]) cudaEventDestroy(h->ev_run[g]);
        if (h->ev_out && h->ev_out[g]) cudaEventDestroy(h->ev_out[g]);
    }
    for (cudaStream_t s : {h->s_in, h->s_out, h->s_run[0], h->s_run[1]})
        if (s) cudaStreamDestroy(s);
    delete[] h->ev_run;
    delete[] h->ev_out;
    delete h;
}

bool make_event(cudaEvent_t *e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; }

}  // namespace

extern "C" {

clis_status_t clis_host_plan_create(const clis_shape_t *shape, int causal, int groups, clis_host_plan_t **plan)
{
    if (!plan) return CLIS_ERR_INVALID_ARG;
    *plan = nullptr;
    Plan P;
    const clis_status_t st = make_plan(shape, causal, groups, &P);
    if (st != CLIS_OK) return st;
    clis_host_plan_t *h = new (std::nothrow) clis_host_plan_t;
    if (!h) return CLIS_ERR_CUDA;
    h->shape = *shape;
    h->causal = causal;
    h->P = P;
    // Nothing to compute (B*H = 0 or Nq = 0): no streams, no events, no CUDA call.
    bool ok = P.groups == 0 || cudaGetDevice(&h->device) == cudaSuccess;
    if (ok && P.groups > 0) {
        h->ev_run = new (std::nothrow) cudaEvent_t[P.groups]();
        h->ev_out = new (std::nothrow) cudaEvent_t[P.groups]();
        ok = h->ev_run && h->ev_out;
        for (cudaStream_t *s : {&h->s_in, &h->s_out, &h->s_run[0], &h->s_run[1]})
            ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
        ok = ok && make_event(&h->ev_entry) && make_event(&h->ev_in) && make_event(&h->ev_done);
        for (int64_t g = 0; ok && g < P.groups; g++) ok = make_event(&h->ev_run[g]) && make_event(&h->ev_out[g]);
    }
    if (!ok) {
        release(h);  // destroys what was created (the event arrays start zeroed)
        return CLIS_ERR_CUDA;
    }
    *plan = h;
    return CLIS_OK;
}

clis_status_t clis_host_plan_workspace_size(const clis_host_plan_t *plan, size_t *bytes)
{
    if (!plan || !bytes) return CLIS_ERR_INVALID_ARG;
    *bytes = plan->P.total;
    return CLIS_OK;
}

clis_status_t clis_host_plan_wait(clis_host_plan_t *plan, clis_stream_t stream)
{
    if (!plan) return CLIS_ERR_INVALID_ARG;
    if (!plan->used) return CLIS_OK;
    return cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), plan->ev_done, 0) == cudaSuccess
               ? CLIS_OK
               : CLIS_ERR_CUDA;
}

clis_status_t clis_host_plan_destroy(clis_host_plan_t *plan)
{
    if (!plan) return CLIS_OK;
    // Queued work keeps running; the runtime frees the streams and events after it.
    release(plan);
    return CLIS_OK;
}

clis_status_t clis_attention_host(clis_host_plan_t *plan, const void *q, const void *k, const void *v, void *o,
                                  float scale_log2, clis_variant_t variant, void *workspace, size_t ws_bytes,
                                  clis_stream_t stream)
{
    if (!plan) return CLIS_ERR_INVALID_ARG;
    const clis_shape_t *shape = &plan->shape;
    const Plan &P = plan->P;
    if (!std::isfinite(scale_log2) || !(scale_log2 > 0.f)) return CLIS_ERR_INVALID_ARG;
    if (variant != CLIS_AUTO && variant != CLIS_ONLINE && variant != CLIS_CERTIFIED_FORCED &&
        variant != CLIS_ONLINE_LAZY)
        return CLIS_ERR_INVALID_ARG;
    if (P.heads == 0 || shape->Nq == 0) return CLIS_OK;  // nothing to compute
    if (!q || !k || !v || !o) return CLIS_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < P.total) return CLIS_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return CLIS_ERR_MISALIGNED;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLIS_ERR_CUDA;
    if (dev != plan->device) return CLIS_ERR_INVALID_ARG;  // the plan's streams live on its device

    const bool certified = variant == CLIS_AUTO || variant == CLIS_CERTIFIED_FORCED;
    const clis_fmt_t exp_fmt = shape->dtype == CLIS_DT_FP16 ? CLIS_FMT_FP16 : CLIS_FMT_BF16;
    uint8_t *base = static_cast<uint8_t *>(workspace);
    float *kbar = reinterpret_cast<float *>(base + P.off_kbar);
    clis_head_cert_t *certs = reinterpret_cast<clis_head_cert_t *>(base + P.off_certs);
    float *mu = reinterpret_cast<float *>(base + P.off_mu);
    uint8_t *dq = base + P.off_q, *dk = base + P.off_k, *dv = base + P.off_v, *dout = base + P.off_o;
    const uint8_t *hq = static_cast<const uint8_t *>(q), *hk = static_cast<const uint8_t *>(k),
                  *hv = static_cast<const uint8_t *>(v);
    uint8_t *ho = static_cast<uint8_t *>(o);
    const cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
    const bool after_previous = plan->used;

    // The copies in follow whatever the caller queued on its stream before.
    clis_status_t st = CLIS_OK;
    bool ok = cudaEventRecord(plan->ev_entry, user) == cudaSuccess &&
              cudaStreamWaitEvent(plan->s_in, plan->ev_entry, 0) == cudaSuccess;
    bool queued = false;
    for (int64_t g = 0; ok && g < P.groups; g++) {
        const int64_t f0 = g * P.per;
        const int64_t n = (f0 + P.per <= P.heads) ? P.per : P.heads - f0;
        const size_t qo_off = static_cast<size_t>(f0) * P.q_head, kv_off = static_cast<size_t>(f0) * P.kv_head;
        const size_t qo_len = static_cast<size_t>(n) * P.q_head, kv_len = static_cast<size_t>(n) * P.kv_head;
        cudaStream_t run = plan->s_run[g & 1];
        queued = true;
        ok = (!after_previous || cudaStreamWaitEvent(plan->s_in, plan->ev_run[g], 0) == cudaSuccess) &&
             cudaMemcpyAsync(dq + qo_off, hq + qo_off, qo_len, cudaMemcpyHostToDevice, plan->s_in) == cudaSuccess &&
             cudaMemcpyAsync(dk + kv_off, hk + kv_off, kv_len, cudaMemcpyHostToDevice, plan->s_in) == cudaSuccess &&
             cudaMemcpyAsync(dv + kv_off, hv + kv_off, kv_len, cudaMemcpyHostToDevice, plan->s_in) == cudaSuccess &&
             cudaEventRecord(plan->ev_in, plan->s_in) == cudaSuccess &&
             cudaStreamWaitEvent(run, plan->ev_in, 0) == cudaSuccess &&
             (!after_previous || cudaStreamWaitEvent(run, plan->ev_out[g], 0) == cudaSuccess);
        if (!ok) break;
        const clis_shape_t gs = group_shape(*shape, n);
        float *gkbar = certified ? kbar + f0 * shape->d : nullptr;
        clis_head_cert_t *gcerts = certified ? certs + f0 : nullptr;
        float *gmu = certified ? mu + f0 * shape->Nq : nullptr;
        if (certified) {
            st = clis_certify(&gs, dq + qo_off, dk + kv_off, dv + kv_off, scale_log2, exp_fmt, CLIS_FMT_FP32, gkbar,
                              gcerts, gmu, base + P.off_ws[g & 1], P.ws_each, reinterpret_cast<clis_stream_t>(run));
            if (st != CLIS_OK) break;
        }
        st = clis_attn_fwd(&gs, dq + qo_off, dk + kv_off, dv + kv_off, dout + qo_off, nullptr, gkbar, gcerts, gmu,
                           scale_log2, plan->causal, variant, reinterpret_cast<clis_stream_t>(run));
        if (st != CLIS_OK) break;
        ok = cudaEventRecord(plan->ev_run[g], run) == cudaSuccess &&
             cudaStreamWaitEvent(plan->s_out, plan->ev_run[g], 0) == cudaSuccess &&
             cudaMemcpyAsync(ho + qo_off, dout + qo_off, qo_len, cudaMemcpyDeviceToHost, plan->s_out) == cudaSuccess &&
             cudaEventRecord(plan->ev_out[g], plan->s_out) == cudaSuccess;
    }
    if (!ok && st == CLIS_OK) st = CLIS_ERR_CUDA;
    if (queued) {
        // ev_done follows everything queued above (on an error too, so that a
        // wait for it covers every copy and kernel of the call), and every
        // group's events are recorded again, so the next call waits for this one.
        bool joined = true;
        if (st != CLIS_OK) {
            for (cudaStream_t s : {plan->s_in, plan->s_run[0], plan->s_run[1]})
                joined = joined && cudaEventRecord(plan->ev_in, s) == cudaSuccess &&
                         cudaStreamWaitEvent(plan->s_out, plan->ev_in, 0) == cudaSuccess;
        }
        joined = joined && cudaEventRecord(plan->ev_done, plan->s_out) == cudaSuccess;
        if (st != CLIS_OK)
            for (int64_t g = 0; joined && g < P.groups; g++)
                joined = cudaEventRecord(plan->ev_run[g], plan->s_out) == cudaSuccess &&
                         cudaEventRecord(plan->ev_out[g], plan->s_out) == cudaSuccess;
        if (!joined) {
            // The events cannot order what follows: wait for the work here.
            for (cudaStream_t s : {plan->s_in, plan->s_run[0], plan->s_run[1], plan->s_out}) cudaStreamSynchronize(s);
            if (st == CLIS_OK) st = CLIS_ERR_CUDA;
        }
        plan->used = true;
    }
    return st;
}

}  // extern "C"
