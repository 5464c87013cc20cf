// certify.cu -- the CLiS certification pre-pass on the GPU.
//
// Implements Algorithm 1, steps 1-7, of "CLiS: Plug-and-Play Attention
// Acceleration for Video Diffusion on TPUs via Certified Stabilization" for
// every (b, h) head, plus the certification decision (finite inputs and
// B_h <= C).  Four launches, all HBM-bandwidth bound:
//
//   certify_ksum      per 1024-row chunk of K: fp32 column sums (step 1) and
//                     the max |k| bit pattern (non-finite detection)
//   certify_kbar      kbar = (sum of chunk sums in chunk order) / Nk
//   certify_norms     per chunk of K: max ||k - kbar||^2 (steps 2-3), of Q:
//                     max ||q||^2 (step 4), of Q and V: max |x| bit patterns
//                     (step 5 and non-finite detection)
//   certify_finalize  one warp per head: kappa, B_h, G, A, C and the flag
//
// K~ = K - 1 kbar^T (step 2) is never materialised: it is only needed inside
// the norm reduction, and the attention kernel moves kbar into the per-row
// stabiliser instead (softmax is invariant to a common key shift).
//
// Conservativeness: every quantity that bounds a score (|k - kbar|, the
// squares, their sums, the square roots and the products forming B_h) is
// rounded upward, so kappa and B_h are upper bounds of the exact values for
// the kbar this pass returns.  Determinism: sums run in a fixed order per
// thread and are combined in a fixed order; maxima are order-independent.
#include <cuda_bf16.h>

#include <mutex>

#include "clis_internal.h"
#include "sm103_ptx.cuh"

namespace clis {

// Scratch for clis_certify_noalloc: a fixed array owned by the library, so
// callers that cannot allocate still get a workspace.  Host code must not pass
// the symbol itself to a kernel (on the host it is only a stand-in); it uses
// the device address returned by certify_static_scratch().
static __device__ __align__(256) unsigned char g_certify_scratch[CLIS_NOALLOC_SCRATCH_BYTES];

namespace {

__device__ __forceinline__ uint32_t abs_bits_max(uint32_t u, uint32_t m)
{
    m = max(m, u & 0x7FFFu);
    m = max(m, (u >> 16) & 0x7FFFu);
    return m;
}

__device__ __forceinline__ uint4 ld_stream(const uint16_t *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red)
{
    __syncthreads();  // `red` may still be read by a previous call
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t x = (lane < (kCertThreads >> 5)) ? red[lane] : 0u;
        x = __reduce_max_sync(0xFFFFFFFFu, x);
        if (lane == 0) red[0] = x;
    }
    __syncthreads();
    return red[0];
}

// Step 1 (partial): column sums of one chunk of K, plus max |k| bits.
// DT: element type (0 bf16, 1 fp16); |x| bit patterns are x & 0x7FFF in both.
template <int D, int DT>
__global__ void __launch_bounds__(kCertThreads) certify_ksum_kernel(CertArgs a, CertWorkspace ws)
{
    constexpr int VPR = D / 8;             // 16-byte vectors per row
    constexpr int RPS = kCertThreads / VPR;  // rows per sweep
    __shared__ float red[RPS * D];
    __shared__ uint32_t redu[kCertThreads / 32];

    const int chunk = blockIdx.x % a.nck;
    const int bh = blockIdx.x / a.nck;
    const int b = bh / a.H, h = bh % a.H;
    const int cv = threadIdx.x % VPR, rp = threadIdx.x / VPR;
    const int r0 = chunk * kCertChunkRows;
    const int r1 = min(a.Nk, r0 + kCertChunkRows);
    const uint16_t *base = a.k + b * a.k_sb + h * a.k_sh + cv * 8;

    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; e++) acc[e] = 0.f;
    uint32_t amax = 0;
#pragma unroll 4
    for (int r = r0 + rp; r < r1; r += RPS) {
        const uint4 u = ld_stream(base + static_cast<int64_t>(r) * a.k_sn);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            acc[2 * e] += elem_lo<DT>(w[e]);
            acc[2 * e + 1] += elem_hi<DT>(w[e]);
            amax = abs_bits_max(w[e], amax);
        }
    }
#pragma unroll
    for (int e = 0; e < 8; e++) red[rp * D + cv * 8 + e] = acc[e];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kCertThreads) {
        float s = 0.f;
        for (int p = 0; p < RPS; p++) s += red[p * D + c];
        ws.ksum[(static_cast<int64_t>(bh) * a.nck + chunk) * D + c] = s;
    }
    const uint32_t m = block_max_u32(amax, redu);
    if (threadIdx.x == 0) ws.kabs[static_cast<int64_t>(bh) * a.nck + chunk] = m;
}

// Step 1 (final): kbar = sum_chunks / Nk, round to nearest.  Also clears the
// head's maxima that the norms kernel accumulates with atomicMax.
__global__ void certify_kbar_kernel(CertArgs a, CertWorkspace ws)
{
    const int bh = blockIdx.x;
    const int c = threadIdx.x;
    for (int i = c; i < a.nck; i += blockDim.x) {
        ws.knorm2[static_cast<int64_t>(bh) * a.nck + i] = 0u;
        ws.vabs[static_cast<int64_t>(bh) * a.nck + i] = 0u;
    }
    for (int i = c; i < a.ncq; i += blockDim.x) {
        ws.qnorm2[static_cast<int64_t>(bh) * a.ncq + i] = 0u;
        ws.qabs[static_cast<int64_t>(bh) * a.ncq + i] = 0u;
    }
    if (c >= a.d) return;
    float s = 0.f;
    for (int ch = 0; ch < a.nck; ch++) s += ws.ksum[(static_cast<int64_t>(bh) * a.nck + ch) * a.d + c];
    a.kbar[static_cast<int64_t>(bh) * a.d + c] = __fdiv_rn(s, static_cast<float>(a.Nk));
}

// Steps 2-5 (partial): one quarter of a chunk of K (centred norms), Q (norms)
// or V (|v|).  Quarter-chunk blocks keep the last wave of the grid short; the
// four quarters of a chunk meet in its partial maximum through atomicMax on the
// bit patterns of non-negative floats, which is exact and order-independent.
template <int D, int DT>
__global__ void __launch_bounds__(kCertThreads) certify_norms_kernel(CertArgs a, CertWorkspace ws)
{
    constexpr int VPR = D / 8;
    constexpr int RPS = kCertThreads / VPR;
    constexpr int SUB = kCertChunkRows / kCertNormSplit;  // rows per block
    __shared__ uint32_t redu[kCertThreads / 32];

    const int per_head = kCertNormSplit * (2 * a.nck + a.ncq);
    const int bh = blockIdx.x / per_head;
    int sub = blockIdx.x % per_head;
    const int b = bh / a.H, h = bh % a.H;
    const int cv = threadIdx.x % VPR, rp = threadIdx.x / VPR;

    int kind;  // 0 = K, 1 = Q, 2 = V
    if (sub < kCertNormSplit * a.nck) {
        kind = 0;
    } else if (sub < kCertNormSplit * (a.nck + a.ncq)) {
        kind = 1;
        sub -= kCertNormSplit * a.nck;
    } else {
        kind = 2;
        sub -= kCertNormSplit * (a.nck + a.ncq);
    }
    const int part = sub / kCertNormSplit;  // chunk whose partial this block feeds
    const int nrows = (kind == 1) ? a.Nq : a.Nk;
    const int r0 = min(nrows, sub * SUB);
    const int r1 = min(nrows, r0 + SUB);
    const int nsweeps = (r1 - r0 + RPS - 1) / RPS;  // uniform across the block

    if (kind == 0) {
        float kb[8];
#pragma unroll
        for (int e = 0; e < 8; e++) kb[e] = a.kbar[static_cast<int64_t>(bh) * D + cv * 8 + e];
        const uint16_t *base = a.k + b * a.k_sb + h * a.k_sh + cv * 8;
        float mx = 0.f;
#pragma unroll 4
        for (int sw = 0; sw < nsweeps; sw++) {
            const int r = r0 + sw * RPS + rp;
            // Every lane runs the same number of sweeps (the shuffles below
            // need all 32 lanes of the warp); rows past r1 contribute nothing.
            float ss = 0.f;
            if (r < r1) {
                const uint4 u = ld_stream(base + static_cast<int64_t>(r) * a.k_sn);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float x0 = elem_lo<DT>(w[e]), x1 = elem_hi<DT>(w[e]);
                    const float d0 = (x0 >= kb[2 * e]) ? __fsub_ru(x0, kb[2 * e]) : __fsub_ru(kb[2 * e], x0);
                    const float d1 = (x1 >= kb[2 * e + 1]) ? __fsub_ru(x1, kb[2 * e + 1])
                                                           : __fsub_ru(kb[2 * e + 1], x1);
                    ss = __fmaf_ru(d0, d0, ss);
                    ss = __fmaf_ru(d1, d1, ss);
                }
            }
#pragma unroll
            for (int off = 1; off < VPR; off <<= 1) ss = __fadd_ru(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
            mx = fmaxf(mx, ss);
        }
        const uint32_t m = block_max_u32(__float_as_uint(mx), redu);
        if (threadIdx.x == 0) {
            atomicMax(&ws.knorm2[static_cast<int64_t>(bh) * a.nck + part], m);
            ws.knorm2s[static_cast<int64_t>(bh) * kCertNormSplit * a.nck + sub] = m;
        }
    } else if (kind == 1) {
        const uint16_t *base = a.q + b * a.q_sb + h * a.q_sh + cv * 8;
        float mx = 0.f;
        uint32_t amax = 0;
        // Optional per-row stabiliser mu_i = scale_log2 * (q_i . kbar) for the
        // attention kernel (the shift Figure 5(a) fixes before the KV loop).
        float kb[8];
#pragma unroll
        for (int e = 0; e < 8; e++) kb[e] = a.mu ? a.kbar[static_cast<int64_t>(bh) * D + cv * 8 + e] : 0.f;
#pragma unroll 4
        for (int sw = 0; sw < nsweeps; sw++) {
            const int r = r0 + sw * RPS + rp;
            float ss = 0.f, dot = 0.f;
            if (r < r1) {
                const uint4 u = ld_stream(base + static_cast<int64_t>(r) * a.q_sn);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float x0 = elem_lo<DT>(w[e]), x1 = elem_hi<DT>(w[e]);
                    ss = __fmaf_ru(x0, x0, ss);
                    ss = __fmaf_ru(x1, x1, ss);
                    dot = fmaf(x0, kb[2 * e], dot);
                    dot = fmaf(x1, kb[2 * e + 1], dot);
                    amax = abs_bits_max(w[e], amax);
                }
            }
#pragma unroll
            for (int off = 1; off < VPR; off <<= 1) {
                ss = __fadd_ru(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
                dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
            }
            mx = fmaxf(mx, ss);
            if (a.mu && cv == 0 && r < r1) a.mu[static_cast<int64_t>(bh) * a.Nq + r] = a.scale_log2 * dot;
        }
        const uint32_t m = block_max_u32(__float_as_uint(mx), redu);
        const uint32_t am = block_max_u32(amax, redu);
        if (threadIdx.x == 0) {
            atomicMax(&ws.qnorm2[static_cast<int64_t>(bh) * a.ncq + part], m);
            atomicMax(&ws.qabs[static_cast<int64_t>(bh) * a.ncq + part], am);
            ws.qnorm2s[static_cast<int64_t>(bh) * kCertNormSplit * a.ncq + sub] = m;
        }
    } else {
        const uint16_t *base = a.v + b * a.v_sb + h * a.v_sh + cv * 8;
        uint32_t amax = 0;
#pragma unroll 4
        for (int r = r0 + rp; r < r1; r += RPS) {
            const uint4 u = ld_stream(base + static_cast<int64_t>(r) * a.v_sn);
            amax = abs_bits_max(u.x, amax);
            amax = abs_bits_max(u.y, amax);
            amax = abs_bits_max(u.z, amax);
            amax = abs_bits_max(u.w, amax);
        }
        const uint32_t am = block_max_u32(amax, redu);
        if (threadIdx.x == 0) atomicMax(&ws.vabs[static_cast<int64_t>(bh) * a.nck + part], am);
    }
}

// ceil(log2 n) for n >= 1, in integers.
__device__ __forceinline__ int ceil_log2_i64(int64_t n)
{
    return (n <= 1) ? 0 : 64 - __clzll(static_cast<unsigned long long>(n - 1));
}

// G = ceil(log2 max(1, m)) for the magnitude m with bit pattern `bits` (sign
// cleared, finite).  bf16: m = (1 + f/2^7) 2^(e-127); fp16: m = (1 + f/2^10)
// 2^(e-15) for a normal number; m <= 1 (zero, subnormals, 1.0) gives 0.
__device__ __forceinline__ int v_exponent_from_bits(uint32_t bits, int dtype)
{
    if (dtype == CLIS_DT_FP16) {
        if (bits <= 0x3C00u) return 0;
        return (static_cast<int>(bits >> 10) - 15) + ((bits & 0x3FFu) != 0u ? 1 : 0);
    }
    if (bits <= 0x3F80u) return 0;
    return (static_cast<int>(bits >> 7) - 127) + ((bits & 0x7Fu) != 0u ? 1 : 0);
}

// Steps 3-7 and the decision: one warp per head.
__global__ void certify_finalize_kernel(CertArgs a, CertWorkspace ws, int BH)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= BH) return;
    const int64_t bh = warp;
    uint32_t kn = 0, ka = 0, va = 0, qn = 0, qa = 0;
    for (int c = lane; c < a.nck; c += 32) {
        kn = max(kn, ws.knorm2[bh * a.nck + c]);
        ka = max(ka, ws.kabs[bh * a.nck + c]);
        va = max(va, ws.vabs[bh * a.nck + c]);
    }
    for (int c = lane; c < a.ncq; c += 32) {
        qn = max(qn, ws.qnorm2[bh * a.ncq + c]);
        qa = max(qa, ws.qabs[bh * a.ncq + c]);
    }
    kn = __reduce_max_sync(0xFFFFFFFFu, kn);
    ka = __reduce_max_sync(0xFFFFFFFFu, ka);
    va = __reduce_max_sync(0xFFFFFFFFu, va);
    qn = __reduce_max_sync(0xFFFFFFFFu, qn);
    qa = __reduce_max_sync(0xFFFFFFFFu, qa);
    if (lane != 0) return;

    clis_head_cert_t c;
    const uint32_t inf_bits = (a.dtype == CLIS_DT_FP16) ? 0x7C00u : 0x7F80u;  // |x| of +infinity
    const bool finite = ka < inf_bits && va < inf_bits && qa < inf_bits;
    c.kappa = __fsqrt_ru(__uint_as_float(kn));   // step 3
    c.qmax = __fsqrt_ru(__uint_as_float(qn));
    if (!finite) {
        c.certified = 0;
        c.reason = 2;
        c.G = c.A = c.C = 0;
        c.B_h = __int_as_float(0x7F800000);
    } else {
        c.B_h = __fmul_ru(__fmul_ru(a.scale_log2, c.qmax), c.kappa);  // step 4
        c.G = v_exponent_from_bits(va, a.dtype);                       // step 5
        c.A = ceil_log2_i64(a.Nk) + c.G;                               // step 6
        // step 7: floor(U_exp) = emax_exp and ceil(U_acc - A) - 1 = emax_acc - A,
        // because log2 of a format's largest finite value lies in (emax, emax + 1).
        c.C = min(a.emax_exp, a.emax_acc - c.A);
        c.certified = (c.B_h <= static_cast<float>(c.C)) ? 1 : 0;
        c.reason = c.certified ? 0 : 1;
    }
    a.certs[bh] = c;
    if (a.tile_certs) {
        // Per-prefix certificates of a causal head: query block b (rows 256b ..
        // 256b + 255) sees keys 0 .. 256b + 255 only, so its bound takes the
        // block's largest query norm and the largest centred key norm of that
        // prefix, rounded up as B_h is; it is compared with the head's budget C.
        uint8_t *tc = a.tile_certs + bh * a.nqb;
        const uint32_t *ks = ws.knorm2s + bh * kCertNormSplit * a.nck;
        const uint32_t *qs = ws.qnorm2s + bh * kCertNormSplit * a.ncq;
        uint32_t kpre = 0;
        for (int b = 0; b < a.nqb; b++) {
            kpre = max(kpre, ks[b]);
            const float Bb = __fmul_ru(__fmul_ru(a.scale_log2, __fsqrt_ru(__uint_as_float(qs[b]))),
                                       __fsqrt_ru(__uint_as_float(kpre)));
            tc[b] = (finite && Bb <= static_cast<float>(c.C)) ? 1 : 0;
        }
    }
}

}  // namespace

size_t cert_workspace_layout(int64_t BH, int64_t nck, int64_t ncq, int64_t d, void *base, CertWorkspace *ws)
{
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    size_t off = 0;
    const size_t o_ksum = off;
    off = up(off + static_cast<size_t>(BH * nck * d) * sizeof(float));
    const size_t o_knorm = off;
    off = up(off + static_cast<size_t>(BH * nck) * 4);
    const size_t o_qnorm = off;
    off = up(off + static_cast<size_t>(BH * ncq) * 4);
    const size_t o_kabs = off;
    off = up(off + static_cast<size_t>(BH * nck) * 4);
    const size_t o_qabs = off;
    off = up(off + static_cast<size_t>(BH * ncq) * 4);
    const size_t o_vabs = off;
    off = up(off + static_cast<size_t>(BH * nck) * 4);
    const size_t o_knorms = off;
    off = up(off + static_cast<size_t>(BH * kCertNormSplit * nck) * 4);
    const size_t o_qnorms = off;
    off = up(off + static_cast<size_t>(BH * kCertNormSplit * ncq) * 4);
    if (ws && base) {
        char *p = static_cast<char *>(base);
        ws->ksum = reinterpret_cast<float *>(p + o_ksum);
        ws->knorm2 = reinterpret_cast<uint32_t *>(p + o_knorm);
        ws->qnorm2 = reinterpret_cast<uint32_t *>(p + o_qnorm);
        ws->kabs = reinterpret_cast<uint32_t *>(p + o_kabs);
        ws->qabs = reinterpret_cast<uint32_t *>(p + o_qabs);
        ws->vabs = reinterpret_cast<uint32_t *>(p + o_vabs);
        ws->knorm2s = reinterpret_cast<uint32_t *>(p + o_knorms);
        ws->qnorm2s = reinterpret_cast<uint32_t *>(p + o_qnorms);
    }
    return off;
}

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry point (no libcuda link).
CtxGetCurrentFn get_ctx_fn()
{
    static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(ptr);
        return nullptr;
    }();
    return fn;
}

}  // namespace

void *certify_static_scratch(cudaStream_t stream)
{
    // The array's device address belongs to one context (each context loads
    // its own copy of the module, and a device reset replaces the primary
    // context), so addresses are kept per (device, context).  Outside stream
    // capture the address is looked up afresh on every call; during capture the
    // one looked up by the last call outside capture in the same context is used.
    constexpr int kSlots = 64;
    struct Slot {
        int dev;
        CUcontext ctx;
        void *addr;
    };
    static std::mutex mu;
    static Slot slots[kSlots];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return nullptr;
    void *ptr = nullptr;
    // Outside capture: look the address up first (this also makes the device's
    // primary context current when the thread has no context yet).
    if (cs == cudaStreamCaptureStatusNone &&
        (cudaGetSymbolAddress(&ptr, g_certify_scratch) != cudaSuccess || !ptr))
        return nullptr;
    CtxGetCurrentFn ctx_fn = get_ctx_fn();
    CUcontext ctx = nullptr;
    if (!ctx_fn || ctx_fn(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    int slot = -1;
    for (int i = 0; i < used; i++)
        if (slots[i].dev == dev && slots[i].ctx == ctx) slot = i;
    if (cs != cudaStreamCaptureStatusNone) return slot >= 0 ? slots[slot].addr : nullptr;
    if (slot < 0) {
        // Table full (many contexts over the process's life): reuse the first slot.
        slot = used < kSlots ? used++ : 0;
        slots[slot].dev = dev;
        slots[slot].ctx = ctx;
    }
    slots[slot].addr = ptr;
    return ptr;
}

cudaError_t launch_certify(const CertArgs &a, const CertWorkspace &ws, cudaStream_t stream)
{
    const int BH = a.B * a.H;
    if (BH == 0) return cudaSuccess;
    const unsigned g1 = static_cast<unsigned>(BH) * static_cast<unsigned>(a.nck);
    const unsigned g3 = static_cast<unsigned>(BH) * static_cast<unsigned>(kCertNormSplit * (2 * a.nck + a.ncq));
    const bool f16 = a.dtype == CLIS_DT_FP16;
    if (a.d == 128) {
        if (f16) certify_ksum_kernel<128, 1><<<g1, kCertThreads, 0, stream>>>(a, ws);
        else certify_ksum_kernel<128, 0><<<g1, kCertThreads, 0, stream>>>(a, ws);
    } else {
        if (f16) certify_ksum_kernel<64, 1><<<g1, kCertThreads, 0, stream>>>(a, ws);
        else certify_ksum_kernel<64, 0><<<g1, kCertThreads, 0, stream>>>(a, ws);
    }
    certify_kbar_kernel<<<BH, 128, 0, stream>>>(a, ws);
    if (a.d == 128) {
        if (f16) certify_norms_kernel<128, 1><<<g3, kCertThreads, 0, stream>>>(a, ws);
        else certify_norms_kernel<128, 0><<<g3, kCertThreads, 0, stream>>>(a, ws);
    } else {
        if (f16) certify_norms_kernel<64, 1><<<g3, kCertThreads, 0, stream>>>(a, ws);
        else certify_norms_kernel<64, 0><<<g3, kCertThreads, 0, stream>>>(a, ws);
    }
    certify_finalize_kernel<<<(BH + 3) / 4, 128, 0, stream>>>(a, ws, BH);
    return cudaGetLastError();
}

}  // namespace clis
