// attn_bwd.cu -- attention backward for sm_103a: dQ, dK, dV of L = sum(dO * O).
//
// The pages report CLiS training results for causal LLMs ("CLiS: Plug-and-Play
// Attention Acceleration for Video Diffusion on TPUs via Certified
// Stabilization", Table 3) but give no backward algorithm, so this is the
// plain chain rule through softmax.  With x_ij = scale_log2 * q_i . k_j (exp2
// units) and the forward's row statistic lse2_i = log2 sum_j 2^x_ij:
//
//   P_ij  = 2^(x_ij - lse2_i)            (exact softmax weights)
//   D_i   = dO_i . O_i                    (= sum_j P_ij dP_ij)
//   dP_ij = dO_i . v_j
//   dS_ij = P_ij (dP_ij - D_i)            (gradient w.r.t. the natural-log logits)
//   dV_j  = sum_i P_ij dO_i
//   dK_j  = scale * sum_i dS_ij q_i,   dQ_i = scale * sum_j dS_ij k_j
//
// where scale = scale_log2 * ln 2 is the softmax scale.  lse2_i is the same
// quantity for both forward paths (mu_i + log2 l_i on the certified path,
// m_i + log2 l_i online), so the backward is one fixed-stabiliser pass: P is
// normalised from the start and no running maximum or rescale exists here.
//
// Three launches:
//   bwd_dot_kernel     D_i, one fp32 per query row (HBM stream of O and dO)
//   bwd_dkdv_kernel    persistent; a work tile is 128 keys of one head, kept in
//                      shared memory while the query blocks stream past:
//                        S^T = K Q^T, dP^T = V dO^T          (SMEM x SMEM)
//                        dV += P^T dO, dK += dS^T Q          (P^T, dS^T from TMEM)
//                      (when K and V are shared by all the heads of a batch entry,
//                      zero head stride, the query blocks of every one of those
//                      heads stream past in turn, so dK and dV sum the group)
//   bwd_dq_kernel      persistent; a work tile is 128 queries of one head:
//                        S = Q K^T, dP = dO V^T, dQ += dS K
// Splitting dQ from dK/dV recomputes S and dP once more (7 matmuls per
// block pair instead of 5) but needs no atomics: every output element is
// written once, in a fixed summation order, so results are deterministic.
//
// Per CTA (320 threads, 1 CTA per SM): warps 0-7 softmax (warps 0-3 take
// columns 0-63 of the step, warps 4-7 columns 64-127; thread = TMEM lane =
// tile row) and the epilogue, warp 8 TMA producer, warp 9 MMA issuer and TMEM
// owner.  Every mbarrier wait is bounded as in the forward kernel.
#include <cuda_bf16.h>

#include "clis_internal.h"
#include "sm103_ptx.cuh"

namespace clis {

__device__ unsigned int g_bwd_error_word = 0;

namespace {

constexpr int BM = 128;  // rows of a work tile (queries in dQ, keys in dK/dV)
constexpr int BN = 128;  // columns of a step (keys in dQ, queries in dK/dV)
constexpr int kThreads = 320;
constexpr int kSoftThreads = 256;

// Error-word bits (the forward's bits shifted up by 16).
constexpr unsigned kErrProducer = 1u << 16;
constexpr unsigned kErrMma = 1u << 17;
constexpr unsigned kErrSoftmax = 1u << 18;
constexpr unsigned kErrDrain = 1u << 20;
constexpr unsigned kErrLayout = 1u << 21;  // shared-memory allocation too small for the aligned layout

template <int D>
struct BCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int BOX_BYTES = 128 * 128;          // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;  // one 128-row tile of Q, K, V or dO
    // dK/dV: K and V resident; Q and dO stream through rings of their own.  Q_n
    // is read by S^T_n and, a step later, by dK_n, so it gets three slots (the
    // tile of step n+1 is loaded while steps n-1 and n still hold theirs); dO_n
    // is done after dV_n and gets two.  Shared memory: the tiles, then the
    // control block (barriers and two slots of -lse2 / -D), 231.6 KB at D = 128.
    static constexpr int QRING = (D == 128) ? 3 : 4;
    static constexpr int ORING = (D == 128) ? 2 : 3;
    static constexpr int LSLOT = 2;
    static constexpr int KV_TILES = (2 + QRING + ORING) * TILE_BYTES;
    // dQ: Q and dO resident; K and V tiles through two rings sized by how long
    // each lives.  K_j is read by S_j and again by dQ_j, issued in the next
    // step, so K_{j+1} takes the slot of K_{j-2} (KRING = 3, freed one and a half
    // steps before it is needed); V_j is read only by dP_j, so V_{j+1} takes the
    // slot of V_{j-1} (VRING = 2, freed two steps before).
    static constexpr int KRING = (D == 128) ? 3 : 4;
    static constexpr int VRING = (D == 128) ? 2 : 4;
    static constexpr int Q_SMEM = 2 * TILE_BYTES + (KRING + VRING) * TILE_BYTES + 1024;
    // TMEM columns (512 allocated).
    static constexpr uint32_t TM_ST = 0, TM_DPT = 128, TM_DV = 256, TM_DK = 256 + D;  // dK/dV kernel
    static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_DP = 256, TM_DQ = 384;       // dQ kernel
};

struct BParams {
    const float *lse2;  // [BH * Nq]
    const float *dvec;  // [BH * Nq] D_i
    uint16_t *dq, *dk, *dv;
    int64_t q_sb, q_sh, q_sn, k_sb, k_sh, k_sn, v_sb, v_sh, v_sn;
    int B, H, Nq, Nk;
    int nqb, nkb;    // 128-row query / key blocks per head
    // dK/dV kernel: query heads per key/value head.  1, or H when K and V are
    // broadcast over the heads (head stride 0: grouped-query attention folded
    // into the batch), in which case a work tile sums the gradients of every
    // query head of its batch entry.
    int kvg;
    int grp;         // causal: heads per scheduling group
    int num_tiles;
    float scale_log2;
    float scale;     // softmax scale = scale_log2 * ln 2
    int smem_bytes;  // dynamic shared memory of the launch
};

// Wait ignoring the abort flag (used only while draining after an abort).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 200000000ull) {
            atomicOr(&g_bwd_error_word, kErrDrain);
            return;
        }
    }
}

// Causal work tiles differ in cost, so heads are taken in groups of p.grp and,
// inside a group, blocks run heaviest first on even groups and lightest first
// on odd ones (static round-robin then balances the CTAs); the K/V or Q/dO of
// one group of heads stays in L2.  Non-causal: head-major.
struct KTile {
    int bh, b, h, kb, q0, nq;  // key block kb meets query blocks q0 .. q0 + nq - 1
    int hq0, nh;               // ... of query heads hq0 .. hq0 + nh - 1: steps nh * nq
};

// A dK/dV work tile is one key block of one key/value head (bh over the
// B * H / kvg key/value heads); its steps run over the query blocks of each of
// the head's kvg query heads in turn.  G: kernels built for grouped heads
// (kvg > 1); otherwise kvg is 1 at compile time.
template <bool CAUSAL, bool G>
__device__ __forceinline__ KTile decode_ktile(const BParams &p, int tile)
{
    KTile t;
    const int kvg = G ? p.kvg : 1;
    const int kv_heads = p.B * p.H / kvg;
    if (CAUSAL) {
        const int per_grp = p.grp * p.nkb;
        const int gi = tile / per_grp;
        const int r = tile % per_grp;
        const int heads = min(p.grp, kv_heads - gi * p.grp);
        const int ki = r / heads;
        t.bh = gi * p.grp + r % heads;
        t.kb = (gi & 1) ? (p.nkb - 1 - ki) : ki;  // key block kb costs nqb - kb steps per query head
        t.q0 = t.kb;                               // queries before the block see none of its keys
        t.nq = p.nqb - t.kb;
    } else {
        t.bh = tile / p.nkb;
        t.kb = tile % p.nkb;
        t.q0 = 0;
        t.nq = p.nqb;
    }
    const int hkv = p.H / kvg;  // key/value heads per batch entry
    t.b = t.bh / hkv;
    t.h = t.bh % hkv;           // key/value head coordinate (0 when broadcast)
    t.hq0 = t.h * kvg;
    t.nh = kvg;
    return t;
}

struct QTile {
    int bh, b, h, qb, nkv;  // query block qb meets key blocks 0 .. nkv - 1
};

template <bool CAUSAL>
__device__ __forceinline__ QTile decode_qtile(const BParams &p, int tile)
{
    QTile t;
    if (CAUSAL) {
        const int per_grp = p.grp * p.nqb;
        const int gi = tile / per_grp;
        const int r = tile % per_grp;
        const int heads = min(p.grp, p.B * p.H - gi * p.grp);
        const int qi = r / heads;
        t.bh = gi * p.grp + r % heads;
        t.qb = (gi & 1) ? qi : (p.nqb - 1 - qi);  // query block qb costs qb + 1 steps
        t.nkv = min(p.nkb, t.qb + 1);
    } else {
        t.bh = tile / p.nqb;
        t.qb = tile % p.nqb;
        t.nkv = p.nkb;
    }
    t.b = t.bh / p.H;
    t.h = t.bh % p.H;
    return t;
}

// ----------------------------------------------------------- MMA helpers
//
// Both run on one elected lane.  K-major operands step 16 elements (32 bytes)
// inside a 128-byte swizzle row, 4 steps per 64-column box; an MN-major B
// operand steps 16 rows (2048 bytes).  The start-address field of a
// descriptor is advanced by adding (byte offset >> 4); every shared address
// stays below 256 KB, so the field never carries.

// D[128 x 128] = A[128 x D] * B[128 x D]^T, both K-major (the scores).
template <int D, int DT>
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc)
{
    using C = BCfg<D>;
    constexpr uint32_t IDESC = idesc_f16kind_f32(BM, BN, false, DT ? 0u : 1u);
#pragma unroll
    for (int kk = 0; kk < D / 16; kk++) {
        const uint32_t off = ((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4;
        umma_ss(d_tmem, a_desc + off, b_desc + off, IDESC, kk > 0 ? 1u : 0u);
    }
}

// D[128 x D] (+)= A[128 x 128] * B[128 x D]: A packed in TMEM, B MN-major.
// The softmax warps store A in two halves: columns 0-63 of the step as 32
// packed columns at a_tmem, columns 64-127 at a_tmem + 64.
template <int D, int DT>
__device__ __forceinline__ void issue_accum(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate)
{
    constexpr uint32_t IDESC = idesc_f16kind_f32(BM, D, true, DT ? 0u : 1u);
#pragma unroll
    for (int kk = 0; kk < BN / 16; kk++)
        umma_ts(d_tmem, a_tmem + kk * 8 + (kk >= 4 ? 32 : 0), b_desc + ((kk * 2048) >> 4), IDESC,
                (accumulate | kk) ? 1u : 0u);
}

// One output row (bf16 or fp16) from D fp32 TMEM columns times `mul`.
template <int NCOL, int DT>
__device__ __forceinline__ void store_row(uint32_t t_src, float mul, uint16_t *dst, bool ok)
{
    const float2 m2 = make_float2(mul, mul);
#pragma unroll 1
    for (int c32 = 0; c32 < NCOL / 32; c32++) {
        uint32_t r[32];
        tmem_ld32(t_src + c32 * 32, r);
        tmem_wait_ld();
        if (ok) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; e++) {
                const float2 v = fmul2(make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), m2);
                pk[e] = pack2<DT>(v.x, v.y);
            }
            uint4 *o = reinterpret_cast<uint4 *>(dst + c32 * 32);
#pragma unroll
            for (int e = 0; e < 4; e++) o[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
    }
}

// =============================================================== dK / dV

template <int D>
struct __align__(16) KCtl {
    // Per slot, for the 128 query rows of a block: -lse2_i and -D_i (rows past
    // Nq: -inf and 0, so P = dS = 0 there).  Slot n % LSLOT serves step n.
    float nlse[BCfg<D>::LSLOT][BN], nd[BCfg<D>::LSLOT][BN];
    uint64_t kv_full, kv_empty;
    uint64_t q_full[BCfg<D>::QRING], q_empty[BCfg<D>::QRING];
    uint64_t o_empty[BCfg<D>::ORING];  // dO_n lands on Q_n's full barrier
    uint64_t ls_full[BCfg<D>::LSLOT], ls_empty[BCfg<D>::LSLOT];
    uint64_t s_full, dp_full, p_full, ds_full, acc_full, acc_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};


template <int D, bool CAUSAL, int DT, bool G>
__device__ void kv_producer(const BParams &p, KCtl<D> &c, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                            const CUtensorMap *tm_v, const CUtensorMap *tm_do, uint32_t sK, uint32_t sV,
                            uint32_t sQ, uint32_t sO, int lane)
{
    using C = BCfg<D>;
    volatile int *ab = &c.abort_flag;
    unsigned *err = &g_bwd_error_word;
    const bool leader = elect_one();
    const uint64_t pol_once = policy_evict_first();  // K, V: read by one work tile
    const uint64_t pol_keep = policy_evict_last();   // Q, dO: read by every key block of the head
    uint32_t nq = 0, no = 0;  // Q and dO tiles issued (one of each per step)
    int w = 0, kv_issued = -1;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++w) {
        const KTile T = decode_ktile<CAUSAL, G>(p, tile);
        if (!mbar_wait_warp(smem_u32(&c.kv_empty), (w & 1) ^ 1, ab, err, kErrProducer)) goto abort;
        if (leader) {
            const uint32_t bar = smem_u32(&c.kv_full);
            mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
#pragma unroll
            for (int bx = 0; bx < C::NBOX; bx++) {
                tma_load_4d_hint(sK + bx * C::BOX_BYTES, tm_k, bar, bx * 64, T.kb * BM, T.h, T.b, pol_once);
                tma_load_4d_hint(sV + bx * C::BOX_BYTES, tm_v, bar, bx * 64, T.kb * BM, T.h, T.b, pol_once);
            }
        }
        __syncwarp();
        kv_issued = w;
        // Steps: the query blocks of each query head of the tile in turn.
        for (int hg = T.hq0, qi = 0, i = 0; i < T.nh * T.nq; i++) {
            const uint32_t n = nq;  // global step index
            const int hq = G ? hg : T.h;
            const int qb = T.q0 + (G ? qi : i);
            // Q_n and dO_n are signalled together on Q_n's full barrier: the MMA warp
            // waits once per step (before S^T_n), and dO_n has landed for dP^T_n.
            const uint32_t qs = n % C::QRING;
            const uint32_t os = n % C::ORING;
            if (!mbar_wait_warp(smem_u32(&c.q_empty[qs]), ((n / C::QRING) & 1) ^ 1, ab, err, kErrProducer))
                goto abort;
            if (!mbar_wait_warp(smem_u32(&c.o_empty[os]), ((n / C::ORING) & 1) ^ 1, ab, err, kErrProducer))
                goto abort;
            if (leader) {
                const uint32_t bar = smem_u32(&c.q_full[qs]);
                mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
#pragma unroll
                for (int bx = 0; bx < C::NBOX; bx++) {
                    tma_load_4d_hint(sQ + qs * C::TILE_BYTES + bx * C::BOX_BYTES, tm_q, bar, bx * 64, qb * BN, hq,
                                     T.b, pol_keep);
                    tma_load_4d_hint(sO + os * C::TILE_BYTES + bx * C::BOX_BYTES, tm_do, bar, bx * 64, qb * BN, hq,
                                     T.b, pol_keep);
                }
            }
            __syncwarp();
            ++nq;
            ++no;
            // -lse2 and -D of the block, once the softmax warps have read the slot's
            // previous step (n - LSLOT).
            const uint32_t ls = n % C::LSLOT;
            if (!mbar_wait_warp(smem_u32(&c.ls_empty[ls]), ((n / C::LSLOT) & 1) ^ 1, ab, err, kErrProducer))
                goto abort;
            const int64_t rbase = (static_cast<int64_t>(T.b) * p.H + hq) * p.Nq;
#pragma unroll
            for (int r = lane; r < BN; r += 32) {
                const int row = qb * BN + r;
                const bool ok = row < p.Nq;
                c.nlse[ls][r] = ok ? -__ldg(p.lse2 + rbase + row) : -INFINITY;
                c.nd[ls][r] = ok ? -__ldg(p.dvec + rbase + row) : 0.f;
            }
            __syncwarp();
            if (leader) mbar_arrive(smem_u32(&c.ls_full[ls]));
            __syncwarp();
            if (++qi == T.nq) {
                qi = 0;
                ++hg;
            }
        }
    }
    return;
abort:
    for (uint32_t k = (nq > C::QRING ? nq - C::QRING : 0); k < nq; k++)
        drain_wait(smem_u32(&c.q_full[k % C::QRING]), (k / C::QRING) & 1);
    if (kv_issued >= 0) drain_wait(smem_u32(&c.kv_full), kv_issued & 1);
}

template <int D, bool CAUSAL, int DT, bool G>
__device__ void kv_mma(const BParams &p, KCtl<D> &c, uint32_t tmem, uint32_t sK, uint32_t sV, uint32_t sQ,
                       uint32_t sO)
{
    using C = BCfg<D>;
    volatile int *ab = &c.abort_flag;
    unsigned *err = &g_bwd_error_word;
    const bool leader = elect_one();
    const uint64_t kd = sdesc_sw128(sK, 16, 1024);
    const uint64_t vd = sdesc_sw128(sV, 16, 1024);
    const uint64_t qd_k = sdesc_sw128(sQ, 16, 1024);            // Q as K-major B
    const uint64_t qd_mn = sdesc_sw128(sQ, C::BOX_BYTES, 1024); // Q as MN-major B
    const uint64_t od_k = sdesc_sw128(sO, 16, 1024);            // dO as K-major B
    const uint64_t od_mn = sdesc_sw128(sO, C::BOX_BYTES, 1024);
    auto qoff = [](uint32_t m) -> uint64_t { return (static_cast<uint64_t>(m % C::QRING) * C::TILE_BYTES) >> 4; };
    auto ooff = [](uint32_t m) -> uint64_t { return (static_cast<uint64_t>(m % C::ORING) * C::TILE_BYTES) >> 4; };
    auto issue_s = [&](uint32_t m) {  // S^T_m = K Q_m^T
        issue_scores<D, DT>(tmem + C::TM_ST, kd, qd_k + qoff(m));
        umma_commit(smem_u32(&c.s_full));
    };
    auto issue_dp = [&](uint32_t m) {  // dP^T_m = V dO_m^T
        issue_scores<D, DT>(tmem + C::TM_DPT, vd, od_k + ooff(m));
        umma_commit(smem_u32(&c.dp_full));
    };
    uint32_t n = 0;
    int w = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++w) {
        const KTile T = decode_ktile<CAUSAL, G>(p, tile);
        if (!mbar_wait_warp(smem_u32(&c.kv_full), w & 1, ab, err, kErrMma)) goto abort;
        // First step of the tile: S^T and dP^T.
        if (!mbar_wait_warp(smem_u32(&c.q_full[n % C::QRING]), (n / C::QRING) & 1, ab, err, kErrMma)) goto abort;
        tc_fence_after();
        if (leader) issue_s(n);
        __syncwarp();
        if (leader) {
            issue_dp(n);  // dO_n landed with Q_n
            if (T.nh * T.nq == 1) umma_commit(smem_u32(&c.kv_empty));
        }
        __syncwarp();
        const int ns = T.nh * T.nq;  // steps of the tile
        for (int i = 0; i < ns; i++, n++) {
            const bool has_next = i + 1 < ns;
            const uint32_t nx = n + 1;
            // The previous tile's epilogue must have read dV and dK before they restart.
            if (i == 0 && w > 0)
                if (!mbar_wait_warp(smem_u32(&c.acc_free), (w - 1) & 1, ab, err, kErrMma)) goto abort;
            if (!mbar_wait_warp(smem_u32(&c.p_full), n & 1, ab, err, kErrMma)) goto abort;
            tc_fence_after();
            if (leader) {
                issue_accum<D, DT>(tmem + C::TM_DV, tmem + C::TM_ST, od_mn + ooff(n), i > 0 ? 1u : 0u);
                umma_commit(smem_u32(&c.o_empty[n % C::ORING]));  // dO_n is done
            }
            __syncwarp();
            // S^T of the next step goes in as soon as its Q tile is there: the S^T
            // columns hold P^T(n), which dV (issued just above) reads first, and the
            // softmax warps then overlap its exponentials with dK and the next dP^T.
            // If the tile has not landed yet (test_wait never blocks), dK goes first.
            bool s_next = false;
            if (has_next &&
                __all_sync(0xFFFFFFFFu, mbar_test_wait(smem_u32(&c.q_full[nx % C::QRING]), (nx / C::QRING) & 1))) {
                tc_fence_after();
                if (leader) issue_s(nx);
                __syncwarp();
                s_next = true;
            }
            if (!mbar_wait_warp(smem_u32(&c.ds_full), n & 1, ab, err, kErrMma)) goto abort;
            tc_fence_after();
            if (leader) {
                issue_accum<D, DT>(tmem + C::TM_DK, tmem + C::TM_DPT, qd_mn + qoff(n), i > 0 ? 1u : 0u);
                umma_commit(smem_u32(&c.q_empty[n % C::QRING]));  // Q_n is done
                if (!has_next) umma_commit(smem_u32(&c.acc_full));
            }
            __syncwarp();
            if (has_next) {
                if (!s_next) {
                    if (!mbar_wait_warp(smem_u32(&c.q_full[nx % C::QRING]), (nx / C::QRING) & 1, ab, err, kErrMma))
                        goto abort;
                    tc_fence_after();
                    if (leader) issue_s(nx);
                    __syncwarp();
                }
                // dP^T of the next step after dK, which read dS^T(n) from the same columns
                // (dO_{n+1} landed with Q_{n+1}).
                if (leader) {
                    issue_dp(nx);
                    if (i + 2 == ns) umma_commit(smem_u32(&c.kv_empty));
                }
                __syncwarp();
            }
        }
    }
    return;
abort:
    if (leader) umma_commit(smem_u32(&c.drain));
    __syncwarp();
    drain_wait(smem_u32(&c.drain), 0);
}

template <int D, bool CAUSAL, int DT, bool G>
__device__ void kv_softmax(const BParams &p, KCtl<D> &c, uint32_t tmem, int warp, int lane)
{
    using C = BCfg<D>;
    volatile int *ab = &c.abort_flag;
    unsigned *err = &g_bwd_error_word;
    const int half = warp >> 2;       // 0: query columns 0-63 of the step, 1: 64-127
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // key row within the tile = TMEM lane
    const int c0 = half * 64;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + C::TM_ST + lane_off + c0;
    const uint32_t tDP = tmem + C::TM_DPT + lane_off + c0;
    const float sl2 = p.scale_log2;
    const float2 sc2 = make_float2(sl2, sl2);
    uint32_t n = 0;
    int w = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++w) {
        const KTile T = decode_ktile<CAUSAL, G>(p, tile);
        for (int i = 0, qi = 0; i < T.nh * T.nq; i++, n++, qi = (qi + 1 == T.nq) ? 0 : qi + 1) {
            const uint32_t s = n % C::LSLOT;
            // The diagonal block: query column c sees this key only if c >= rl.
            const bool diag = CAUSAL && (T.q0 + (G ? qi : i) == T.kb);
            if (!mbar_wait(smem_u32(&c.s_full), n & 1, ab, err, kErrSoftmax)) return;
            // -lse2 and -D of this step's query block, staged by the producer warp.
            if (!mbar_wait(smem_u32(&c.ls_full[s]), (n / C::LSLOT) & 1, ab, err, kErrSoftmax)) return;
            tc_fence_after();
            uint32_t r[64];
            tmem_ld32(tS, r);
            tmem_ld32(tS + 32, r + 32);
            tmem_wait_ld();
            // P^T = exp2(scale_log2 * s - lse2_i), packed in place over the first
            // 32 of this half's 64 score columns.
            float pr[64];
            uint32_t pk[32];
            const float4 *nl4 = reinterpret_cast<const float4 *>(&c.nlse[s][c0]);
#pragma unroll
            for (int e4 = 0; e4 < 16; e4++) {
                const float4 nl = nl4[e4];
#pragma unroll
                for (int h2 = 0; h2 < 2; h2++) {
                    const int e = 4 * e4 + 2 * h2;
                    float2 x = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sc2,
                                     h2 ? make_float2(nl.z, nl.w) : make_float2(nl.x, nl.y));
                    if (diag) {
                        if (c0 + e < rl) x.x = -INFINITY;
                        if (c0 + e + 1 < rl) x.y = -INFINITY;
                    }
                    pr[e] = ex2_approx(x.x);
                    pr[e + 1] = ex2_approx(x.y);
                    pk[e >> 1] = pack2<DT>(pr[e], pr[e + 1]);
                }
            }
            tmem_st16(tS, pk);
            tmem_st16(tS + 16, pk + 16);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&c.p_full));

            // dS^T = P^T (dP^T - D_i), packed over the first 32 dP^T columns of this half.
            if (!mbar_wait(smem_u32(&c.dp_full), n & 1, ab, err, kErrSoftmax)) return;
            tc_fence_after();
            tmem_ld32(tDP, r);
            tmem_ld32(tDP + 32, r + 32);
            tmem_wait_ld();
            const float4 *nd4 = reinterpret_cast<const float4 *>(&c.nd[s][c0]);
#pragma unroll
            for (int e4 = 0; e4 < 16; e4++) {
                const float4 nd = nd4[e4];
#pragma unroll
                for (int h2 = 0; h2 < 2; h2++) {
                    const int e = 4 * e4 + 2 * h2;
                    const float2 t = fadd2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                           h2 ? make_float2(nd.z, nd.w) : make_float2(nd.x, nd.y));
                    const float2 ds = fmul2(t, make_float2(pr[e], pr[e + 1]));
                    pk[e >> 1] = pack2<DT>(ds.x, ds.y);
                }
            }
            mbar_arrive(smem_u32(&c.ls_empty[s]));  // the slot's -lse2 and -D are read
            tmem_st16(tDP, pk);
            tmem_st16(tDP + 16, pk + 16);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&c.ds_full));
        }
        // Epilogue: warps 0-3 write dV, warps 4-7 dK (times the softmax scale).
        if (!mbar_wait(smem_u32(&c.acc_full), w & 1, ab, err, kErrSoftmax)) return;
        tc_fence_after();
        const int key = T.kb * BM + rl;
        const bool ok = key < p.Nk;
        if (half == 0)
            store_row<D, DT>(tmem + C::TM_DV + lane_off, 1.f, p.dv + T.b * p.v_sb + T.h * p.v_sh +
                             static_cast<int64_t>(ok ? key : 0) * p.v_sn, ok);
        else
            store_row<D, DT>(tmem + C::TM_DK + lane_off, p.scale, p.dk + T.b * p.k_sb + T.h * p.k_sh +
                             static_cast<int64_t>(ok ? key : 0) * p.k_sn, ok);
        tc_fence_before();
        mbar_arrive(smem_u32(&c.acc_free));
    }
}

template <int D, bool CAUSAL, int DT, bool G>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BParams p)
{
    using C = BCfg<D>;
    // Dynamic shared memory: [K][V][Q x QRING][dO x ORING] from the first
    // 1024-byte boundary (128-byte swizzle atoms), then the control block.
    extern __shared__ __align__(1024) uint8_t dsmem[];
    const uint32_t dbase = smem_u32(dsmem);
    const uint32_t sbase = (dbase + 1023u) & ~1023u;
    const uint32_t ctl_off = sbase - dbase + C::KV_TILES;
    if (ctl_off + sizeof(KCtl<D>) > static_cast<uint32_t>(p.smem_bytes)) {
        // The allocation cannot hold the aligned layout: report, touch nothing.
        if (threadIdx.x == 0) atomicOr(&g_bwd_error_word, kErrLayout);
        return;
    }
    KCtl<D> &ctl = *reinterpret_cast<KCtl<D> *>(dsmem + ctl_off);
    const uint32_t sK = sbase, sV = sbase + C::TILE_BYTES, sQ = sbase + 2 * C::TILE_BYTES;
    const uint32_t sO = sQ + C::QRING * C::TILE_BYTES;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl.kv_full), 1);
        mbar_init(smem_u32(&ctl.kv_empty), 1);
        for (int s = 0; s < C::QRING; s++) {
            mbar_init(smem_u32(&ctl.q_full[s]), 1);
            mbar_init(smem_u32(&ctl.q_empty[s]), 1);
        }
        for (int s = 0; s < C::ORING; s++) mbar_init(smem_u32(&ctl.o_empty[s]), 1);
        for (int s = 0; s < C::LSLOT; s++) {
            mbar_init(smem_u32(&ctl.ls_full[s]), 1);
            mbar_init(smem_u32(&ctl.ls_empty[s]), kSoftThreads);
        }
        mbar_init(smem_u32(&ctl.s_full), 1);
        mbar_init(smem_u32(&ctl.dp_full), 1);
        mbar_init(smem_u32(&ctl.p_full), kSoftThreads);
        mbar_init(smem_u32(&ctl.ds_full), kSoftThreads);
        mbar_init(smem_u32(&ctl.acc_full), 1);
        mbar_init(smem_u32(&ctl.acc_free), kSoftThreads);
        mbar_init(smem_u32(&ctl.drain), 1);
        ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(&ctl.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    if (warp < 8)
        kv_softmax<D, CAUSAL, DT, G>(p, ctl, tmem, warp, lane);
    else if (warp == 8)
        kv_producer<D, CAUSAL, DT, G>(p, ctl, &tm_q, &tm_k, &tm_v, &tm_do, sK, sV, sQ, sO, lane);
    else
        kv_mma<D, CAUSAL, DT, G>(p, ctl, tmem, sK, sV, sQ, sO);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ==================================================================== dQ

template <int D>
struct __align__(16) QCtl {
    uint64_t qo_full, qo_empty;
    uint64_t k_full[BCfg<D>::KRING], k_empty[BCfg<D>::KRING];
    uint64_t v_empty[BCfg<D>::VRING];  // V_j lands on K_j's full barrier
    uint64_t s_full[2], dp_full, ds_full, acc_full, acc_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D, bool CAUSAL, int DT>
__device__ void q_producer(const BParams &p, QCtl<D> &c, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                           const CUtensorMap *tm_v, const CUtensorMap *tm_do, uint32_t sQ, uint32_t sDO, uint32_t sK,
                           uint32_t sV)
{
    using C = BCfg<D>;
    volatile int *ab = &c.abort_flag;
    unsigned *err = &g_bwd_error_word;
    const bool leader = elect_one();
    const uint64_t pol_keep = policy_evict_last();   // K, V: read by every query block of the head
    const uint64_t pol_once = policy_evict_first();  // Q, dO: read by one work tile
    uint32_t nk = 0, nv = 0;  // K and V tiles issued (one of each per step)
    int w = 0, q_issued = -1;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++w) {
        const QTile T = decode_qtile<CAUSAL>(p, tile);
        if (!mbar_wait_warp(smem_u32(&c.qo_empty), (w & 1) ^ 1, ab, err, kErrProducer)) goto abort;
        if (leader) {
            const uint32_t bar = smem_u32(&c.qo_full);
            mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
#pragma unroll
            for (int bx = 0; bx < C::NBOX; bx++) {
                tma_load_4d_hint(sQ + bx * C::BOX_BYTES, tm_q, bar, bx * 64, T.qb * BM, T.h, T.b, pol_once);
                tma_load_4d_hint(sDO + bx * C::BOX_BYTES, tm_do, bar, bx * 64, T.qb * BM, T.h, T.b, pol_once);
            }
        }
        __syncwarp();
        q_issued = w;
        // K_j and V_j are signalled together on K_j's full barrier: the MMA warp waits
        // once per step (before S_j), and V_j has landed by the time dP_j needs it.
        for (int j = 0; j < T.nkv; j++) {
            const uint32_t ks = nk % C::KRING;
            const uint32_t vs = nv % C::VRING;
            if (!mbar_wait_warp(smem_u32(&c.k_empty[ks]), ((nk / C::KRING) & 1) ^ 1, ab, err, kErrProducer))
                goto abort;
            if (!mbar_wait_warp(smem_u32(&c.v_empty[vs]), ((nv / C::VRING) & 1) ^ 1, ab, err, kErrProducer))
                goto abort;
            if (leader) {
                const uint32_t bar = smem_u32(&c.k_full[ks]);
                mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES);
#pragma unroll
                for (int bx = 0; bx < C::NBOX; bx++) {
                    tma_load_4d_hint(sK + ks * C::TILE_BYTES + bx * C::BOX_BYTES, tm_k, bar, bx * 64, j * BN, T.h,
                                     T.b, pol_keep);
                    tma_load_4d_hint(sV + vs * C::TILE_BYTES + bx * C::BOX_BYTES, tm_v, bar, bx * 64, j * BN, T.h,
                                     T.b, pol_keep);
                }
            }
            __syncwarp();
            ++nk;
            ++nv;
        }
    }
    return;
abort:
    // Let every copy already issued land before the CTA leaves.
    for (uint32_t k = (nk > C::KRING ? nk - C::KRING : 0); k < nk; k++)
        drain_wait(smem_u32(&c.k_full[k % C::KRING]), (k / C::KRING) & 1);
    if (q_issued >= 0) drain_wait(smem_u32(&c.qo_full), q_issued & 1);
}

template <int D, bool CAUSAL, int DT>
__device__ void q_mma(const BParams &p, QCtl<D> &c, uint32_t tmem, uint32_t sQ, uint32_t sDO, uint32_t sK,
                      uint32_t sV)
{
    using C = BCfg<D>;
    volatile int *ab = &c.abort_flag;
    unsigned *err = &g_bwd_error_word;
    const bool leader = elect_one();
    const uint64_t qd = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dod = sdesc_sw128(sDO, 16, 1024);
    const uint64_t kd_k = sdesc_sw128(sK, 16, 1024);             // K slot as K-major B (S = Q K^T)
    const uint64_t kd_mn = sdesc_sw128(sK, C::BOX_BYTES, 1024);  // K slot as MN-major B (dQ += dS K)
    const uint64_t vd_k = sdesc_sw128(sV, 16, 1024);             // V slot as K-major B (dP = dO V^T)
    auto slot_off = [](uint32_t s) -> uint64_t { return (static_cast<uint64_t>(s) * C::TILE_BYTES) >> 4; };
    uint32_t n = 0;  // global step index; K_n and V_n are the rings' n-th tiles
    int w = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++w) {
        const QTile T = decode_qtile<CAUSAL>(p, tile);
        if (!mbar_wait_warp(smem_u32(&c.qo_full), w & 1, ab, err, kErrMma)) goto abort;
        for (int j = 0; j < T.nkv; j++, n++) {
            // S_j = Q K_j^T into S[n & 1].
            const uint32_t ks = n % C::KRING;
            if (!mbar_wait_warp(smem_u32(&c.k_full[ks]), (n / C::KRING) & 1, ab, err, kErrMma)) goto abort;
            tc_fence_after();
            if (leader) {
                issue_scores<D, DT>(tmem + ((n & 1) ? C::TM_S1 : C::TM_S0), qd, kd_k + slot_off(ks));
                umma_commit(smem_u32(&c.s_full[n & 1]));
            }
            __syncwarp();
            // dQ += dS_{j-1} K_{j-1} once the softmax warps stored dS_{j-1}.
            if (j > 0) {
                if (j == 1 && w > 0)
                    if (!mbar_wait_warp(smem_u32(&c.acc_free), (w - 1) & 1, ab, err, kErrMma)) goto abort;
                if (!mbar_wait_warp(smem_u32(&c.ds_full), (n - 1) & 1, ab, err, kErrMma)) goto abort;
                tc_fence_after();
                if (leader) {
                    issue_accum<D, DT>(tmem + C::TM_DQ, tmem + C::TM_DP, kd_mn + slot_off((n - 1) % C::KRING),
                                       j > 1 ? 1u : 0u);
                    umma_commit(smem_u32(&c.k_empty[(n - 1) % C::KRING]));
                }
                __syncwarp();
            }
            // dP_j = dO V_j^T (after dQ has read dS_{j-1} from the same columns); V_j
            // landed with K_j.
            const uint32_t vs = n % C::VRING;
            if (leader) {
                issue_scores<D, DT>(tmem + C::TM_DP, dod, vd_k + slot_off(vs));
                umma_commit(smem_u32(&c.dp_full));
                umma_commit(smem_u32(&c.v_empty[vs]));
                if (j == T.nkv - 1) umma_commit(smem_u32(&c.qo_empty));
            }
            __syncwarp();
        }
        if (T.nkv == 1 && w > 0)
            if (!mbar_wait_warp(smem_u32(&c.acc_free), (w - 1) & 1, ab, err, kErrMma)) goto abort;
        if (!mbar_wait_warp(smem_u32(&c.ds_full), (n - 1) & 1, ab, err, kErrMma)) goto abort;
        tc_fence_after();
        if (leader) {
            issue_accum<D, DT>(tmem + C::TM_DQ, tmem + C::TM_DP, kd_mn + slot_off((n - 1) % C::KRING),
                               T.nkv > 1 ? 1u : 0u);
            umma_commit(smem_u32(&c.k_empty[(n - 1) % C::KRING]));
            umma_commit(smem_u32(&c.acc_full));
        }
        __syncwarp();
    }
    return;
abort:
    if (leader) umma_commit(smem_u32(&c.drain));
    __syncwarp();
    drain_wait(smem_u32(&c.drain), 0);
}

template <int D, bool CAUSAL, int DT>
__device__ void q_softmax(const BParams &p, QCtl<D> &c, uint32_t tmem, int warp, int lane)
{
    using C = BCfg<D>;
    volatile int *ab = &c.abort_flag;
    unsigned *err = &g_bwd_error_word;
    const int half = warp >> 2;  // 0: key columns 0-63 of the step, 1: 64-127
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // query row within the tile = TMEM lane
    const int c0 = half * 64;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tDP = tmem + C::TM_DP + lane_off + c0;
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
    uint32_t n = 0;
    int w = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++w) {
        const QTile T = decode_qtile<CAUSAL>(p, tile);
        const int row = T.qb * BM + rl;
        const bool row_ok = row < p.Nq;
        const int64_t ridx = static_cast<int64_t>(T.bh) * p.Nq + row;
        // Rows past Nq: -lse2 = -inf gives P = 0.
        const float nl = row_ok ? -__ldg(p.lse2 + ridx) : -INFINITY;
        const float ndi = row_ok ? -__ldg(p.dvec + ridx) : 0.f;
        const float2 nl2 = make_float2(nl, nl), nd2 = make_float2(ndi, ndi);
        // Keys [0, lim) are visible to this row.
        const int lim = CAUSAL ? min(p.Nk, row + 1) : p.Nk;
        for (int j = 0; j < T.nkv; j++, n++) {
            const uint32_t tS = tmem + ((n & 1) ? C::TM_S1 : C::TM_S0) + lane_off + c0;
            if (!mbar_wait(smem_u32(&c.s_full[n & 1]), (n >> 1) & 1, ab, err, kErrSoftmax)) return;
            tc_fence_after();
            uint32_t r[64];
            tmem_ld32(tS, r);
            tmem_ld32(tS + 32, r + 32);
            tmem_wait_ld();
            const int key0 = j * BN + c0;
            const bool mask = key0 + 64 > lim;
            float pr[64];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                float2 x = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sc2, nl2);
                if (mask) {
                    if (key0 + e >= lim) x.x = -INFINITY;
                    if (key0 + e + 1 >= lim) x.y = -INFINITY;
                }
                pr[e] = ex2_approx(x.x);
                pr[e + 1] = ex2_approx(x.y);
            }
            if (!mbar_wait(smem_u32(&c.dp_full), n & 1, ab, err, kErrSoftmax)) return;
            tc_fence_after();
            tmem_ld32(tDP, r);
            tmem_ld32(tDP + 32, r + 32);
            tmem_wait_ld();
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 64; e += 2) {
                const float2 t = fadd2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), nd2);
                const float2 ds = fmul2(t, make_float2(pr[e], pr[e + 1]));
                pk[e >> 1] = pack2<DT>(ds.x, ds.y);
            }
            tmem_st16(tDP, pk);
            tmem_st16(tDP + 16, pk + 16);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&c.ds_full));
        }
        // Epilogue: each half writes D/2 columns of dQ (times the softmax scale).
        if (!mbar_wait(smem_u32(&c.acc_full), w & 1, ab, err, kErrSoftmax)) return;
        tc_fence_after();
        store_row<D / 2, DT>(tmem + C::TM_DQ + lane_off + half * (D / 2), p.scale,
                             p.dq + T.b * p.q_sb + T.h * p.q_sh + static_cast<int64_t>(row_ok ? row : 0) * p.q_sn +
                                 half * (D / 2),
                             row_ok);
        tc_fence_before();
        mbar_arrive(smem_u32(&c.acc_free));
    }
}

template <int D, bool CAUSAL, int DT>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BParams p)
{
    using C = BCfg<D>;
    extern __shared__ uint8_t dsmem[];
    __shared__ QCtl<D> ctl;
    const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
    const uint32_t sQ = sbase, sDO = sbase + C::TILE_BYTES, sK = sbase + 2 * C::TILE_BYTES;
    const uint32_t sV = sK + C::KRING * C::TILE_BYTES;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&ctl.qo_full), 1);
        mbar_init(smem_u32(&ctl.qo_empty), 1);
        for (int s = 0; s < C::KRING; s++) {
            mbar_init(smem_u32(&ctl.k_full[s]), 1);
            mbar_init(smem_u32(&ctl.k_empty[s]), 1);
        }
        for (int s = 0; s < C::VRING; s++) mbar_init(smem_u32(&ctl.v_empty[s]), 1);
        mbar_init(smem_u32(&ctl.s_full[0]), 1);
        mbar_init(smem_u32(&ctl.s_full[1]), 1);
        mbar_init(smem_u32(&ctl.dp_full), 1);
        mbar_init(smem_u32(&ctl.ds_full), kSoftThreads);
        mbar_init(smem_u32(&ctl.acc_full), 1);
        mbar_init(smem_u32(&ctl.acc_free), kSoftThreads);
        mbar_init(smem_u32(&ctl.drain), 1);
        ctl.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(&ctl.tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    if (warp < 8)
        q_softmax<D, CAUSAL, DT>(p, ctl, tmem, warp, lane);
    else if (warp == 8)
        q_producer<D, CAUSAL, DT>(p, ctl, &tm_q, &tm_k, &tm_v, &tm_do, sQ, sDO, sK, sV);
    else
        q_mma<D, CAUSAL, DT>(p, ctl, tmem, sQ, sDO, sK, sV);
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================= small kernels

// D_i = dO_i . O_i in fp32; d/8 threads per row, 8 elements (16 bytes) each,
// reduced by a fixed butterfly (deterministic).
template <int DT>
__global__ void bwd_dot_kernel(const uint16_t *o, const uint16_t *dout, int64_t sb, int64_t sh, int64_t sn, int H,
                               int Nq, int d, int64_t nrows, float *dvec)
{
    const int tpr = d / 8;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t rg = idx / tpr;
    const int part = static_cast<int>(idx % tpr);
    float acc = 0.f;
    if (rg < nrows) {
        const int64_t bh = rg / Nq;
        const int64_t i = rg % Nq;
        const int64_t off = (bh / H) * sb + (bh % H) * sh + i * sn + part * 8;
        const uint4 a = *reinterpret_cast<const uint4 *>(o + off);
        const uint4 g = *reinterpret_cast<const uint4 *>(dout + off);
        acc = elem_lo<DT>(a.x) * elem_lo<DT>(g.x);
        acc = fmaf(elem_hi<DT>(a.x), elem_hi<DT>(g.x), acc);
        acc = fmaf(elem_lo<DT>(a.y), elem_lo<DT>(g.y), acc);
        acc = fmaf(elem_hi<DT>(a.y), elem_hi<DT>(g.y), acc);
        acc = fmaf(elem_lo<DT>(a.z), elem_lo<DT>(g.z), acc);
        acc = fmaf(elem_hi<DT>(a.z), elem_hi<DT>(g.z), acc);
        acc = fmaf(elem_lo<DT>(a.w), elem_lo<DT>(g.w), acc);
        acc = fmaf(elem_hi<DT>(a.w), elem_hi<DT>(g.w), acc);
    }
    for (int m = tpr / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
    if (rg < nrows && part == 0) dvec[rg] = acc;
}

// Zero-fill of a strided [B, H, N, d] tensor (gradients with no contribution).
__global__ void bwd_zero_kernel(uint16_t *x, int64_t sb, int64_t sh, int64_t sn, int H, int N, int d, int64_t n8)
{
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= n8) return;
    const int per_row = d / 8;
    const int64_t rg = idx / per_row;
    const int c8 = static_cast<int>(idx % per_row);
    const int64_t bh = rg / N, i = rg % N;
    *reinterpret_cast<uint4 *>(x + (bh / H) * sb + (bh % H) * sh + i * sn + c8 * 8) = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 4-D map over [B, H, N, d] (innermost first), 64 x 128 boxes, 128-byte swizzle.
bool tile_map(CUtensorMap *map, const void *base, int dtype, int64_t B, int64_t H, int64_t N, int64_t d, int64_t sb,
              int64_t sh, int64_t sn)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    if (H == 1) sh = sn * N;  // the stride of a size-1 dimension is never used
    if (B == 1) sb = sh * H;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(sn * 2), static_cast<cuuint64_t>(sh * 2),
                             static_cast<cuuint64_t>(sb * 2)};
    cuuint32_t box[4] = {64, 128, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, dtype == CLIS_DT_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

clis_status_t zero_fill(uint16_t *x, int64_t sb, int64_t sh, int64_t sn, int B, int H, int N, int d,
                        cudaStream_t stream)
{
    const int64_t n8 = static_cast<int64_t>(B) * H * N * (d / 8);
    if (n8 == 0) return CLIS_OK;
    bwd_zero_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(x, sb, sh, sn, H, N, d, n8);
    return cudaGetLastError() == cudaSuccess ? CLIS_OK : CLIS_ERR_CUDA;
}

template <int D, bool CAUSAL, int DT>
clis_status_t launch_impl(const AttnBwdArgs &a, cudaStream_t stream)
{
    using C = BCfg<D>;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CLIS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CLIS_ERR_CUDA;
    // dK/dV: tiles + control block + alignment slack, capped at the device's
    // per-block maximum (the kernel checks that its aligned layout fits).
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return CLIS_ERR_CUDA;
    const int kv_need = C::KV_TILES + static_cast<int>(sizeof(KCtl<D>));
    if (kv_need > optin) return CLIS_ERR_UNSUPPORTED;
    const int kv_smem = kv_need + 1023 < optin ? kv_need + 1023 : optin;
    // K and V broadcast over the heads (head stride 0): one key/value head per
    // batch entry, shared by all H query heads (grouped-query attention folded
    // into the batch); the dK/dV kernel built for it sums each group.
    const bool grouped = a.H > 1 && a.k_sh == 0 && a.v_sh == 0;
    if (cudaFuncSetAttribute(grouped ? bwd_dkdv_kernel<D, CAUSAL, DT, true> : bwd_dkdv_kernel<D, CAUSAL, DT, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kv_smem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dq_kernel<D, CAUSAL, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::Q_SMEM) != cudaSuccess)
        return CLIS_ERR_CUDA;

    // D_i = dO_i . O_i
    const int64_t nrows = static_cast<int64_t>(a.B) * a.H * a.Nq;
    {
        const int64_t nthr = nrows * (D / 8);
        bwd_dot_kernel<DT><<<static_cast<unsigned>((nthr + 255) / 256), 256, 0, stream>>>(
            a.o, a.dout, a.o_sb, a.o_sh, a.o_sn, a.H, a.Nq, D, nrows, a.dvec);
        if (cudaGetLastError() != cudaSuccess) return CLIS_ERR_CUDA;
    }

    CUtensorMap mq, mk, mv, mdo;
    if (!tile_map(&mq, a.q, DT, a.B, a.H, a.Nq, D, a.q_sb, a.q_sh, a.q_sn) ||
        !tile_map(&mk, a.k, DT, a.B, a.H, a.Nk, D, a.k_sb, a.k_sh, a.k_sn) ||
        !tile_map(&mv, a.v, DT, a.B, a.H, a.Nk, D, a.v_sb, a.v_sh, a.v_sn) ||
        !tile_map(&mdo, a.dout, DT, a.B, a.H, a.Nq, D, a.o_sb, a.o_sh, a.o_sn))
        return CLIS_ERR_CUDA;

    BParams p;
    p.lse2 = a.lse2;
    p.dvec = a.dvec;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.q_sb = a.q_sb;
    p.q_sh = a.q_sh;
    p.q_sn = a.q_sn;
    p.k_sb = a.k_sb;
    p.k_sh = a.k_sh;
    p.k_sn = a.k_sn;
    p.v_sb = a.v_sb;
    p.v_sh = a.v_sh;
    p.v_sn = a.v_sn;
    p.B = a.B;
    p.H = a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.nqb = (a.Nq + BM - 1) / BM;
    p.nkb = (a.Nk + BN - 1) / BN;
    p.scale_log2 = a.scale_log2;
    p.scale = a.scale_log2 * 0.693147180559945309f;
    const int BH = a.B * a.H;
    p.kvg = grouped ? a.H : 1;
    const int KVH = BH / p.kvg;

    // dK, dV: one work tile per (key/value head, key block).
    p.num_tiles = KVH * p.nkb;
    p.grp = (2 * nsm + p.nkb - 1) / p.nkb;
    p.grp = p.grp > KVH ? KVH : (p.grp < 1 ? 1 : p.grp);
    int grid = p.num_tiles < nsm ? p.num_tiles : nsm;
    p.smem_bytes = kv_smem;
    if (grouped)
        bwd_dkdv_kernel<D, CAUSAL, DT, true><<<grid, kThreads, kv_smem, stream>>>(mq, mk, mv, mdo, p);
    else
        bwd_dkdv_kernel<D, CAUSAL, DT, false><<<grid, kThreads, kv_smem, stream>>>(mq, mk, mv, mdo, p);
    if (cudaGetLastError() != cudaSuccess) return CLIS_ERR_CUDA;

    // dQ: one work tile per (head, query block).
    p.num_tiles = BH * p.nqb;
    p.grp = (2 * nsm + p.nqb - 1) / p.nqb;
    p.grp = p.grp > BH ? BH : (p.grp < 1 ? 1 : p.grp);
    grid = p.num_tiles < nsm ? p.num_tiles : nsm;
    bwd_dq_kernel<D, CAUSAL, DT><<<grid, kThreads, C::Q_SMEM, stream>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError() == cudaSuccess ? CLIS_OK : CLIS_ERR_CUDA;
}

template <int D, int DT>
clis_status_t launch_causal(const AttnBwdArgs &a, cudaStream_t s)
{
    return a.causal ? launch_impl<D, true, DT>(a, s) : launch_impl<D, false, DT>(a, s);
}

}  // namespace

clis_status_t launch_attn_bwd(const AttnBwdArgs &a, cudaStream_t stream)
{
    if (a.B * a.H == 0) return CLIS_OK;
    if (a.Nq == 0)  // no query sees any key: dK = dV = 0
        return zero_fill(a.dk, a.k_sb, a.k_sh, a.k_sn, a.B, a.H, a.Nk, a.d, stream) == CLIS_OK
                   ? zero_fill(a.dv, a.v_sb, a.v_sh, a.v_sn, a.B, a.H, a.Nk, a.d, stream)
                   : CLIS_ERR_CUDA;
    const bool fp16 = a.dtype == CLIS_DT_FP16;
    if (a.d == 128) return fp16 ? launch_causal<128, 1>(a, stream) : launch_causal<128, 0>(a, stream);
    return fp16 ? launch_causal<64, 1>(a, stream) : launch_causal<64, 0>(a, stream);
}

clis_status_t read_bwd_error(uint32_t *code)
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_bwd_error_word, sizeof v) != cudaSuccess) return CLIS_ERR_CUDA;
    *code = v;
    return CLIS_OK;
}

clis_status_t clear_bwd_error()
{
    const unsigned int z = 0;
    return cudaMemcpyToSymbol(g_bwd_error_word, &z, sizeof z) == cudaSuccess ? CLIS_OK : CLIS_ERR_CUDA;
}

}  // namespace clis
