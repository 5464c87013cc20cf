/*
 * clis_oracle.c -- CPU reference ("oracle") for CLiS attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA implementation; it is written from the paper "CLiS: Plug-and-Play
 * Attention Acceleration for Video Diffusion on TPUs via Certified
 * Stabilization" (Tsai et al., 2026), Algorithm 1, and from the plain
 * definition of softmax attention.
 *
 * Precision: everything is fp64.  Inputs are bf16 or IEEE binary16 (fp16) bit
 * patterns (uint16) or, for the identity tests, fp64 arrays.  Layout is
 * contiguous [BH][N][d].
 *
 * Two routines:
 *
 *  oracle_certify   Algorithm 1, steps 1-7, for every head, followed by the
 *                   certification decision.  The pages lose the text after
 *                   step 7; the decision used here is "all inputs finite and
 *                   B_h <= C" (readings listed below).
 *
 *  oracle_certify_prefix_tiles  per-prefix certificates of causal heads, one
 *                   per block of query rows (a finer reading; see there).
 *
 *  oracle_attn_*    O_i = sum_j softmax_j(scale * q_i . k_j) v_j, two passes
 *                   per row (max, then exp/sum/PV), optional causal mask
 *                   (key j visible to query i iff j <= i).  Since a stabiliser
 *                   cancels between numerator and denominator, this plain
 *                   definition is the exact result CLiS must reproduce.
 *
 *  oracle_attn_bwd_*  gradients dQ, dK, dV of L = sum_i dO_i . O_i for the
 *                   same attention (the backward pass of causal training,
 *                   Table 3's setting).  The pages give no backward
 *                   algorithm; this is the plain chain rule through softmax.
 *
 * Readings of the pages (where they are silent or garbled):
 *  - kappa (Alg. 1 step 3 asks only for an upper bound of the largest centred
 *    key norm, without saying how tight): the oracle computes the exact fp64
 *    maximum of the centred key norms.
 *  - BoundUp (Alg. 1 step 4, never defined): Cauchy-Schwarz,
 *    BoundUp(q, kappa) = scale_log2 * ||q||_2 * kappa, so B_h is a bound on
 *    |scale_log2 * q_r . (k_j - kbar)| in exp2-argument units.
 *  - "||V_jr||" in step 5: entry-wise absolute value.
 *  - U_exp, U_acc (Figure 3's table is lost): log2 of the largest finite
 *    value of the format holding exp2 outputs / the accumulator,
 *    (2 - 2^(1-p)) * 2^emax for a format with p significand bits.
 *  - Decision: certified <=> all of Q, K, V finite and B_h <= C.
 *  - Non-finite heads report G = A = C = 0 and B_h = +inf (reason 2).
 *
 * Parity pins: every routine here is checked by tests/test_oracle_pins.py
 * against brute force, closed forms, identities and hand-built heads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Format codes of this file (the Python wrapper maps names onto them). */
enum { ORC_FMT_FP16 = 0, ORC_FMT_BF16 = 1, ORC_FMT_FP32 = 2, ORC_FMT_E4M3 = 3 };

typedef struct {
    int32_t certified; /* 1 = fixed-stabiliser path is safe for this head     */
    int32_t G;         /* Alg. 1 step 5                                        */
    int32_t A;         /* Alg. 1 step 6                                        */
    int32_t C;         /* Alg. 1 step 7                                        */
    int32_t reason;    /* 0 certified, 1 B_h > C, 2 non-finite input           */
    int32_t band;      /* 1 if B_h*(1 -/+ 2^-12) falls on both sides of C      */
    double B_h;        /* Alg. 1 step 4                                        */
    double kappa;      /* Alg. 1 step 3 (exact max centred key norm)           */
    double qmax;       /* max_r ||q_r||_2                                      */
    double vmax;       /* max_{j,r} |V_jr|                                     */
} oracle_cert_t;

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double fp16_bits_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 10) & 0x1F;
    int f = b & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)f, -24);                  /* zero and subnormals: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* Input element formats of this file. */
enum { ORC_IN_BF16 = 0, ORC_IN_FP16 = 1 };

static double bits_to_double(uint16_t b, int in_fmt)
{
    return in_fmt == ORC_IN_FP16 ? fp16_bits_to_double(b) : bf16_bits_to_double(b);
}

double oracle_decode(uint16_t bits, int in_fmt) { return bits_to_double(bits, in_fmt); }

/* Largest finite value of a binary floating-point format with p significand
 * bits (implicit bit included) and maximum exponent emax: (2 - 2^(1-p)) 2^emax.
 * E4M3 (the 8-bit format one step below Figure 3's FP16, as the OCP 8-bit
 * floating-point definition fixes it: 4 exponent bits with bias 7, 3 fraction
 * bits, no infinities) keeps its all-ones pattern for NaN, so its largest
 * finite significand is 1.110b = 1.75 and its maximum 1.75 * 2^8 = 448. */
static double format_max_finite(int fmt)
{
    int p, emax;
    switch (fmt) {
    case ORC_FMT_FP16: p = 11; emax = 15; break;
    case ORC_FMT_BF16: p = 8; emax = 127; break;
    case ORC_FMT_FP32: p = 24; emax = 127; break;
    case ORC_FMT_E4M3: return (2.0 - ldexp(1.0, -2)) * ldexp(1.0, 8);
    default: return NAN;
    }
    return (2.0 - ldexp(1.0, 1 - p)) * ldexp(1.0, emax);
}

/* U for a format: log2 of its largest finite value (Figure 3's exp2 limit). */
double oracle_format_log2_max(int fmt) { return log2(format_max_finite(fmt)); }

/* Least integer a >= 0 with 2^a >= n  (= ceil(log2 n) for n >= 1). */
int32_t oracle_ceil_log2_count(int64_t n)
{
    int32_t a = 0;
    while (a < 62 && ((int64_t)1 << a) < n) a++;
    return a;
}

/* G = ceil(log2(max(1, m))) for finite m >= 0, exactly (Alg. 1 step 5). */
int32_t oracle_v_exponent(double m)
{
    if (!(m > 1.0)) return 0;
    int e;
    double f = frexp(m, &e); /* m = f * 2^e, f in [0.5, 1) */
    return (f == 0.5) ? e - 1 : e;
}

/* C = min(floor(U_exp), ceil(U_acc - A) - 1)  (Alg. 1 step 7). */
int32_t oracle_exponent_budget(int exp_fmt, int acc_fmt, int32_t A)
{
    double u_exp = oracle_format_log2_max(exp_fmt);
    double u_acc = oracle_format_log2_max(acc_fmt);
    double c1 = floor(u_exp);
    double c2 = ceil(u_acc - (double)A) - 1.0;
    return (int32_t)(c1 < c2 ? c1 : c2);
}

/* Algorithm 1, steps 1-7, plus the decision, for BH heads.
 * q: [BH][Nq][d], k, v: [BH][Nk][d] bit patterns in format in_fmt.
 * kbar_out: [BH][d] (may be NULL). */
int oracle_certify(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v, int in_fmt,
                   double scale_log2, int exp_fmt, int acc_fmt,
                   double *kbar_out, oracle_cert_t *out)
{
    if (in_fmt != ORC_IN_BF16 && in_fmt != ORC_IN_FP16) return 1;
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || !out) return 1;
    if (!isfinite(format_max_finite(exp_fmt)) || !isfinite(format_max_finite(acc_fmt))) return 1;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t h = 0; h < BH; h++) {
        const uint16_t *qh = q + h * Nq * d;
        const uint16_t *kh = k + h * Nk * d;
        const uint16_t *vh = v + h * Nk * d;
        double *kbar = (double *)malloc((size_t)d * sizeof(double));
        int finite = 1;

        /* step 1: kbar = N_k^-1 sum_r k_r */
        for (int64_t c = 0; c < d; c++) kbar[c] = 0.0;
        for (int64_t r = 0; r < Nk; r++)
            for (int64_t c = 0; c < d; c++) {
                double x = bits_to_double(kh[r * d + c], in_fmt);
                if (!isfinite(x)) finite = 0;
                kbar[c] += x;
            }
        for (int64_t c = 0; c < d; c++) kbar[c] /= (double)Nk;

        /* steps 2-3: kappa = max_r ||k_r - kbar||_2 (K~ is only used here) */
        double kappa = 0.0;
        for (int64_t r = 0; r < Nk; r++) {
            double ss = 0.0;
            for (int64_t c = 0; c < d; c++) {
                double t = bits_to_double(kh[r * d + c], in_fmt) - kbar[c];
                ss += t * t;
            }
            double nrm = sqrt(ss);
            if (nrm > kappa) kappa = nrm;
        }

        /* step 4: B_h = max_r BoundUp(q_r, kappa) = scale_log2 * max_r ||q_r|| * kappa */
        double qmax = 0.0;
        for (int64_t r = 0; r < Nq; r++) {
            double ss = 0.0;
            for (int64_t c = 0; c < d; c++) {
                double x = bits_to_double(qh[r * d + c], in_fmt);
                if (!isfinite(x)) finite = 0;
                ss += x * x;
            }
            double nrm = sqrt(ss);
            if (nrm > qmax) qmax = nrm;
        }
        double B = scale_log2 * qmax * kappa;

        /* step 5: G = ceil(log2 max(1, max |V|)) */
        double m = 0.0;
        for (int64_t r = 0; r < Nk; r++)
            for (int64_t c = 0; c < d; c++) {
                double x = bits_to_double(vh[r * d + c], in_fmt);
                if (!isfinite(x)) finite = 0;
                else if (fabs(x) > m) m = fabs(x);
            }

        oracle_cert_t res;
        memset(&res, 0, sizeof res);
        res.kappa = kappa;
        res.qmax = qmax;
        res.vmax = m;
        if (!finite) {
            res.certified = 0;
            res.reason = 2;
            res.B_h = INFINITY;
        } else {
            res.G = oracle_v_exponent(m);
            /* step 6 */
            res.A = oracle_ceil_log2_count(Nk) + res.G;
            /* step 7 */
            res.C = oracle_exponent_budget(exp_fmt, acc_fmt, res.A);
            res.B_h = B;
            res.certified = (B <= (double)res.C) ? 1 : 0;
            res.reason = res.certified ? 0 : 1;
            int lo = B * (1.0 - ldexp(1.0, -12)) <= (double)res.C;
            int hi = B * (1.0 + ldexp(1.0, -12)) <= (double)res.C;
            res.band = (lo != hi);
        }
        out[h] = res;
        if (kbar_out)
            for (int64_t c = 0; c < d; c++) kbar_out[h * d + c] = kbar[c];
        free(kbar);
    }
    return 0;
}

/* Per-prefix certificates for causal attention (Nq == Nk), one per block of
 * tile_rows consecutive query rows.  Reading (the pages certify causal heads
 * with the head's bound and state no finer rule): a causal row i sees keys
 * 0..i only, so |scale_log2 q_i . (k_j - kbar)| <= scale_log2 ||q_i|| kappa_i
 * with kappa_i = max_{j <= i} ||k_j - kbar||.  Over the rows of block b this
 * gives B_b = scale_log2 * max_{i in b} ||q_i|| * max_{j <= last row of b}
 * ||k_j - kbar||, compared with the head's budget C (steps 5-7 over the whole
 * head).  kbar is the head's mean, as the stabiliser mu_i uses it.
 * Outputs [BH][nb], nb = ceil(Nq / tile_rows): certified, band, B. */
int oracle_certify_prefix_tiles(int64_t BH, int64_t N, int64_t d, int64_t tile_rows,
                                const uint16_t *q, const uint16_t *k, const uint16_t *v, int in_fmt,
                                double scale_log2, int exp_fmt, int acc_fmt,
                                int32_t *cert_out, int32_t *band_out, double *B_out)
{
    if (in_fmt != ORC_IN_BF16 && in_fmt != ORC_IN_FP16) return 1;
    if (BH < 0 || N < 1 || d < 1 || tile_rows < 1 || !cert_out || !band_out || !B_out) return 1;
    if (!isfinite(format_max_finite(exp_fmt)) || !isfinite(format_max_finite(acc_fmt))) return 1;
    const int64_t nb = (N + tile_rows - 1) / tile_rows;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t h = 0; h < BH; h++) {
        const uint16_t *qh = q + h * N * d;
        const uint16_t *kh = k + h * N * d;
        const uint16_t *vh = v + h * N * d;
        double *kbar = (double *)malloc((size_t)d * sizeof(double));
        double *kpre = (double *)malloc((size_t)N * sizeof(double));
        int finite = 1;
        for (int64_t c = 0; c < d; c++) kbar[c] = 0.0;
        for (int64_t r = 0; r < N; r++)
            for (int64_t c = 0; c < d; c++) {
                double x = bits_to_double(kh[r * d + c], in_fmt);
                if (!isfinite(x)) finite = 0;
                kbar[c] += x;
            }
        for (int64_t c = 0; c < d; c++) kbar[c] /= (double)N;
        /* prefix maxima of the centred key norms */
        double run = 0.0;
        for (int64_t r = 0; r < N; r++) {
            double ss = 0.0;
            for (int64_t c = 0; c < d; c++) {
                double t = bits_to_double(kh[r * d + c], in_fmt) - kbar[c];
                ss += t * t;
            }
            double nrm = sqrt(ss);
            if (nrm > run) run = nrm;
            kpre[r] = run;
        }
        double m = 0.0;
        for (int64_t r = 0; r < N; r++)
            for (int64_t c = 0; c < d; c++) {
                double x = bits_to_double(vh[r * d + c], in_fmt);
                if (!isfinite(x)) finite = 0;
                else if (fabs(x) > m) m = fabs(x);
            }
        int32_t C = 0;
        if (finite) {
            int32_t A = oracle_ceil_log2_count(N) + oracle_v_exponent(m);
            C = oracle_exponent_budget(exp_fmt, acc_fmt, A);
        }
        for (int64_t b = 0; b < nb; b++) {
            const int64_t r0 = b * tile_rows;
            const int64_t r1 = (r0 + tile_rows < N) ? r0 + tile_rows : N;
            double qmax = 0.0;
            for (int64_t r = r0; r < r1; r++) {
                double ss = 0.0;
                for (int64_t c = 0; c < d; c++) {
                    double x = bits_to_double(qh[r * d + c], in_fmt);
                    if (!isfinite(x)) finite = 0;
                    ss += x * x;
                }
                double nrm = sqrt(ss);
                if (nrm > qmax) qmax = nrm;
            }
            const int64_t o = h * nb + b;
            B_out[o] = scale_log2 * qmax * kpre[r1 - 1];
            cert_out[o] = 0;
            band_out[o] = 0;
        }
        /* a non-finite value anywhere in the head (Q rows of later blocks
         * included) leaves every block uncertified */
        for (int64_t b = 0; b < nb && finite; b++) {
            const int64_t o = h * nb + b;
            const double B = B_out[o];
            cert_out[o] = (B <= (double)C) ? 1 : 0;
            int lo = B * (1.0 - ldexp(1.0, -12)) <= (double)C;
            int hi = B * (1.0 + ldexp(1.0, -12)) <= (double)C;
            band_out[o] = (lo != hi);
        }
        if (!finite)
            for (int64_t b = 0; b < nb; b++) B_out[h * nb + b] = INFINITY;
        free(kbar);
        free(kpre);
    }
    return 0;
}

/* One output row of softmax attention, two passes, fp64.
 * kh, vh: [Nk][d] already in fp64; jmax: last visible key (inclusive). */
static void attn_row(const double *qi, const double *kh, const double *vh,
                     int64_t jmax, int64_t d, double scale, double *s,
                     double *o, double *lse2)
{
    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int64_t j = 0; j <= jmax; j++) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; c++) acc += qi[c] * kh[j * d + c];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    /* pass 2: exp, row sum, P V */
    for (int64_t c = 0; c < d; c++) o[c] = 0.0;
    double l = 0.0;
    for (int64_t j = 0; j <= jmax; j++) {
        double p = exp(s[j] - m);
        l += p;
        for (int64_t c = 0; c < d; c++) o[c] += p * vh[j * d + c];
    }
    for (int64_t c = 0; c < d; c++) o[c] /= l;
    if (lse2) *lse2 = (m + log(l)) / log(2.0);
}

/* Shared driver: el = 0 -> inputs are bf16 bits, el = 1 -> inputs are fp64,
 * el = 2 -> inputs are fp16 bits.
 * rows: n_rows query indices (same for every head), or NULL for all rows.
 * out: [BH][n_rows][d]; lse2 (may be NULL): [BH][n_rows] = log2 sum_j exp(s_ij). */
static int attn_driver(int el, int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                       const void *q, const void *k, const void *v, double scale,
                       int causal, int64_t n_rows, const int64_t *rows,
                       double *out, double *lse2)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1) return 1;
    if (causal && Nq != Nk) return 1;
    if (!rows) n_rows = Nq;
    for (int64_t t = 0; rows && t < n_rows; t++)
        if (rows[t] < 0 || rows[t] >= Nq) return 1;

    double *kh = (double *)malloc((size_t)(Nk * d) * sizeof(double));
    double *vh = (double *)malloc((size_t)(Nk * d) * sizeof(double));
    if (!kh || !vh) { free(kh); free(vh); return 2; }

    for (int64_t h = 0; h < BH; h++) {
        for (int64_t e = 0; e < Nk * d; e++) {
            if (el != 1) {
                const int f = el == 2 ? ORC_IN_FP16 : ORC_IN_BF16;
                kh[e] = bits_to_double(((const uint16_t *)k)[h * Nk * d + e], f);
                vh[e] = bits_to_double(((const uint16_t *)v)[h * Nk * d + e], f);
            } else {
                kh[e] = ((const double *)k)[h * Nk * d + e];
                vh[e] = ((const double *)v)[h * Nk * d + e];
            }
        }
#pragma omp parallel
        {
            double *s = (double *)malloc((size_t)Nk * sizeof(double));
            double *qi = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < n_rows; t++) {
                int64_t i = rows ? rows[t] : t;
                for (int64_t c = 0; c < d; c++) {
                    int64_t e = (h * Nq + i) * d + c;
                    qi[c] = (el == 1) ? ((const double *)q)[e]
                                      : bits_to_double(((const uint16_t *)q)[e],
                                                       el == 2 ? ORC_IN_FP16 : ORC_IN_BF16);
                }
                int64_t jmax = causal ? i : Nk - 1;
                attn_row(qi, kh, vh, jmax, d, scale, s, out + (h * n_rows + t) * d,
                         lse2 ? lse2 + h * n_rows + t : NULL);
            }
            free(s);
            free(qi);
        }
    }
    free(kh);
    free(vh);
    return 0;
}

int oracle_attn_bf16(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     double scale, int causal, int64_t n_rows, const int64_t *rows,
                     double *out, double *lse2)
{
    return attn_driver(0, BH, Nq, Nk, d, q, k, v, scale, causal, n_rows, rows, out, lse2);
}

int oracle_attn_fp16(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     double scale, int causal, int64_t n_rows, const int64_t *rows,
                     double *out, double *lse2)
{
    return attn_driver(2, BH, Nq, Nk, d, q, k, v, scale, causal, n_rows, rows, out, lse2);
}

int oracle_attn_f64(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                    const double *q, const double *k, const double *v,
                    double scale, int causal, int64_t n_rows, const int64_t *rows,
                    double *out, double *lse2)
{
    return attn_driver(1, BH, Nq, Nk, d, q, k, v, scale, causal, n_rows, rows, out, lse2);
}

/* ---------------------------------------------------------------- backward
 *
 * For one head with scores x_ij = scale * q_i . k_j over the visible keys and
 * P_ij = softmax_j(x_ij) (row i sums to one):
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij
 *   dX_ij = P_ij (dP_ij - D_i)        (softmax Jacobian times dP, row i)
 *   dQ_i  = scale sum_j dX_ij k_j
 *   dK_j  = scale sum_i dX_ij q_i
 *
 * Pass 1 runs over rows (in parallel): the row's log-sum-exp, D_i and dQ_i.
 * Pass 2 runs over keys (in parallel): P_ij = exp(x_ij - lse_i) for every row
 * that sees key j, then dV_j and dK_j.  Inputs are decoded to fp64 first.
 * el: 0 bf16 bits, 1 fp64, 2 fp16 bits.  Outputs [BH][N][d] fp64.
 */
static double load_el(const void *a, int64_t e, int el)
{
    if (el == 1) return ((const double *)a)[e];
    return bits_to_double(((const uint16_t *)a)[e], el == 2 ? ORC_IN_FP16 : ORC_IN_BF16);
}

static int attn_bwd_driver(int el, int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                           const void *q, const void *k, const void *v, const void *dout,
                           double scale, int causal, double *dq, double *dk, double *dv)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1) return 1;
    if (causal && Nq != Nk) return 1;
    size_t nq = (size_t)(Nq * d), nk = (size_t)(Nk * d);
    double *qh = (double *)malloc((nq ? nq : 1) * sizeof(double));
    double *gh = (double *)malloc((nq ? nq : 1) * sizeof(double));
    double *kh = (double *)malloc(nk * sizeof(double));
    double *vh = (double *)malloc(nk * sizeof(double));
    double *lse = (double *)malloc((Nq ? (size_t)Nq : 1) * sizeof(double));
    double *D = (double *)malloc((Nq ? (size_t)Nq : 1) * sizeof(double));
    if (!qh || !gh || !kh || !vh || !lse || !D) {
        free(qh); free(gh); free(kh); free(vh); free(lse); free(D);
        return 2;
    }
    for (int64_t h = 0; h < BH; h++) {
        for (size_t e = 0; e < nq; e++) {
            qh[e] = load_el(q, (int64_t)(h * nq + e), el);
            gh[e] = load_el(dout, (int64_t)(h * nq + e), el);
        }
        for (size_t e = 0; e < nk; e++) {
            kh[e] = load_el(k, (int64_t)(h * nk + e), el);
            vh[e] = load_el(v, (int64_t)(h * nk + e), el);
        }
        double *dqh = dq + h * nq, *dkh = dk + h * nk, *dvh = dv + h * nk;

        /* pass 1: rows */
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)Nk * sizeof(double));
            double *dp = (double *)malloc((size_t)Nk * sizeof(double));
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < Nq; i++) {
                const double *qi = qh + i * d, *gi = gh + i * d;
                int64_t jmax = causal ? i : Nk - 1;
                double m = -INFINITY;
                for (int64_t j = 0; j <= jmax; j++) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; c++) acc += qi[c] * kh[j * d + c];
                    x[j] = scale * acc;
                    if (x[j] > m) m = x[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j <= jmax; j++) l += exp(x[j] - m);
                lse[i] = m + log(l);
                double Di = 0.0;
                for (int64_t j = 0; j <= jmax; j++) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; c++) acc += gi[c] * vh[j * d + c];
                    dp[j] = acc;
                    Di += exp(x[j] - lse[i]) * acc;
                }
                D[i] = Di;
                double *o = dqh + i * d;
                for (int64_t c = 0; c < d; c++) o[c] = 0.0;
                for (int64_t j = 0; j <= jmax; j++) {
                    double dx = exp(x[j] - lse[i]) * (dp[j] - Di);
                    for (int64_t c = 0; c < d; c++) o[c] += dx * kh[j * d + c];
                }
                for (int64_t c = 0; c < d; c++) o[c] *= scale;
            }
            free(x);
            free(dp);
        }

        /* pass 2: keys */
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t j = 0; j < Nk; j++) {
            const double *kj = kh + j * d, *vj = vh + j * d;
            double *gk = dkh + j * d, *gv = dvh + j * d;
            for (int64_t c = 0; c < d; c++) { gk[c] = 0.0; gv[c] = 0.0; }
            for (int64_t i = causal ? j : 0; i < Nq; i++) {
                const double *qi = qh + i * d, *gi = gh + i * d;
                double s = 0.0, dpij = 0.0;
                for (int64_t c = 0; c < d; c++) {
                    s += qi[c] * kj[c];
                    dpij += gi[c] * vj[c];
                }
                double pij = exp(scale * s - lse[i]);
                double dx = pij * (dpij - D[i]);
                for (int64_t c = 0; c < d; c++) {
                    gv[c] += pij * gi[c];
                    gk[c] += dx * qi[c];
                }
            }
            for (int64_t c = 0; c < d; c++) gk[c] *= scale;
        }
    }
    free(qh); free(gh); free(kh); free(vh); free(lse); free(D);
    return 0;
}

/* dQ for selected query rows only (each row's pass 1 needs only its own
 * scores), for sizes where the key-side pass is out of reach.  rows: n_rows
 * indices shared by every head; dq: [BH][n_rows][d]. */
static int attn_bwd_dq_rows_driver(int el, int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                                   const void *q, const void *k, const void *v, const void *dout,
                                   double scale, int causal, int64_t n_rows, const int64_t *rows,
                                   double *dq)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || n_rows < 0 || !rows) return 1;
    if (causal && Nq != Nk) return 1;
    for (int64_t t = 0; t < n_rows; t++)
        if (rows[t] < 0 || rows[t] >= Nq) return 1;
    size_t nk = (size_t)(Nk * d);
    double *kh = (double *)malloc(nk * sizeof(double));
    double *vh = (double *)malloc(nk * sizeof(double));
    if (!kh || !vh) { free(kh); free(vh); return 2; }
    for (int64_t h = 0; h < BH; h++) {
        for (size_t e = 0; e < nk; e++) {
            kh[e] = load_el(k, (int64_t)(h * nk + e), el);
            vh[e] = load_el(v, (int64_t)(h * nk + e), el);
        }
#pragma omp parallel
        {
            double *x = (double *)malloc((size_t)Nk * sizeof(double));
            double *dp = (double *)malloc((size_t)Nk * sizeof(double));
            double *qi = (double *)malloc((size_t)d * sizeof(double));
            double *gi = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < n_rows; t++) {
                int64_t i = rows[t];
                for (int64_t c = 0; c < d; c++) {
                    qi[c] = load_el(q, (h * Nq + i) * d + c, el);
                    gi[c] = load_el(dout, (h * Nq + i) * d + c, el);
                }
                int64_t jmax = causal ? i : Nk - 1;
                double m = -INFINITY;
                for (int64_t j = 0; j <= jmax; j++) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; c++) acc += qi[c] * kh[j * d + c];
                    x[j] = scale * acc;
                    if (x[j] > m) m = x[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j <= jmax; j++) l += exp(x[j] - m);
                double lse = m + log(l), Di = 0.0;
                for (int64_t j = 0; j <= jmax; j++) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < d; c++) acc += gi[c] * vh[j * d + c];
                    dp[j] = acc;
                    Di += exp(x[j] - lse) * acc;
                }
                double *o = dq + (h * n_rows + t) * d;
                for (int64_t c = 0; c < d; c++) o[c] = 0.0;
                for (int64_t j = 0; j <= jmax; j++) {
                    double dx = exp(x[j] - lse) * (dp[j] - Di);
                    for (int64_t c = 0; c < d; c++) o[c] += dx * kh[j * d + c];
                }
                for (int64_t c = 0; c < d; c++) o[c] *= scale;
            }
            free(x); free(dp); free(qi); free(gi);
        }
    }
    free(kh);
    free(vh);
    return 0;
}

int oracle_attn_bwd_dq_rows(int el, int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                            const void *q, const void *k, const void *v, const void *dout,
                            double scale, int causal, int64_t n_rows, const int64_t *rows, double *dq)
{
    if (el < 0 || el > 2) return 1;
    return attn_bwd_dq_rows_driver(el, BH, Nq, Nk, d, q, k, v, dout, scale, causal, n_rows, rows, dq);
}

int oracle_attn_bwd_bf16(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                         const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                         double scale, int causal, double *dq, double *dk, double *dv)
{
    return attn_bwd_driver(0, BH, Nq, Nk, d, q, k, v, dout, scale, causal, dq, dk, dv);
}

int oracle_attn_bwd_fp16(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                         const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                         double scale, int causal, double *dq, double *dk, double *dv)
{
    return attn_bwd_driver(2, BH, Nq, Nk, d, q, k, v, dout, scale, causal, dq, dk, dv);
}

int oracle_attn_bwd_f64(int64_t BH, int64_t Nq, int64_t Nk, int64_t d,
                        const double *q, const double *k, const double *v, const double *dout,
                        double scale, int causal, double *dq, double *dk, double *dv)
{
    return attn_bwd_driver(1, BH, Nq, Nk, d, q, k, v, dout, scale, causal, dq, dk, dv);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
