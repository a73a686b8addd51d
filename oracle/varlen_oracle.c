/*
 * varlen_oracle.c -- plain fp64 CPU oracle for packed variable-length
 * (cu_seqlens) multi-head scaled-dot-product attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker for the CUDA
 * library in packed_variable_length_varlen_gb300/.  Only tests/, the smoke
 * check in __graft_entry__.py and the CPU-baseline leg of bench.py may load it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (the definition, written out; no online rescaling, no
 * tiling, no fusion):
 *
 *   Inputs are bf16 (or, for finite-difference pins, fp64) tensors in NHD
 *   layout: element (row r, head h, dim d) sits at
 *       base + r*row_stride + h*head_stride + d            (int64 elements).
 *   Segment b owns q rows [cu_q[b], cu_q[b+1]) and kv rows [cu_k[b], cu_k[b+1]).
 *   This is the packed "cu_seqlens" interface of flash_attn_varlen_func as used
 *   on the flash-attention issue pages ("[FA4] cute varlen backward: int32
 *   overflow in _bwd_preprocess", section "Minimal repro", and "[FA4][SM120]
 *   flash_attn_varlen_func ... illegal memory access at >=4 varlen segments",
 *   section "Bug 2 details": cu_seqlens_q / cu_seqlens_k, non-causal).
 *
 *   For q row i of segment b, head h, kv rows j of the same segment:
 *     s_ij   = scale * sum_d q[i,h,d] k[j,h,d]
 *     m_i    = max_j s_ij
 *     LSE_i  = m_i + ln sum_j exp(s_ij - m_i)        (natural log)
 *     P_ij   = exp(s_ij - LSE_i)
 *     o_i    = sum_j P_ij v_j
 *   An empty key set (Sk_b = 0) gives LSE_i = -inf and o_i = 0.
 *
 *   Backward, for an upstream gradient dO (the varlen backward of the same
 *   issue page, "Summary": gradients dQ/dK/dV of the attention output):
 *     delta_i = sum_d dO_i[d] o_i[d]        (exact fp64 o_i)
 *     dP_ij   = dO_i . v_j
 *     dS_ij   = P_ij (dP_ij - delta_i)
 *     dq_i    = scale sum_j dS_ij k_j
 *     dk_j    = scale sum_i dS_ij q_i
 *     dv_j    = sum_i P_ij dO_i
 *   Empty sums are zero (dq of an empty-key segment, dk/dv of an empty-query
 *   segment).
 *
 *   Masks (window_left, window_right).  The pages call the varlen function
 *   with causal=False and no window only; for the masked forms this oracle
 *   takes the conventions of the API they call.  The diagonal meets the last
 *   key at the last query: with d = Sk - Sq, q row ii of a segment (0-based
 *   within it) sees the kv rows jj (0-based) with
 *       ii + d - window_left  <=  jj  <=  ii + d + window_right,
 *   a negative window side being unbounded.  Causal is window_right = 0
 *   (jj <= ii + d); no mask is (-1, -1).  Every sum over j above then runs
 *   over the visible keys only; a row that sees none gets LSE = -inf, o = 0
 *   and dq = 0, and adds nothing to dk / dv.
 *
 * All index arithmetic is int64.  Rows are looked up in cu_seqlens by a
 * linear scan.  OpenMP parallelises over independent (row, head) pairs only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    const void *q, *k, *v, *dout;   /* element type given by dtype          */
    int64_t q_rs, q_hs;             /* row / head strides, in elements      */
    int64_t k_rs, k_hs;
    int64_t v_rs, v_hs;
    int64_t do_rs, do_hs;
    const int32_t *cu_q, *cu_k;     /* batch + 1 entries each               */
    int32_t batch, num_heads, head_dim;
    int32_t dtype;                  /* 0 = bf16 bit patterns, 1 = fp64      */
    double scale;
    int32_t window_left;            /* mask sides, < 0 unbounded (see       */
    int32_t window_right;           /* visible_range); causal = (-1, 0)     */
} oracle_problem;

/* Exact widening of a bf16 bit pattern: the bf16 bits are the top half of an
 * IEEE binary32. */
static double bf16_bits_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load(const void *base, int32_t dtype, int64_t idx) {
    if (dtype == 0) return bf16_bits_to_f64(((const uint16_t *)base)[idx]);
    return ((const double *)base)[idx];
}

/* Row vector x[d] = T[row, h, :] widened to fp64. */
static void load_row(const void *base, int32_t dtype, int64_t rs, int64_t hs,
                     int64_t row, int32_t h, int32_t D, double *x) {
    int64_t off = row * rs + (int64_t)h * hs;
    for (int32_t d = 0; d < D; ++d) x[d] = load(base, dtype, off + d);
}

static double dot(const double *a, const double *b, int32_t D) {
    double acc = 0.0;
    for (int32_t d = 0; d < D; ++d) acc += a[d] * b[d];
    return acc;
}

/* The segment that holds row i: the b with cu[b] <= i < cu[b+1].  Returns -1
 * when no segment holds it. */
static int32_t segment_of(const int32_t *cu, int32_t batch, int64_t i) {
    for (int32_t b = 0; b < batch; ++b)
        if ((int64_t)cu[b] <= i && i < (int64_t)cu[b + 1]) return b;
    return -1;
}

/* The keys [*lo, *hi) (0-based within the segment) that q row ii of a
 * segment with Sq query and Sk key rows sees: all Sk without a mask; else,
 * with diag = ii + Sk - Sq, those with jj >= diag - window_left (if
 * window_left >= 0) and jj <= diag + window_right (if window_right >= 0).
 * Empty: *lo == *hi. */
static void band_range(int64_t Sq, int64_t Sk, int64_t ii, int32_t window_left, int32_t window_right,
                       int64_t *lo, int64_t *hi) {
    const int64_t diag = ii + (Sk - Sq);
    int64_t a = 0, e = Sk;
    if (window_left >= 0 && diag - window_left > a) a = diag - window_left;
    if (window_right >= 0 && diag + window_right + 1 < e) e = diag + window_right + 1;
    if (e < a) e = a;
    *lo = a;
    *hi = e;
}

/* band_range for q row ii of segment b of a bf16 / fp64 problem. */
static void visible_range(const oracle_problem *pb, int32_t b, int64_t ii,
                          int64_t *lo, int64_t *hi) {
    band_range((int64_t)pb->cu_q[b + 1] - pb->cu_q[b], (int64_t)pb->cu_k[b + 1] - pb->cu_k[b], ii,
               pb->window_left, pb->window_right, lo, hi);
}

/* Forward for one (q row, head): s, LSE, P and o by the definition above.
 * s is scratch of length >= Sk (s[j] for the visible keys j).  Returns the segment, -1 if the row is
 * in none. */
static int32_t row_forward(const oracle_problem *pb, int64_t i, int32_t h,
                           double *qi, double *kj, double *s, double *out_o,
                           double *out_lse) {
    const int32_t D = pb->head_dim;
    int32_t b = segment_of(pb->cu_q, pb->batch, i);
    if (b < 0) return -1;
    const int64_t k0 = pb->cu_k[b];
    int64_t jlo, jhi;
    visible_range(pb, b, i - pb->cu_q[b], &jlo, &jhi);
    load_row(pb->q, pb->dtype, pb->q_rs, pb->q_hs, i, h, D, qi);
    for (int32_t d = 0; d < D; ++d) out_o[d] = 0.0;
    if (jhi <= jlo) {
        *out_lse = -INFINITY;
        return b;
    }
    double m = -INFINITY;
    for (int64_t j = jlo; j < jhi; ++j) {
        load_row(pb->k, pb->dtype, pb->k_rs, pb->k_hs, k0 + j, h, D, kj);
        s[j] = pb->scale * dot(qi, kj, D);
        if (s[j] > m) m = s[j];
    }
    double sum = 0.0;
    for (int64_t j = jlo; j < jhi; ++j) sum += exp(s[j] - m);
    const double lse = m + log(sum);
    for (int64_t j = jlo; j < jhi; ++j) {
        const double p = exp(s[j] - lse);
        load_row(pb->v, pb->dtype, pb->v_rs, pb->v_hs, k0 + j, h, D, kj);
        for (int32_t d = 0; d < D; ++d) out_o[d] += p * kj[d];
    }
    *out_lse = lse;
    return b;
}

static int64_t max_seg_len(const int32_t *cu, int32_t batch) {
    int64_t mx = 1;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t len = (int64_t)cu[b + 1] - cu[b];
        if (len > mx) mx = len;
    }
    return mx;
}

/*
 * Forward on selected (q row, head) pairs.
 *   rows[n], heads[n] : packed q row index and head of each pair.
 *   out : [n][D] fp64;  lse : [n] fp64.
 * Rows outside every segment get NaN.  Returns 0.
 */
int oracle_fwd(const oracle_problem *pb, int64_t n, const int64_t *rows,
               const int32_t *heads, double *out, double *lse) {
    const int32_t D = pb->head_dim;
    const int64_t smax = max_seg_len(pb->cu_k, pb->batch);
#pragma omp parallel
    {
        double *qi = malloc(sizeof(double) * D), *kj = malloc(sizeof(double) * D);
        double *s = malloc(sizeof(double) * smax);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; ++t) {
            double *o = out + t * D;
            if (row_forward(pb, rows[t], heads[t], qi, kj, s, o, lse + t) < 0) {
                for (int32_t d = 0; d < D; ++d) o[d] = NAN;
                lse[t] = NAN;
            }
        }
        free(qi); free(kj); free(s);
    }
    return 0;
}

/*
 * Backward, query side, on selected (q row, head) pairs:
 *   dq    : [n][D]   scale * sum_j dS_ij k_j
 *   delta : [n]      dO_i . o_i with the exact o_i
 * Requires pb->dout.
 */
int oracle_bwd_q(const oracle_problem *pb, int64_t n, const int64_t *rows,
                 const int32_t *heads, double *dq, double *delta) {
    const int32_t D = pb->head_dim;
    const int64_t smax = max_seg_len(pb->cu_k, pb->batch);
#pragma omp parallel
    {
        double *qi = malloc(sizeof(double) * D), *kj = malloc(sizeof(double) * D);
        double *oi = malloc(sizeof(double) * D), *doi = malloc(sizeof(double) * D);
        double *s = malloc(sizeof(double) * smax);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t i = rows[t];
            const int32_t h = heads[t];
            double *g = dq + t * D, lse;
            int32_t b = row_forward(pb, i, h, qi, kj, s, oi, &lse);
            for (int32_t d = 0; d < D; ++d) g[d] = 0.0;
            if (b < 0) {
                for (int32_t d = 0; d < D; ++d) g[d] = NAN;
                delta[t] = NAN;
                continue;
            }
            load_row(pb->dout, pb->dtype, pb->do_rs, pb->do_hs, i, h, D, doi);
            const double dlt = dot(doi, oi, D);
            delta[t] = dlt;
            const int64_t k0 = pb->cu_k[b];
            int64_t jlo, jhi;
            visible_range(pb, b, i - pb->cu_q[b], &jlo, &jhi);
            for (int64_t j = jlo; j < jhi; ++j) {
                const double p = exp(s[j] - lse);
                load_row(pb->v, pb->dtype, pb->v_rs, pb->v_hs, k0 + j, h, D, kj);
                const double dp = dot(doi, kj, D);
                const double ds = p * (dp - dlt);
                load_row(pb->k, pb->dtype, pb->k_rs, pb->k_hs, k0 + j, h, D, kj);
                for (int32_t d = 0; d < D; ++d) g[d] += pb->scale * ds * kj[d];
            }
        }
        free(qi); free(kj); free(oi); free(doi); free(s);
    }
    return 0;
}

/* dk_j and dv_j of kv row j (segment b, head h) by the sums over the
 * segment's q rows i of the definition, given L[ii] = LSE_i and E[ii] =
 * delta_i of every q row (ii = i - cu_q[b]).  Scratch: qi, kj, vj, doi of
 * length D each. */
static void kv_row_grad(const oracle_problem *pb, int32_t b, int32_t h, int64_t j, const double *L,
                        const double *E, double *qi, double *kj, double *vj, double *doi,
                        double *gk, double *gv) {
    const int32_t D = pb->head_dim;
    for (int32_t d = 0; d < D; ++d) gk[d] = gv[d] = 0.0;
    load_row(pb->k, pb->dtype, pb->k_rs, pb->k_hs, j, h, D, kj);
    load_row(pb->v, pb->dtype, pb->v_rs, pb->v_hs, j, h, D, vj);
    const int64_t q0 = pb->cu_q[b], Sq = (int64_t)pb->cu_q[b + 1] - pb->cu_q[b];
    const int64_t jj = j - pb->cu_k[b];  /* key index within the segment */
    for (int64_t ii = 0; ii < Sq; ++ii) {
        int64_t jlo, jhi;
        visible_range(pb, b, ii, &jlo, &jhi);
        if (jj < jlo || jj >= jhi) continue;  /* masked: P_ij = 0 */
        load_row(pb->q, pb->dtype, pb->q_rs, pb->q_hs, q0 + ii, h, D, qi);
        load_row(pb->dout, pb->dtype, pb->do_rs, pb->do_hs, q0 + ii, h, D, doi);
        const double sij = pb->scale * dot(qi, kj, D);
        const double p = exp(sij - L[ii]);
        const double dp = dot(doi, vj, D);
        const double ds = p * (dp - E[ii]);
        for (int32_t d = 0; d < D; ++d) {
            gv[d] += p * doi[d];
            gk[d] += pb->scale * ds * qi[d];
        }
    }
}

/*
 * Backward, key/value side, on selected (kv row, head) pairs:
 *   dk : [n][D]   scale * sum_i dS_ij q_i
 *   dv : [n][D]   sum_i P_ij dO_i
 * dk_j and dv_j need LSE_i and delta_i of every q row i of the segment, so
 * this first runs the row forward for all q rows of each (segment, head)
 * touched by the request, then sums over i.  Cost: O(Sq_b * Sk_b * D) per
 * touched (segment, head).
 */
int oracle_bwd_kv(const oracle_problem *pb, int64_t n, const int64_t *rows,
                  const int32_t *heads, double *dk, double *dv) {
    const int32_t D = pb->head_dim, B = pb->batch, H = pb->num_heads;
    const int64_t smax = max_seg_len(pb->cu_k, B);
    int32_t *seg = malloc(sizeof(int32_t) * (n > 0 ? n : 1));
    /* stats[b*H + h]: LSE_i and delta_i for all q rows of segment b, head h. */
    double **st_lse = calloc((size_t)B * H, sizeof(double *));
    double **st_dlt = calloc((size_t)B * H, sizeof(double *));
    for (int64_t t = 0; t < n; ++t) {
        seg[t] = segment_of(pb->cu_k, B, rows[t]);
        if (seg[t] < 0 || heads[t] < 0 || heads[t] >= H) { seg[t] = -1; continue; }
        const int64_t x = (int64_t)seg[t] * H + heads[t];
        if (st_lse[x]) continue;
        const int32_t b = seg[t], h = heads[t];
        const int64_t q0 = pb->cu_q[b], Sq = (int64_t)pb->cu_q[b + 1] - pb->cu_q[b];
        double *L = malloc(sizeof(double) * (Sq > 0 ? Sq : 1));
        double *E = malloc(sizeof(double) * (Sq > 0 ? Sq : 1));
        st_lse[x] = L;
        st_dlt[x] = E;
#pragma omp parallel
        {
            double *qi = malloc(sizeof(double) * D), *kj = malloc(sizeof(double) * D);
            double *oi = malloc(sizeof(double) * D), *doi = malloc(sizeof(double) * D);
            double *s = malloc(sizeof(double) * smax);
#pragma omp for schedule(dynamic, 8)
            for (int64_t ii = 0; ii < Sq; ++ii) {
                row_forward(pb, q0 + ii, h, qi, kj, s, oi, &L[ii]);
                load_row(pb->dout, pb->dtype, pb->do_rs, pb->do_hs, q0 + ii, h, D, doi);
                E[ii] = dot(doi, oi, D);
            }
            free(qi); free(kj); free(oi); free(doi); free(s);
        }
    }
#pragma omp parallel
    {
        double *qi = malloc(sizeof(double) * D), *kj = malloc(sizeof(double) * D);
        double *vj = malloc(sizeof(double) * D), *doi = malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t j = rows[t];
            const int32_t h = heads[t], b = seg[t];
            double *gk = dk + t * D, *gv = dv + t * D;
            for (int32_t d = 0; d < D; ++d) gk[d] = gv[d] = 0.0;
            if (b < 0) {
                for (int32_t d = 0; d < D; ++d) gk[d] = gv[d] = NAN;
                continue;
            }
            const double *L = st_lse[(int64_t)b * H + h], *E = st_dlt[(int64_t)b * H + h];
            kv_row_grad(pb, b, h, j, L, E, qi, kj, vj, doi, gk, gv);
        }
        free(qi); free(kj); free(vj); free(doi);
    }
    for (int64_t x = 0; x < (int64_t)B * H; ++x) { free(st_lse[x]); free(st_dlt[x]); }
    free(st_lse); free(st_dlt); free(seg);
    return 0;
}

/*
 * Backward, key/value side, for kv rows of one (segment b, head h), given the
 * statistics of every q row of that segment: lse[ii] = LSE_i and
 * delta[ii] = delta_i for ii = 0 .. Sq_b - 1 (the values oracle_fwd and
 * oracle_bwd_q return for those rows).  The sums over i are those of
 * oracle_bwd_kv; only where LSE_i and delta_i come from differs, so that a
 * caller can compute them once per (segment, head) of a long segment.
 *   dk, dv : [n][D].  Rows outside segment b's kv rows get NaN.
 */
int oracle_bwd_kv_stats(const oracle_problem *pb, int32_t b, int32_t h, int64_t n, const int64_t *rows,
                        const double *lse, const double *delta, double *dk, double *dv) {
    const int32_t D = pb->head_dim;
    if (b < 0 || b >= pb->batch || h < 0 || h >= pb->num_heads) return -1;
#pragma omp parallel
    {
        double *qi = malloc(sizeof(double) * D), *kj = malloc(sizeof(double) * D);
        double *vj = malloc(sizeof(double) * D), *doi = malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t j = rows[t];
            double *gk = dk + t * D, *gv = dv + t * D;
            if (j < pb->cu_k[b] || j >= pb->cu_k[b + 1]) {
                for (int32_t d = 0; d < D; ++d) gk[d] = gv[d] = NAN;
                continue;
            }
            kv_row_grad(pb, b, h, j, lse, delta, qi, kj, vj, doi, gk, gv);
        }
        free(qi); free(kj); free(vj); free(doi);
    }
    return 0;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------ FP8 forward
 *
 * Low-precision forward.  The pages quote quantised attention only by its
 * accuracy (the ffpa-attn NVFP4 pull request, "Summary": cos ~0.982 against
 * SDPA) and mention an fp8 fallback (the "[FA4][SM120]" issue, "Practical
 * workaround"); neither defines the arithmetic.  This oracle takes the
 * plainest reading for OCP FP8 E4M3 ("e4m3fn": 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits, no infinities, largest finite 448, code 0x7F / 0xFF NaN):
 * Q, K, V are E4M3 codes with one fp32 descale factor per (segment, head)
 * and tensor, and for q row i of segment b, head h:
 *     s_ij  = scale * qd[b,h] * kd[b,h] * sum_d q8[i,d] k8[j,d]
 *     m_i   = max_j s_ij,   p_ij = exp(s_ij - m_i),   l_i = sum_j p_ij
 *     o_i   = vd[b,h] * sum_j e4m3(p_ij) v8[j] / l_i
 *     LSE_i = m_i + ln l_i
 * where e4m3(x) rounds to the nearest E4M3 value, ties to even, saturating
 * at +-448 (P is rounded to E4M3 for the P V product; the row sum uses the
 * unrounded p).  quantize_p = 0 skips that rounding.  Empty key sets give
 * LSE = -inf and o = 0, as above.  With a mask (window_left, window_right,
 * the band of the bf16 forward above: band_range) j runs over the keys row
 * i sees; a row that sees none gets LSE = -inf and o = 0.
 */

/* Value of an E4M3 code. */
static double e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);           /* subnormal: m * 2^-9 */
    else v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Nearest E4M3 value to x (ties to even), saturating at +-448; NaN stays. */
static double e4m3_round(double x) {
    if (isnan(x)) return x;
    const double a = fabs(x);
    if (a == 0.0) return x;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E < -6) E = -6;           /* below the smallest normal the spacing stays 2^-9 */
    const double q = ldexp(1.0, E - 3);
    double r = nearbyint(a / q) * q;   /* default rounding mode: to nearest, ties to even */
    if (r > 448.0) r = 448.0;
    return x < 0 ? -r : r;
}

/* Code of an E4M3 value (x must be one: e4m3_round's output). */
static uint8_t e4m3_code(double x) {
    if (isnan(x)) return 0x7F;
    const uint8_t s = (signbit(x) ? 0x80 : 0);
    const double a = fabs(x);
    if (a == 0.0) return s;
    int e;
    frexp(a, &e);
    const int E = e - 1;
    if (E < -6) return (uint8_t)(s | (uint8_t)(a / ldexp(1.0, -9)));        /* subnormal */
    const int m = (int)(a / ldexp(1.0, E - 3)) - 8;
    return (uint8_t)(s | ((E + 7) << 3) | m);
}

int oracle_e4m3_round(int64_t n, const double *in, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_round(in[i]);
    return 0;
}

int oracle_e4m3_decode(int64_t n, const uint8_t *in, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
    return 0;
}

/* Codes of the values nearest to in[i] (rounded as e4m3_round). */
int oracle_e4m3_encode(int64_t n, const double *in, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_code(e4m3_round(in[i]));
    return 0;
}

typedef struct {
    const uint8_t *q, *k, *v;       /* E4M3 codes                           */
    int64_t q_rs, q_hs;             /* row / head strides, in elements      */
    int64_t k_rs, k_hs;
    int64_t v_rs, v_hs;
    const int32_t *cu_q, *cu_k;     /* batch + 1 entries each               */
    int32_t batch, num_heads, head_dim;
    double scale;
    const double *q_descale, *k_descale, *v_descale;  /* [batch * num_heads] */
    int32_t quantize_p;             /* 1: P rounded to E4M3 for P V         */
    int32_t window_left;            /* mask sides, < 0 unbounded            */
    int32_t window_right;           /* (band_range); causal = (-1, 0)       */
} oracle_fp8_problem;

static void load_row8(const uint8_t *base, int64_t rs, int64_t hs, int64_t row, int32_t h, int32_t D, double *x) {
    const int64_t off = row * rs + (int64_t)h * hs;
    for (int32_t d = 0; d < D; ++d) x[d] = e4m3_value(base[off + d]);
}

/*
 * FP8 forward on selected (q row, head) pairs, by the definition above.
 *   out : [n][D] fp64;  lse : [n] fp64.  Rows outside every segment: NaN.
 */
int oracle_fwd_fp8(const oracle_fp8_problem *pb, int64_t n, const int64_t *rows, const int32_t *heads,
                   double *out, double *lse) {
    const int32_t D = pb->head_dim, H = pb->num_heads;
    const int64_t smax = max_seg_len(pb->cu_k, pb->batch);
#pragma omp parallel
    {
        double *qi = malloc(sizeof(double) * D), *kj = malloc(sizeof(double) * D);
        double *s = malloc(sizeof(double) * smax);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; ++t) {
            const int64_t i = rows[t];
            const int32_t h = heads[t];
            double *o = out + t * D;
            const int32_t b = segment_of(pb->cu_q, pb->batch, i);
            if (b < 0) {
                for (int32_t d = 0; d < D; ++d) o[d] = NAN;
                lse[t] = NAN;
                continue;
            }
            const int64_t k0 = pb->cu_k[b], Sk = (int64_t)pb->cu_k[b + 1] - pb->cu_k[b];
            const int64_t Sq = (int64_t)pb->cu_q[b + 1] - pb->cu_q[b];
            const int64_t bh = (int64_t)b * H + h;
            const double sqk = pb->scale * pb->q_descale[bh] * pb->k_descale[bh];
            int64_t jlo, jhi;
            band_range(Sq, Sk, i - pb->cu_q[b], pb->window_left, pb->window_right, &jlo, &jhi);
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (jhi <= jlo) {
                lse[t] = -INFINITY;
                continue;
            }
            load_row8(pb->q, pb->q_rs, pb->q_hs, i, h, D, qi);
            double m = -INFINITY;
            for (int64_t j = jlo; j < jhi; ++j) {
                load_row8(pb->k, pb->k_rs, pb->k_hs, k0 + j, h, D, kj);
                s[j] = sqk * dot(qi, kj, D);
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t j = jlo; j < jhi; ++j) l += exp(s[j] - m);
            for (int64_t j = jlo; j < jhi; ++j) {
                double p = exp(s[j] - m);
                if (pb->quantize_p) p = e4m3_round(p);
                load_row8(pb->v, pb->v_rs, pb->v_hs, k0 + j, h, D, kj);
                for (int32_t d = 0; d < D; ++d) o[d] += p * kj[d];
            }
            for (int32_t d = 0; d < D; ++d) o[d] *= pb->v_descale[bh] / l;
            lse[t] = m + log(l);
        }
        free(qi); free(kj); free(s);
    }
    return 0;
}
