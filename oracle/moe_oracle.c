/*
 * fp64 CPU oracle for the MoE-layer forward.  TEST INFRASTRUCTURE ONLY: it is
 * called by the tests, by the smoke check and by the benchmark's CPU-baseline
 * leg, never by the product path.  It shares no code with the CUDA library.
 *
 * What it computes is the plain definition of the layer, taken from
 * "Mixture-of-Kittens: MoE Megakernel for NVL72s" (Sec. 2.1, Eq. "MoE") and the
 * vendor blog post ("Overlapping computation and communication in MoE", the
 * MoE(x,s) and E_i(x) formulas):
 *
 *   MoE(x) = f_shared(x) + sum_{i in E} g_i f_i(x),   g_i = s_i / sum_{j in E} s_j
 *   f_i(x) = W_down^(i) ( SiLU(W_gate^(i) x) * W_up^(i) x )
 *
 * with E the k experts of highest router score.  Everything is evaluated in
 * fp64 on the exact values of the bf16 (or dequantised MXFP8) inputs; nothing
 * is rounded in between.  Readings where the pages are silent:
 *   - router bias beta is added to the logits before the score function;
 *   - score: sigmoid(logit) or softmax over all E logits;
 *   - top-k = the first k of a full sort by (score descending, expert id
 *     ascending); the k selected experts are then listed by ascending expert
 *     id ("slot order"), route j = t*k + slot;
 *   - out = f_shared + sum over slots 0..k-1 in that order.
 * The schedule follows Algorithm 1 (pull-based dispatch schedule) with one
 * rank.  The MX quantiser follows the OCP Microscaling Formats (MX) v1.0
 * specification for MXFP8 E4M3 with 32-element blocks, the format the paper
 * cites for its MXFP8 mode (Sec. 3.4, "MXFP8 Support").
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { SCORE_SIGMOID = 0, SCORE_SOFTMAX = 1 };

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* exact value of a bf16 bit pattern */
static inline double bf(uint16_t v) {
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* sum_d w[d] * v[d] for a bf16 row w and an fp64 vector v (four partial sums) */
static double dot_bf16(const uint16_t *w, const double *v, int64_t n) {
    double a0 = 0, a1 = 0, a2 = 0, a3 = 0;
    int64_t d = 0;
    for (; d + 4 <= n; d += 4) {
        a0 += bf(w[d]) * v[d];
        a1 += bf(w[d + 1]) * v[d + 1];
        a2 += bf(w[d + 2]) * v[d + 2];
        a3 += bf(w[d + 3]) * v[d + 3];
    }
    for (; d < n; ++d) a0 += bf(w[d]) * v[d];
    return (a0 + a1) + (a2 + a3);
}

static double dot_f64(const double *w, const double *v, int64_t n) {
    double a0 = 0, a1 = 0, a2 = 0, a3 = 0;
    int64_t d = 0;
    for (; d + 4 <= n; d += 4) {
        a0 += w[d] * v[d];
        a1 += w[d + 1] * v[d + 1];
        a2 += w[d + 2] * v[d + 2];
        a3 += w[d + 3] * v[d + 3];
    }
    for (; d < n; ++d) a0 += w[d] * v[d];
    return (a0 + a1) + (a2 + a3);
}

static inline double silu(double v) { return v / (1.0 + exp(-v)); }

/* ------------------------------------------------------------------ MX (OCP MX v1.0) */

/* value of an FP8 E4M3 (OCP "E4M3", no infinities, S.1111.111 = NaN) code */
double oracle_e4m3_value(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0xF && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* round-to-nearest-even to E4M3, saturating at +-448 (largest normal) */
uint8_t oracle_e4m3_encode(double v) {
    uint8_t sign = (v < 0) ? 0x80 : 0;
    double a = fabs(v);
    if (!(a == a)) return 0x7F; /* NaN in -> NaN */
    int e;
    if (a < ldexp(1.0, -6)) {
        e = -6; /* subnormal range: quantum 2^-9 */
    } else {
        frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
        e -= 1;       /* floor(log2 a) */
    }
    double quantum = ldexp(1.0, e - 3);
    double q = nearbyint(a / quantum) * quantum; /* exact scaling; RNE */
    if (q > 448.0) q = 448.0;
    if (q == 0.0) return sign;
    int qe;
    frexp(q, &qe);
    qe -= 1;
    if (qe < -6) { /* subnormal: m * 2^-9 */
        int m = (int)(q / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int m = (int)(q / ldexp(1.0, qe - 3)) - 8;
    return sign | (uint8_t)((qe + 7) << 3) | (uint8_t)m;
}

/* e8m0 scale code for a block with max magnitude amax: X = 2^(floor(log2 amax) - 8),
 * 8 being the exponent of E4M3's largest normal; amax == 0 takes X = 2^-127. */
static uint8_t mx_scale_code(double amax) {
    if (amax == 0.0) return 0;
    int e;
    frexp(amax, &e);
    int se = (e - 1) - 8;
    if (se < -127) se = -127;
    if (se > 127) se = 127;
    return (uint8_t)(se + 127);
}

/* Quantise rows x K values (K multiple of 32) in blocks of 32 along K:
 * q[r, c] = E4M3(v[r, c] / X_b), s[r, c/32] = code of X_b. */
void oracle_mx_quantize_f64(const double *v, int64_t rows, int64_t K, uint8_t *q, uint8_t *s) {
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const double *blk = v + r * K + b * 32;
            double amax = 0;
            for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(blk[i]));
            uint8_t code = mx_scale_code(amax);
            s[r * nb + b] = code;
            double X = ldexp(1.0, (int)code - 127);
            for (int i = 0; i < 32; ++i)
                q[r * K + b * 32 + i] = (amax == 0.0) ? 0 : oracle_e4m3_encode(blk[i] / X);
        }
    }
}

void oracle_mx_quantize_bf16(const uint16_t *v, int64_t rows, int64_t K, uint8_t *q, uint8_t *s) {
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double blk[32];
        for (int64_t b = 0; b < nb; ++b) {
            double amax = 0;
            for (int i = 0; i < 32; ++i) {
                blk[i] = bf(v[r * K + b * 32 + i]);
                amax = fmax(amax, fabs(blk[i]));
            }
            uint8_t code = mx_scale_code(amax);
            s[r * nb + b] = code;
            double X = ldexp(1.0, (int)code - 127);
            for (int i = 0; i < 32; ++i)
                q[r * K + b * 32 + i] = (amax == 0.0) ? 0 : oracle_e4m3_encode(blk[i] / X);
        }
    }
}

void oracle_mx_dequantize(const uint8_t *q, const uint8_t *s, int64_t rows, int64_t K, double *out) {
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < K; ++c)
            out[r * K + c] = oracle_e4m3_value(q[r * K + c]) * ldexp(1.0, (int)s[r * nb + c / 32] - 127);
}

/* in-place: v <- dequant(quant(v)) over one vector of n (multiple of 32) values */
static void mx_roundtrip(double *v, int64_t n) {
    for (int64_t b = 0; b < n / 32; ++b) {
        double *blk = v + b * 32;
        double amax = 0;
        for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(blk[i]));
        uint8_t code = mx_scale_code(amax);
        double X = ldexp(1.0, (int)code - 127);
        for (int i = 0; i < 32; ++i)
            blk[i] = (amax == 0.0) ? 0.0 : oracle_e4m3_value(oracle_e4m3_encode(blk[i] / X)) * X;
    }
}

/* dot of an MX row (codes q, scales s, n values) with an fp64 vector */
static double dot_mx(const uint8_t *q, const uint8_t *s, const double *v, int64_t n) {
    double acc = 0;
    for (int64_t b = 0; b < n / 32; ++b) {
        double X = ldexp(1.0, (int)s[b] - 127);
        double a0 = 0, a1 = 0;
        for (int i = 0; i < 32; i += 2) {
            a0 += oracle_e4m3_value(q[b * 32 + i]) * X * v[b * 32 + i];
            a1 += oracle_e4m3_value(q[b * 32 + i + 1]) * X * v[b * 32 + i + 1];
        }
        acc += a0 + a1;
    }
    return acc;
}

/* ------------------------------------------------------------------ router */

/* logits[i, e] = x[row_i] . W_r[e] + beta[e] (beta may be NULL).  rows_of
 * lists the x rows to use (NULL: rows 0..n-1). */
void oracle_router_logits(const uint16_t *x, int64_t D, const int64_t *rows_of, int64_t n,
                          const uint16_t *Wr, const float *beta, int64_t E, double *logits) {
#pragma omp parallel
    {
        double *xv = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < n; ++i) {
            int64_t t = rows_of ? rows_of[i] : i;
            for (int64_t d = 0; d < D; ++d) xv[d] = bf(x[t * D + d]);
            for (int64_t e = 0; e < E; ++e)
                logits[i * E + e] = dot_bf16(Wr + e * D, xv, D) + (beta ? (double)beta[e] : 0.0);
        }
        free(xv);
    }
}

typedef struct { double s; int e; } scored_t;

static int by_score_then_id(const void *a, const void *b) {
    const scored_t *p = (const scored_t *)a, *q = (const scored_t *)b;
    if (p->s > q->s) return -1;
    if (p->s < q->s) return 1;
    return (p->e > q->e) - (p->e < q->e);
}

static int by_int(const void *a, const void *b) {
    int p = *(const int *)a, q = *(const int *)b;
    return (p > q) - (p < q);
}

/* scores from logits, top-k by full sort, slot order, normalised weights.
 * work holds E scored_t entries. */
static void score_select(const double *logit, int64_t E, int64_t k, int score_fn,
                         scored_t *work, int32_t *idx, double *g) {
    if (score_fn == SCORE_SOFTMAX) {
        double m = logit[0];
        for (int64_t e = 1; e < E; ++e) m = fmax(m, logit[e]);
        double z = 0;
        for (int64_t e = 0; e < E; ++e) z += exp(logit[e] - m);
        for (int64_t e = 0; e < E; ++e) { work[e].s = exp(logit[e] - m) / z; work[e].e = (int)e; }
    } else {
        for (int64_t e = 0; e < E; ++e) { work[e].s = 1.0 / (1.0 + exp(-logit[e])); work[e].e = (int)e; }
    }
    qsort(work, (size_t)E, sizeof(scored_t), by_score_then_id);
    int sel[64];
    double ssel[64];
    for (int64_t j = 0; j < k; ++j) sel[j] = work[j].e;
    qsort(sel, (size_t)k, sizeof(int), by_int); /* slot order: ascending expert id */
    double sum = 0;
    for (int64_t j = 0; j < k; ++j) {
        /* score of expert sel[j] */
        double sj = 0;
        for (int64_t q = 0; q < k; ++q)
            if (work[q].e == sel[j]) sj = work[q].s;
        ssel[j] = sj;
        sum += sj;
    }
    for (int64_t j = 0; j < k; ++j) {
        idx[j] = sel[j];
        g[j] = ssel[j] / sum;
    }
}

/* top-k and g for n tokens from precomputed (biased) logits [n, E] */
int oracle_topk(const double *logits, int64_t n, int64_t E, int64_t k, int score_fn,
                int32_t *idx, double *g) {
    if (k < 1 || k > 64 || k > E) return -1;
#pragma omp parallel
    {
        scored_t *work = (scored_t *)malloc(sizeof(scored_t) * E);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < n; ++i)
            score_select(logits + i * E, E, k, score_fn, work, idx + i * k, g + i * k);
        free(work);
    }
    return 0;
}

/* ------------------------------------------------------------------ layer forward */

typedef struct {
    int64_t D, I, E, k, I_s;
    int score_fn;
    const uint16_t *x;      /* [*, D] */
    const uint16_t *Wr;     /* [E, D] */
    const float *beta;      /* [E] or NULL */
    /* bf16 experts (mx == 0) */
    const uint16_t *Wup, *Wgate, *Wdown; /* [E,I,D], [E,I,D], [E,D,I] */
    /* MXFP8 experts (mx == 1): codes and e8m0 scales, blocks of 32 along the contraction dim */
    const uint8_t *Wup_q, *Wup_s, *Wgate_q, *Wgate_s, *Wdown_q, *Wdown_s;
    int mx;
    const uint16_t *Ws_up, *Ws_gate, *Ws_down; /* [I_s,D], [I_s,D], [D,I_s] or NULL */
} oracle_layer_t;

/* y[D] = f(x) for one expert of the layer (bf16 or MX weights) */
static void expert_ffn(const oracle_layer_t *L, int e, const double *xv, double *u, double *v,
                       double *h, double *y) {
    const int64_t D = L->D, I = L->I;
    if (!L->mx) {
        const uint16_t *Wu = L->Wup + (int64_t)e * I * D, *Wg = L->Wgate + (int64_t)e * I * D;
        const uint16_t *Wd = L->Wdown + (int64_t)e * D * I;
        for (int64_t i = 0; i < I; ++i) {
            u[i] = dot_bf16(Wu + i * D, xv, D);
            v[i] = dot_bf16(Wg + i * D, xv, D);
            h[i] = silu(v[i]) * u[i];
        }
        for (int64_t d = 0; d < D; ++d) y[d] = dot_bf16(Wd + d * I, h, I);
    } else {
        const int64_t nbD = D / 32, nbI = I / 32;
        for (int64_t i = 0; i < I; ++i) {
            int64_t r = (int64_t)e * I + i;
            u[i] = dot_mx(L->Wup_q + r * D, L->Wup_s + r * nbD, xv, D);
            v[i] = dot_mx(L->Wgate_q + r * D, L->Wgate_s + r * nbD, xv, D);
            h[i] = silu(v[i]) * u[i];
        }
        mx_roundtrip(h, I); /* the gated activation is quantised before the down projection */
        for (int64_t d = 0; d < D; ++d) {
            int64_t r = (int64_t)e * D + d;
            y[d] = dot_mx(L->Wdown_q + r * I, L->Wdown_s + r * nbI, h, I);
        }
    }
}

static void shared_ffn(const oracle_layer_t *L, const double *xv, double *u, double *v, double *h,
                       double *y) {
    const int64_t D = L->D, I = L->I_s;
    for (int64_t i = 0; i < I; ++i) {
        u[i] = dot_bf16(L->Ws_up + i * D, xv, D);
        v[i] = dot_bf16(L->Ws_gate + i * D, xv, D);
        h[i] = silu(v[i]) * u[i];
    }
    for (int64_t d = 0; d < D; ++d) y[d] = dot_bf16(L->Ws_down + d * I, h, I);
}

/* Forward for the tokens rows_of[0..n) (NULL: 0..n-1).  Outputs per listed
 * token: out [n, D], idx [n, k], g [n, k] (idx/g may be NULL). */
int oracle_moe_fwd(const oracle_layer_t *L, const int64_t *rows_of, int64_t n, double *out,
                   int32_t *idx_out, double *g_out) {
    const int64_t D = L->D, I = L->I, E = L->E, k = L->k, I_s = L->I_s;
    if (k < 1 || k > 64 || k > E) return -1;
    if (L->mx && (D % 32 || I % 32)) return -2;
    const int64_t Imax = I > I_s ? I : I_s;
    int has_shared = (I_s > 0 && L->Ws_up && L->Ws_gate && L->Ws_down);
#pragma omp parallel
    {
        double *xv = (double *)malloc(sizeof(double) * D);
        double *xq = (double *)malloc(sizeof(double) * D);
        double *logit = (double *)malloc(sizeof(double) * E);
        scored_t *work = (scored_t *)malloc(sizeof(scored_t) * E);
        double *u = (double *)malloc(sizeof(double) * Imax);
        double *v = (double *)malloc(sizeof(double) * Imax);
        double *h = (double *)malloc(sizeof(double) * Imax);
        double *y = (double *)malloc(sizeof(double) * D);
        int32_t sel[64];
        double g[64];
#pragma omp for schedule(dynamic, 1)
        for (int64_t ti = 0; ti < n; ++ti) {
            int64_t t = rows_of ? rows_of[ti] : ti;
            for (int64_t d = 0; d < D; ++d) xv[d] = bf(L->x[t * D + d]);
            /* 1. router logits (+ bias); 2.-4. scores, top-k, g */
            for (int64_t e = 0; e < E; ++e)
                logit[e] = dot_bf16(L->Wr + e * D, xv, D) + (L->beta ? (double)L->beta[e] : 0.0);
            score_select(logit, E, k, L->score_fn, work, sel, g);
            /* 5.-6. experts and weighted sum; the shared expert first */
            double *o = out + ti * D;
            if (has_shared) {
                shared_ffn(L, xv, u, v, h, y);
                for (int64_t d = 0; d < D; ++d) o[d] = y[d];
            } else {
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            }
            const double *xin = xv;
            if (L->mx) { /* routed experts see the MX-quantised token */
                memcpy(xq, xv, sizeof(double) * D);
                mx_roundtrip(xq, D);
                xin = xq;
            }
            for (int64_t j = 0; j < k; ++j) {
                expert_ffn(L, sel[j], xin, u, v, h, y);
                for (int64_t d = 0; d < D; ++d) o[d] += g[j] * y[d];
            }
            if (idx_out) for (int64_t j = 0; j < k; ++j) idx_out[ti * k + j] = sel[j];
            if (g_out) for (int64_t j = 0; j < k; ++j) g_out[ti * k + j] = g[j];
        }
        free(xv); free(xq); free(logit); free(work); free(u); free(v); free(h); free(y);
    }
    return 0;
}

/* ------------------------------------------------------------------ schedule */

/* Algorithm 1 (pull-based dispatch schedule construction) with a single rank
 * (R = 1, c = 0, L = E), routes A_j = topk_idx[j], j = t*k + slot:
 *   M_l   = |{j : A_j = l}|
 *   S_l   = sum_{l' < l} M_l'
 *   o     = |{j' < j : A_j' = A_j}|   (counted with one running counter per expert)
 *   p     = min(M_l, o) + |{r' < 0 : ...}| = o
 *   Phi_{S_l + p} = j
 * Table row P = S_l + p holds {src_index = t, expert = l, dst_index = j}; the
 * inverse route_row[j] = P.  S has E + 1 entries (S_E = T*k).
 * Returns -1 if an index is out of range. */
int oracle_schedule(const int32_t *topk_idx, int64_t T, int64_t k, int64_t E, int32_t *M,
                    int32_t *S, int32_t *sched, int32_t *route_row) {
    const int64_t R = T * k;
    for (int64_t l = 0; l < E; ++l) M[l] = 0;
    for (int64_t j = 0; j < R; ++j) {
        int32_t a = topk_idx[j];
        if (a < 0 || a >= E) return -1;
        M[a] += 1;
    }
    S[0] = 0;
    for (int64_t l = 0; l < E; ++l) S[l + 1] = S[l] + M[l];
    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t j = 0; j < R; ++j) {
        int32_t l = topk_idx[j];
        int32_t o = seen[l]++;
        int32_t p = o; /* min(M_l, o) with o < M_l */
        int64_t P = (int64_t)S[l] + p;
        sched[P * 3 + 0] = (int32_t)(j / k);
        sched[P * 3 + 1] = l;
        sched[P * 3 + 2] = (int32_t)j;
        route_row[j] = (int32_t)P;
    }
    free(seen);
    return 0;
}
