/*
 * CPU oracle for the routed-expert MoE FFN layer -- TEST INFRASTRUCTURE ONLY.
 * Plain fp64 C; see oracle.h for the sources and the readings it takes.
 * Build with contraction off (-ffp-contract=off): the fp32 routing and
 * quantisation steps below are specified operation by operation.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))
#define QBLOCK 128

/* ------------------------------------------------------------------------
 * E4M3FN codec.  The format is the public OCP 8-bit float "E4M3FN" named by
 * the FP8 GEMV section of [HYB]: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent 0 encodes subnormals m/8 * 2^-6; the single
 * code S.1111.111 is NaN; there are no infinities; the largest finite
 * magnitude is 1.75 * 2^8 = 448.
 * ---------------------------------------------------------------------- */
ORACLE_API double oracle_e4m3_decode(uint8_t code) {
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round to the nearest E4M3FN value, ties to even mantissa, finite values
 * beyond the range saturate to +-448, NaN maps to the NaN code. */
ORACLE_API uint8_t oracle_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: spacing 2^-9; nearbyint rounds half to even */
        double m = nearbyint(a * 512.0);           /* 0..8, exact scaling */
        return sign | (uint8_t)m;                  /* m = 8 is code 8 = 2^-6 */
    }
    int ex;
    frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                /* a / 2^E in [1, 2)          */
    double m = nearbyint((ldexp(a, -E) - 1.0) * 8.0);
    if (m == 8.0) { E += 1; m = 0.0; }
    int code = ((E + 7) << 3) | (int)m;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* ------------------------------------------------------------------------
 * exp for the gate weights, in fp32, one fixed operation sequence.
 * Method: Cody & Waite argument reduction (x = n ln2 + r, ln2 split into a
 * short head that makes n*head exact and a tail), a degree-7 Taylor
 * polynomial for e^r on |r| <= ln2/2 evaluated by Horner's rule with fused
 * multiply-adds, and an exact scaling by 2^n.  Arguments below -86 return 0
 * (e^-86 ~ 4e-38 is below every weight that matters and keeps 2^n normal).
 * ---------------------------------------------------------------------- */
ORACLE_API float oracle_exp32(float x) {
    const float log2e  = (float)1.4426950408889634;
    const float ln2_hi = 0x1.62e4p-1f;                              /* 15 significant bits */
    const float ln2_lo = (float)(0.69314718055994530942 - 0.693145751953125);
    const float c2 = (float)(1.0 / 2.0),    c3 = (float)(1.0 / 6.0);
    const float c4 = (float)(1.0 / 24.0),   c5 = (float)(1.0 / 120.0);
    const float c6 = (float)(1.0 / 720.0),  c7 = (float)(1.0 / 5040.0);
    if (!(x >= -86.0f)) return 0.0f;
    if (x > 88.0f) return INFINITY;
    float t = x * log2e;
    float n = nearbyintf(t);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ni = (int)n;                              /* -124 <= ni <= 127 */
    uint32_t bits = (uint32_t)(ni + 127) << 23;   /* 2^ni, a normal float */
    float two_n;
    memcpy(&two_n, &bits, 4);
    return p * two_n;
}

/* ------------------------------------------------------------------------
 * Activation quantisation, 1 x 128 (reading of the FP8 GEMV section of
 * [HYB]: the weight format's 128-element input blocks, applied to the
 * activation side as well so that both GEMM operands are E4M3FN).
 * For each group of 128 consecutive values:
 *   amax = max |v|;  s = amax / 448 (fp32), or 1 when amax = 0;
 *   q_i  = E4M3FN(fp32(v_i / s)).
 * n must be a multiple of 128; s has n/128 entries.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_quant_1x128(const float* v, int32_t n, uint8_t* q, float* s) {
    for (int32_t g = 0; g < n / QBLOCK; ++g) {
        const float* vg = v + (int64_t)g * QBLOCK;
        float amax = 0.0f;
        for (int i = 0; i < QBLOCK; ++i) {
            float a = fabsf(vg[i]);
            if (a > amax) amax = a;
        }
        float sc = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        s[g] = sc;
        for (int i = 0; i < QBLOCK; ++i) {
            float ratio = vg[i] / sc;
            q[(int64_t)g * QBLOCK + i] = oracle_e4m3_encode(ratio);
        }
    }
}

static inline double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> bf16 bits, one rounding to nearest even (finite inputs). */
static uint16_t double_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    int ex;
    frexp(a, &ex);
    int E = ex - 1;                         /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;                 /* bf16 subnormal spacing 2^-133 */
    double ulp = ldexp(1.0, E - 7);
    double r = nearbyint(a / ulp) * ulp;    /* exact: a/ulp < 2^8 * 2 */
    float f = (float)r;                     /* r is a bf16 value: exact */
    uint32_t u;
    memcpy(&u, &f, 4);
    if (f > 3.3895313892515355e38f) u = 0x7F800000u;  /* overflow -> inf */
    uint16_t out = (uint16_t)(u >> 16);
    return signbit(v) ? (uint16_t)(out | 0x8000) : out;
}

/* ------------------------------------------------------------------------
 * Router logits ([KT] section 1.2: a router assigns each token to experts).
 *   L[t][e] = sum_h x[t][h] * W[e][h] + b[e]
 * accumulated in fp64 and rounded to fp32 once.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_logits(const uint16_t* x, const float* W, const float* b,
                              int32_t T, int32_t H, int32_t E, int32_t n_threads, float* L) {
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
    #pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int32_t h = 0; h < H; ++h)
                acc += bf16_to_double(x[(int64_t)t * H + h]) * (double)W[(int64_t)e * H + h];
            if (b) acc += (double)b[e];
            L[(int64_t)t * E + e] = (float)acc;
        }
    }
    (void)n_threads;
}

/* ------------------------------------------------------------------------
 * Gating and sorting ([HYB] SmallEP section, Fig. 5: gating and sorting
 * precede dispatch; [KT] section 2.2: tokens of one expert are grouped).
 *
 * Per token t (fp32 logits L[t][0..E-1]):
 *   1. order experts by (L desc, index asc) -- -0 equals +0, so the index
 *      decides -- and keep the first k as ids[t][0..k-1];
 *   2. m = L[ids0]; e_j = exp32(L[ids_j] - m); S = (((e_0 + e_1) + e_2) ...);
 *      w_j = e_j / S, every step an fp32 operation rounded to nearest.
 *      (Equal to a softmax over all E experts renormalised over the
 *      selected k: the full denominator cancels.)
 * Grouping by expert:
 *   counts[e] = #{(t,j) : ids[t][j] = e};  offsets = exclusive prefix sum of
 *   counts (E+1 entries); within expert e the rows are the tokens that chose
 *   it in ascending t; sorted_token[row] = t; inv_row[t][j] = row of (t,j).
 * Any output pointer may be NULL.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_route_from_logits(const float* L, int32_t T, int32_t E, int32_t k,
                                         int32_t* ids_out, float* w_out, int32_t* offsets,
                                         int32_t* sorted_token, int32_t* inv_row) {
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * (size_t)k);
    char* taken = (char*)malloc((size_t)E);
    for (int32_t t = 0; t < T; ++t) {
        const float* Lt = L + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int32_t j = 0; j < k; ++j) {          /* selection by repeated max */
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || Lt[e] > Lt[best]) best = e;   /* strict: lower index wins ties */
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        float m = Lt[ids[(int64_t)t * k]];
        float ev[1024];
        float S = 0.0f;
        for (int32_t j = 0; j < k; ++j) {
            float d = Lt[ids[(int64_t)t * k + j]] - m;
            ev[j] = oracle_exp32(d);
            S = (j == 0) ? ev[0] : S + ev[j];
        }
        for (int32_t j = 0; j < k; ++j) {
            float wj = ev[j] / S;
            if (w_out) w_out[(int64_t)t * k + j] = wj;
            if (ids_out) ids_out[(int64_t)t * k + j] = ids[(int64_t)t * k + j];
        }
    }
    int32_t* counts = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    for (int64_t i = 0; i < (int64_t)T * k; ++i) counts[ids[i]]++;
    int32_t* off = (int32_t*)malloc(sizeof(int32_t) * ((size_t)E + 1));
    off[0] = 0;
    for (int32_t e = 0; e < E; ++e) off[e + 1] = off[e] + counts[e];
    if (offsets) memcpy(offsets, off, sizeof(int32_t) * ((size_t)E + 1));
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int32_t t = 0; t < T; ++t)                  /* t-major walk keeps rows ascending */
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = ids[(int64_t)t * k + j];
            int32_t row = off[e] + fill[e]++;
            if (sorted_token) sorted_token[row] = t;
            if (inv_row) inv_row[(int64_t)t * k + j] = row;
        }
    free(fill); free(off); free(counts); free(taken); free(ids);
}

/* ------------------------------------------------------------------------
 * One expert's FFN on one token ([HYB] "CPU fine-grained parallelism":
 * gate and up, then activation and elementwise product, then down).
 *   g_i = sum_h Wg[i][h] a[h],  u_i = sum_h Wu[i][h] a[h]
 *   h_i = SiLU(g_i) * u_i = g_i / (1 + e^-g_i) * u_i
 *   o_j = sum_i Wd[j][i] h~[i]
 * Weights are dequantised by block: W[i][h] = E4M3(q[i][h]) * s[i/128][h/128].
 * Quantised mode: a = E4M3(xq[h]) * sx[h/128] and h~ = E4M3(hq[i]) * sh[i/128]
 * with h rounded to fp32 before its 1x128 quantisation.  Exact mode: a = x
 * and h~ = h in fp64.  Dot products follow the post-scaling order of the FP8
 * GEMV section ([HYB] Fig. 9-10): within one 128-block the products are
 * summed first (exactly, in fp64: every product of two E4M3 values is a
 * short dyadic number), then the block's scales are applied once.
 * ---------------------------------------------------------------------- */
typedef struct {
    const uint8_t *wg, *wu, *wd;
    const float *sg, *su, *sd;
    int32_t H, I;
} expert_view;

static double g_dec[256];     /* decode table, filled once */
static int g_dec_ready = 0;

static void expert_ffn(const expert_view* ev, int exact_act,
                       const uint8_t* xq, const float* sx, const double* xe,
                       const uint8_t* hq_in, const float* sh_in,
                       double* o, double* hbuf, float* h32, uint8_t* hq, float* sh) {
    const int32_t H = ev->H, I = ev->I, HB = H / QBLOCK, IB = I / QBLOCK;
    for (int32_t i = 0; i < I; ++i) {
        const uint8_t* rg = ev->wg + (int64_t)i * H;
        const uint8_t* ru = ev->wu + (int64_t)i * H;
        double g = 0.0, u = 0.0;
        for (int32_t kb = 0; kb < HB; ++kb) {
            double pg = 0.0, pu = 0.0;
            if (exact_act) {
                for (int32_t h = kb * QBLOCK; h < (kb + 1) * QBLOCK; ++h) {
                    pg += g_dec[rg[h]] * xe[h];
                    pu += g_dec[ru[h]] * xe[h];
                }
                g += pg * (double)ev->sg[(int64_t)(i / QBLOCK) * HB + kb];
                u += pu * (double)ev->su[(int64_t)(i / QBLOCK) * HB + kb];
            } else {
                for (int32_t h = kb * QBLOCK; h < (kb + 1) * QBLOCK; ++h) {
                    double a = g_dec[xq[h]];
                    pg += g_dec[rg[h]] * a;
                    pu += g_dec[ru[h]] * a;
                }
                g += pg * ((double)ev->sg[(int64_t)(i / QBLOCK) * HB + kb] * (double)sx[kb]);
                u += pu * ((double)ev->su[(int64_t)(i / QBLOCK) * HB + kb] * (double)sx[kb]);
            }
        }
        double hv = g / (1.0 + exp(-g)) * u;
        hbuf[i] = hv;
        h32[i] = (float)hv;
    }
    if (!exact_act) oracle_quant_1x128(h32, I, hq, sh);
    /* down projection input: the codes just computed, or the caller's */
    const uint8_t* hq_use = hq_in ? hq_in : hq;
    const float* sh_use = hq_in ? sh_in : sh;
    for (int32_t j = 0; j < H; ++j) {
        const uint8_t* rd = ev->wd + (int64_t)j * I;
        double acc = 0.0;
        for (int32_t kb = 0; kb < IB; ++kb) {
            double p = 0.0;
            if (exact_act) {
                for (int32_t i = kb * QBLOCK; i < (kb + 1) * QBLOCK; ++i) p += g_dec[rd[i]] * hbuf[i];
                acc += p * (double)ev->sd[(int64_t)(j / QBLOCK) * IB + kb];
            } else {
                for (int32_t i = kb * QBLOCK; i < (kb + 1) * QBLOCK; ++i) p += g_dec[rd[i]] * g_dec[hq_use[i]];
                acc += p * ((double)ev->sd[(int64_t)(j / QBLOCK) * IB + kb] * (double)sh_use[kb]);
            }
        }
        o[j] = acc;
    }
}

/* ------------------------------------------------------------------------
 * The layer, token by token ([HYB] SmallEP section: expert outputs are
 * returned to their token and reduced with the gate weights; [KT] section
 * 1.2: the shared expert is always active).
 *   y[t] = bf16( o_shared(t) + sum_{j=0..k-1} w[t][j] * o_{ids[t][j]}(t) )
 * summed in fp64 in that order, rounded once to bf16.
 * Routing (ids, w) is an input so the layer can be evaluated under any
 * routing (normally oracle_route_from_logits on some fp32 logits).
 * rows: the tokens to evaluate (NULL = all T); outputs are [n_rows][H].
 *
 * h records, per (token, slot) with slots 0..k-1 the routed experts in rank
 * order and slot k the shared expert, each Imax = max(I, SI) wide:
 *   h32_out/hq_out/sh_out [n_rows][slots][Imax (/128)]  -- the fp32 h, its
 *     E4M3 codes and 1x128 scales as this oracle computes them (optional);
 *   hq_in/sh_in [T][slots][Imax (/128)] -- optional override: the down
 *     projection then consumes these codes instead of its own.  Used to
 *     evaluate the layer under another implementation's h codes where the
 *     fp32 rounding of h sits on an E4M3 rounding boundary and either code
 *     is a correct result (the same idea as routing under given logits).
 * Returns 0, or -1 on a bad argument.
 * ---------------------------------------------------------------------- */
ORACLE_API int oracle_forward_ex(const oracle_layer* L, const uint16_t* x, int32_t T,
                                 const int32_t* ids, const float* w,
                                 const int32_t* rows, int32_t n_rows, int32_t exact_act,
                                 const uint8_t* hq_in, const float* sh_in,
                                 float* h32_out, uint8_t* hq_out, float* sh_out,
                                 int32_t n_threads, uint16_t* y_bf16, double* y64) {
    if (!L || !x || !ids || !w) return -1;
    const int32_t H = L->H, I = L->I, E = L->E, k = L->k, SI = L->SI;
    if (H % QBLOCK || I % QBLOCK || (L->n_shared && SI % QBLOCK) || k < 1 || k > E || E > 1024) return -1;
    if (!g_dec_ready) {
        for (int c = 0; c < 256; ++c) g_dec[c] = oracle_e4m3_decode((uint8_t)c);
        g_dec_ready = 1;
    }
    if (!rows) n_rows = T;
    const int32_t Imax = (L->n_shared && SI > I) ? SI : I;
#ifdef _OPENMP
    if (n_threads <= 0) n_threads = omp_get_max_threads();
    #pragma omp parallel num_threads(n_threads)
#endif
    {
        double* xe = (double*)malloc(sizeof(double) * (size_t)H);
        double* acc = (double*)malloc(sizeof(double) * (size_t)H);
        double* o = (double*)malloc(sizeof(double) * (size_t)H);
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)Imax);
        float* h32 = (float*)malloc(sizeof(float) * (size_t)Imax);
        uint8_t* hq = (uint8_t*)malloc((size_t)Imax);
        float* sh = (float*)malloc(sizeof(float) * (size_t)(Imax / QBLOCK));
        float* xf = (float*)malloc(sizeof(float) * (size_t)H);
        uint8_t* xq = (uint8_t*)malloc((size_t)H);
        float* sx = (float*)malloc(sizeof(float) * (size_t)(H / QBLOCK));
#ifdef _OPENMP
        #pragma omp for schedule(dynamic, 1)
#endif
        for (int32_t r = 0; r < n_rows; ++r) {
            const int32_t t = rows ? rows[r] : r;
            for (int32_t h = 0; h < H; ++h) {
                xe[h] = bf16_to_double(x[(int64_t)t * H + h]);
                xf[h] = (float)xe[h];
            }
            if (!exact_act) oracle_quant_1x128(xf, H, xq, sx);
            for (int32_t h = 0; h < H; ++h) acc[h] = 0.0;
            /* per (token, slot) h records: slots 0..k-1 routed (rank order), slot k shared */
            const int32_t S = k + (L->n_shared ? 1 : 0);
#define SLOT_IN(ptr, tok, slot, len) ((ptr) ? (ptr) + ((int64_t)(tok) * S + (slot)) * (len) : NULL)
#define SLOT_OUT(slot) do { \
                if (h32_out) memcpy(h32_out + ((int64_t)r * S + (slot)) * Imax, h32, sizeof(float) * (size_t)Imax); \
                if (hq_out) memcpy(hq_out + ((int64_t)r * S + (slot)) * Imax, hq, (size_t)Imax); \
                if (sh_out) memcpy(sh_out + ((int64_t)r * S + (slot)) * (Imax / QBLOCK), sh, sizeof(float) * (size_t)(Imax / QBLOCK)); \
            } while (0)
            if (L->n_shared) {
                expert_view sv = {L->sh_gate, L->sh_up, L->sh_down,
                                  L->sh_s_gate, L->sh_s_up, L->sh_s_down, H, SI};
                expert_ffn(&sv, exact_act, xq, sx, xe, SLOT_IN(hq_in, t, k, Imax), SLOT_IN(sh_in, t, k, Imax / QBLOCK),
                           o, hbuf, h32, hq, sh);
                SLOT_OUT(k);
                for (int32_t h = 0; h < H; ++h) acc[h] = o[h];
            }
            for (int32_t j = 0; j < k; ++j) {
                const int32_t e = ids[(int64_t)t * k + j];
                const double wj = (double)w[(int64_t)t * k + j];
                expert_view rv = {
                    L->w_gate + (int64_t)e * I * H, L->w_up + (int64_t)e * I * H,
                    L->w_down + (int64_t)e * H * I,
                    L->s_gate + (int64_t)e * (I / QBLOCK) * (H / QBLOCK),
                    L->s_up + (int64_t)e * (I / QBLOCK) * (H / QBLOCK),
                    L->s_down + (int64_t)e * (H / QBLOCK) * (I / QBLOCK), H, I};
                expert_ffn(&rv, exact_act, xq, sx, xe, SLOT_IN(hq_in, t, j, Imax), SLOT_IN(sh_in, t, j, Imax / QBLOCK),
                           o, hbuf, h32, hq, sh);
                SLOT_OUT(j);
                for (int32_t h = 0; h < H; ++h) acc[h] += wj * o[h];
            }
#undef SLOT_IN
#undef SLOT_OUT
            for (int32_t h = 0; h < H; ++h) {
                if (y64) y64[(int64_t)r * H + h] = acc[h];
                if (y_bf16) y_bf16[(int64_t)r * H + h] = double_to_bf16(acc[h]);
            }
        }
        free(xe); free(acc); free(o); free(hbuf); free(h32); free(hq); free(sh);
        free(xf); free(xq); free(sx);
    }
    (void)n_threads;
    return 0;
}

/* Batch helpers for the tests (elementwise, same definitions as above). */
ORACLE_API void oracle_e4m3_encode_n(const float* v, int64_t n, uint8_t* q) {
    for (int64_t i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(v[i]);
}
ORACLE_API void oracle_e4m3_decode_n(const uint8_t* q, int64_t n, double* v) {
    for (int64_t i = 0; i < n; ++i) v[i] = oracle_e4m3_decode(q[i]);
}
ORACLE_API void oracle_exp32_n(const float* x, int64_t n, float* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp32(x[i]);
}

ORACLE_API int oracle_forward(const oracle_layer* L, const uint16_t* x, int32_t T,
                              const int32_t* ids, const float* w,
                              const int32_t* rows, int32_t n_rows, int32_t exact_act,
                              int32_t n_threads, uint16_t* y_bf16, double* y64) {
    return oracle_forward_ex(L, x, T, ids, w, rows, n_rows, exact_act, NULL, NULL, NULL, NULL, NULL,
                             n_threads, y_bf16, y64);
}

ORACLE_API int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
