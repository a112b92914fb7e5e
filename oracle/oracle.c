/*
 * oracle.c -- plain CPU oracle for the FarSkip-Collective MoE layer stack.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct definition
 * that the CUDA library is checked against.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline / reference arm load it; the
 * product path never does.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Everything is accumulated in fp64.  Inputs (activations and weights) are the
 * exact fp32 / bf16 values the GPU receives, widened to fp64 element by
 * element.  No blocking, no fusion, no reordering beyond what the definitions
 * state: every sum is a plain loop in index order.
 *
 * Source of every formula: "FarSkip-Collective: Unhobbling Blocking
 * Communication in Mixture of Experts Models" (papercache.org summary):
 *   - §2.1, MLP equation:   MLP(A) = sigma(A W1^T . g(A W2^T)) W3^T,
 *                           W1, W2 in R^{c x d}, W3 in R^{d x c}
 *   - §2.1, MoE equation:   MoE(A) = sum_j G(A)_j . MLP^j(A),  G(A) = s(A W_R^T)
 *   - §2.1, Dispatch/Combine paragraph: tokens grouped by their expert set,
 *                           a permute, then the matching aggregate-and-sum;
 *                           a shared expert processes every token.
 *   - §3, FarSkip equation: o_k = o_0 + f_1(o_0) + f_2(o_1*) + ... + f_k(o_{k-1}*)
 *   - §3, eq. (8a)/(8b):    o_k* = o_{k-1} ("outdated") or
 *                           o_k* = o_{k-1} + f_k*(o_{k-1}*) ("partial")
 *
 * Readings where the page is silent (each one is listed in the design notes):
 *   - g = SiLU on the W2 (gate) projection, "." = elementwise product,
 *     sigma = identity (the SwiGLU form the named models use).
 *   - s() = top-k on the logits z = u W_R^T + b, descending, ties to the lower
 *     expert index; slot s = rank.  Weights per gate rule (see oracle_router).
 *   - f_k* = the shared-expert part of block k; u_1 = o_0* = o_0 = x.
 *   - Storage: the configurations store activations in bf16 (or fp32) between
 *     steps.  With storage != ORACLE_EXACT the oracle rounds (RNE) exactly the
 *     tensors the layer writes out: the expert hidden h, each routed expert
 *     output y and every block input u_k (k >= 2; the operand of the block's
 *     GEMMs).  The residual stream o_k, o_k* and the shared output S, which is
 *     only ever added into it, are carried in fp32, and the stack outputs
 *     o_L, o_L* are returned at that precision:
 *     storing them in bf16 is the layer's own output rounding, which the
 *     comparison tolerance covers.  All sums stay fp64.
 *   - FP8 experts (cfg->fp8; the pages run inference with FP8 quantisation
 *     and fused MoE kernels but give no format): the operands of the expert
 *     GEMMs are FP8 E4M3 values times one power-of-two scale per row along
 *     the contraction -- per token for the activations (the block input u,
 *     quantised once per token; the stored hidden h, quantised per row after
 *     its storage rounding), per output channel for the weights (rows of W1,
 *     W2 along d, rows of W3 along c).  Because each scale multiplies a whole
 *     row of the contraction it factors out of the sum, so the GEMM is the
 *     plain sum over the dequantised values.  The router, Combine and the
 *     residual stream are unchanged.  The shared experts are quantised as the
 *     one MLP over their concatenated width that they sum to (§2.1).
 *   - Block-scaled FP8 (cfg->fp8 = 2, the MX form): the same, with one
 *     power-of-two scale per block of 32 consecutive elements along the
 *     contraction instead of one per row -- every activation row, hidden row
 *     and weight row is cut into 32-element blocks and each block gets its own
 *     exponent by the same rule.  A block scale still multiplies every term it
 *     covers by the same power of two, so the GEMM is again the plain sum over
 *     the dequantised values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- elements */

static double elem(const void* p, size_t i, int dtype) {
    if (dtype == ORACLE_F64) return ((const double*)p)[i];
    if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
    /* bf16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round x to the nearest value with `sig` significant bits (ties to even),
 * with the binary32 exponent range (min normal 2^-126, overflow at 2^128).
 * sig = 8 gives bf16, sig = 24 gives binary32. */
static double round_sig(double x, int sig) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    (void)frexp(x, &e);            /* x = m * 2^e, 0.5 <= |m| < 1 */
    if (e < -125) e = -125;        /* subnormal range: fixed quantum */
    double q = ldexp(1.0, e - sig);
    double r = nearbyint(x / q) * q; /* default rounding mode: to nearest, ties to even */
    if (fabs(r) >= ldexp(1.0, 128)) return r > 0 ? INFINITY : -INFINITY;
    return r;
}

double oracle_round(double x, int storage) {
    if (storage == ORACLE_STORE_BF16) return round_sig(x, 8);
    if (storage == ORACLE_STORE_F32) return round_sig(x, 24);
    return x;
}

/* ---------------------------------------------------------------- FP8 E4M3 */

/* FP8 E4M3, the "e4m3fn" format of the OCP 8-bit floating-point formats: a
 * sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, and
 * the code S.1111.111 is NaN.  Finite magnitudes: normals (1 + m/8) 2^(E-7)
 * for exponent fields E = 1..15 (m = 0..7, except m = 7 at E = 15), the
 * largest 1.75 * 2^8 = 448; subnormals m 2^-9 for m = 1..7 (E = 0).
 * oracle_e4m3(x): the value of that set nearest to x, ties to the even
 * mantissa; magnitudes above 448 saturate to 448 (a "satfinite" conversion). */
double oracle_e4m3(double x) {
    if (isnan(x)) return x;
    if (isinf(x)) return x < 0 ? -448.0 : 448.0;
    double a = fabs(x);
    if (a == 0.0) return x;
    int e;
    (void)frexp(a, &e);             /* a in [2^(e-1), 2^e) */
    int lead = e - 1;               /* exponent of the leading bit */
    if (lead < -6) lead = -6;       /* below the smallest normal 2^-6 the quantum stays 2^-9 */
    double q = ldexp(1.0, lead - 3);
    double r = nearbyint(a / q) * q; /* ties to even */
    if (r > 448.0) r = 448.0;
    return x < 0 ? -r : r;
}

/* The E4M3 code of a value v from oracle_e4m3. */
static uint8_t e4m3_code(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sgn = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (a < ldexp(1.0, -6)) return sgn | (uint8_t)(a / ldexp(1.0, -9));   /* subnormal or zero */
    int e;
    (void)frexp(a, &e);
    int lead = e - 1;
    int m = (int)((a / ldexp(1.0, lead) - 1.0) * 8.0);
    return sgn | (uint8_t)((lead + 7) << 3) | (uint8_t)m;
}

int oracle_e4m3_array(int64_t n, const double* x, double* out, uint8_t* codes) {
    for (int64_t i = 0; i < n; ++i) {
        double v = oracle_e4m3(x[i]);
        if (out) out[i] = v;
        if (codes) codes[i] = e4m3_code(v);
    }
    return 0;
}

/* Scale of one FP8 operand row: the power of two 2^e with the smallest integer
 * e such that max_i |x_i| 2^-e <= 448, so the row's largest element lands in
 * (224, 448]; e = 0 for a row of zeros. */
static int fp8_row_exp(double amax) {
    if (!(amax > 0.0)) return 0;
    int e;
    (void)frexp(amax, &e);          /* 2^(e-1) <= amax < 2^e, so the answer is e-9 or e-8 */
    int s = e - 10;
    while (amax > ldexp(448.0, s)) ++s;
    return s;
}

/* Quantise one row in place: x_i <- e4m3(x_i 2^-e) 2^e with e = fp8_row_exp(max |x|);
 * returns e and, when codes is set, the E4M3 codes of e4m3(x_i 2^-e). */
static int quant_row(double* x, int n, uint8_t* codes) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i)
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    int e = fp8_row_exp(amax);
    for (int i = 0; i < n; ++i) {
        double v = oracle_e4m3(ldexp(x[i], -e));
        if (codes) codes[i] = e4m3_code(v);
        x[i] = ldexp(v, e);
    }
    return e;
}

/* Elements per block of the MX form. */
#define ORACLE_MX_BLOCK 32

/* Block length of the FP8 operands of cfg along a contraction of length len:
 * the whole row (row scales) or ORACLE_MX_BLOCK (block scales). */
static int fp8_blk(const oracle_cfg* cfg, int len) { return cfg->fp8 == 2 ? ORACLE_MX_BLOCK : len; }

/* Quantise x[n] in place as n / blk consecutive blocks of blk elements, each
 * with its own exponent (quant_row on each block); exps[b] receives block b's
 * exponent, codes its E4M3 codes (either may be NULL).  blk = n is one row
 * scale. */
static void quant_blocks(double* x, int n, int blk, uint8_t* codes, int32_t* exps) {
    for (int b = 0; b < n / blk; ++b) {
        int e = quant_row(x + (size_t)b * blk, blk, codes ? codes + (size_t)b * blk : NULL);
        if (exps) exps[b] = e;
    }
}

int oracle_quant_blocks(int rows, int cols, int blk, const void* x, int x_dtype,
                        uint8_t* codes, int32_t* exps, double* deq) {
    if (rows < 0 || cols <= 0 || blk <= 0 || cols % blk) return -1;
    int bad = 0;
    const int nb = cols / blk;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        double* row = (double*)malloc(sizeof(double) * (size_t)cols);
        if (!row) { bad = 1; continue; }
        for (int i = 0; i < cols; ++i) row[i] = elem(x, (size_t)r * cols + i, x_dtype);
        quant_blocks(row, cols, blk, codes ? codes + (size_t)r * cols : NULL, exps ? exps + (size_t)r * nb : NULL);
        if (deq) memcpy(deq + (size_t)r * cols, row, sizeof(double) * (size_t)cols);
        free(row);
    }
    return bad ? -2 : 0;
}

int oracle_quant_rows(int rows, int cols, const void* x, int x_dtype,
                      uint8_t* codes, int32_t* exps, double* deq) {
    if (rows < 0 || cols <= 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        double* row = (double*)malloc(sizeof(double) * (size_t)cols);
        if (!row) { bad = 1; continue; }
        for (int i = 0; i < cols; ++i) row[i] = elem(x, (size_t)r * cols + i, x_dtype);
        int e = quant_row(row, cols, codes ? codes + (size_t)r * cols : NULL);
        if (exps) exps[r] = e;
        if (deq) memcpy(deq + (size_t)r * cols, row, sizeof(double) * (size_t)cols);
        free(row);
    }
    return bad ? -2 : 0;
}

/* Exponents of `rows` weight rows of length K, one per block of blk elements
 * along K (blk = K: one per row): out[r * (K / blk) + b]. */
static void weight_block_exps(const void* w, int dt, size_t rows, int K, int blk, int32_t* out) {
    const int nb = K / blk;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < (long long)rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int i = b * blk; i < (b + 1) * blk; ++i) {
                double v = fabs(elem(w, (size_t)r * K + i, dt));
                if (v > amax) amax = v;
            }
            out[(size_t)r * nb + b] = fp8_row_exp(amax);
        }
    }
}

/* One weight element quantised with its row's exponent e. */
static double wq_value(double v, int e) { return ldexp(oracle_e4m3(ldexp(v, -e)), e); }

/* Memo of wq_value for bf16 weights: a bf16 element has 65536 possible bit
 * patterns, so for each row exponent e in use the quantised value of every
 * pattern is computed once (wq_value itself) and then looked up.  The values
 * are identical to calling wq_value; only the repeated work per token goes. */
enum { WQ_EMIN = -64, WQ_EMAX = 63 };
static double* g_wq_tab[WQ_EMAX - WQ_EMIN + 1];

static void wq_tables_for(const int32_t* exps, size_t n) {
#pragma omp critical(oracle_wq_tables)
    for (size_t r = 0; r < n; ++r) {
        int e = exps[r];
        if (e < WQ_EMIN || e > WQ_EMAX || g_wq_tab[e - WQ_EMIN]) continue;
        double* t = (double*)malloc(sizeof(double) * 65536);
        if (!t) continue;    /* no memo: wq computes the value directly */
        for (uint32_t b = 0; b < 65536; ++b) {
            uint16_t h = (uint16_t)b;
            t[b] = wq_value(elem(&h, 0, ORACLE_BF16), e);
        }
        g_wq_tab[e - WQ_EMIN] = t;
    }
}

static double wq(const void* w, size_t i, int dt, int e) {
    if (dt == ORACLE_BF16 && e >= WQ_EMIN && e <= WQ_EMAX && g_wq_tab[e - WQ_EMIN])
        return g_wq_tab[e - WQ_EMIN][((const uint16_t*)w)[i]];
    return wq_value(elem(w, i, dt), e);
}

static double silu(double v) { return v / (1.0 + exp(-v)); }
static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* ------------------------------------------------------------------ router */

/* Router for n_tok token rows u[n_tok, d] (dtype u_dtype):
 *   z[t, j] = sum_i u[t, i] W_R[j, i] + b[j]                    (§2.1, G(A) = s(A W_R^T))
 *   top-k of z[t, :]: repeatedly take the largest remaining z, the lower j on ties.
 *   weights for the k chosen experts e_0..e_{k-1}:
 *     ORACLE_GATE_SOFTMAX        w_s = exp(z_{e_s}) / sum_{j<E} exp(z_j)
 *     ORACLE_GATE_SOFTMAX_RENORM w_s = exp(z_{e_s}) / sum_{s'<k} exp(z_{e_s'})
 *     ORACLE_GATE_SIGMOID        w_s = 1 / (1 + exp(-z_{e_s}))
 *     ORACLE_GATE_SIGMOID_NORM   w_s = sigmoid(z_{e_s}) / sum_{s'<k} sigmoid(z_{e_s'})
 */
int oracle_router(const oracle_cfg* cfg, int n_tok, const void* u, int u_dtype,
                  const void* w_r, const float* bias,
                  double* logits, int32_t* topk_idx, double* topk_w) {
    const int d = cfg->d, E = cfg->E, k = cfg->k;
    if (n_tok < 0 || d <= 0 || E <= 0 || k <= 0 || k > E) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 16)
    for (int t = 0; t < n_tok; ++t) {
        double* z = logits + (size_t)t * E;
        for (int j = 0; j < E; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += elem(u, (size_t)t * d + i, u_dtype) * elem(w_r, (size_t)j * d + i, cfg->in_dtype);
            if (bias) acc += (double)bias[j];
            z[j] = acc;
        }
        /* top-k selection */
        char* taken = (char*)calloc((size_t)E, 1);
        if (!taken) { bad = 1; continue; }
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int j = 0; j < E; ++j) {
                if (taken[j]) continue;
                if (best < 0 || z[j] > z[best]) best = j;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + s] = best;
        }
        free(taken);
        /* gate weights */
        const int32_t* e = topk_idx + (size_t)t * k;
        double* w = topk_w + (size_t)t * k;
        double zmax = z[e[0]];      /* the largest logit overall */
        if (cfg->gate == ORACLE_GATE_SOFTMAX) {
            double den = 0.0;
            for (int j = 0; j < E; ++j) den += exp(z[j] - zmax);
            for (int s = 0; s < k; ++s) w[s] = exp(z[e[s]] - zmax) / den;
        } else if (cfg->gate == ORACLE_GATE_SOFTMAX_RENORM) {
            double den = 0.0;
            for (int s = 0; s < k; ++s) den += exp(z[e[s]] - zmax);
            for (int s = 0; s < k; ++s) w[s] = exp(z[e[s]] - zmax) / den;
        } else if (cfg->gate == ORACLE_GATE_SIGMOID) {
            for (int s = 0; s < k; ++s) w[s] = sigmoid(z[e[s]]);
        } else {
            double den = 0.0;
            for (int s = 0; s < k; ++s) den += sigmoid(z[e[s]]);
            for (int s = 0; s < k; ++s) w[s] = sigmoid(z[e[s]]) / den;
        }
    }
    return bad ? -2 : 0;
}

/* --------------------------------------------------------------- expert MLP */

/* One expert on one activation row a[d] (fp64):
 *   h[j] = SiLU(sum_i a[i] W2[j, i]) * (sum_i a[i] W1[j, i]),   j < c    (stored: rounded)
 *   y[i] = sum_j h[j] W3[i, j],                                  i < d    (not rounded here)
 * W1, W2 are [c, d] and W3 is [d, c], row-major, as §2.1 writes them; `base*`
 * are element offsets of this expert inside the weight arrays. */
static void mlp_row(int d, int c, const double* a,
                    const void* w1, size_t base1, const void* w2, size_t base2,
                    const void* w3, size_t base3, int wdt, int storage,
                    double* h, double* y) {
    for (int j = 0; j < c; ++j) {
        double gate = 0.0, up = 0.0;
        for (int i = 0; i < d; ++i) {
            gate += a[i] * elem(w2, base2 + (size_t)j * d + i, wdt);
            up += a[i] * elem(w1, base1 + (size_t)j * d + i, wdt);
        }
        h[j] = oracle_round(silu(gate) * up, storage);
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < c; ++j) acc += h[j] * elem(w3, base3 + (size_t)i * c + j, wdt);
        y[i] = acc;
    }
}

/* The FP8 form of one expert (cfg->fp8 = 1 row scales, 2 block scales).  aq[d]
 * is the token row already quantised (quant_blocks; once per token, shared by
 * all its experts).  The expert has width c made of sub-experts of width cw
 * side by side (cw = c for a routed expert; the shared experts form one MLP
 * over their concatenated width, the TP-slicing identity of §2.1).  Blocks
 * along the contraction are bd elements of d (W1, W2 rows) and bc elements of
 * c (the hidden row and W3 rows); bd = d, bc = c is one scale per row.  W1, W2
 * are [c, d] from element base12, element (j, i) quantised with the exponent
 * of its block, e1 / e2[j (d / bd) + i / bd]; W3 element (i, jj) sits at
 * base3 + (jj / cw) d cw + i cw + jj % cw with exponent e3[i (c / bc) + jj / bc].
 *   gate_j = sum_i aq[i] Wq2[j, i],  up_j = sum_i aq[i] Wq1[j, i]
 *   h_j    = SiLU(gate_j) up_j, rounded per storage (the stored hidden)
 *   hq     = h quantised in blocks of bc (quant_blocks over its c elements)
 *   y_i    = sum_jj hq[jj] Wq3[i, jj]
 * h returns the stored hidden before its quantisation. */
static void mlp_row_fp8(int d, int c, int cw, int bd, int bc, const double* aq,
                        const void* w1, const void* w2, size_t base12, const int32_t* e1, const int32_t* e2,
                        const void* w3, size_t base3, const int32_t* e3, int wdt, int storage,
                        double* h, double* hq, double* y) {
    const size_t nbd = (size_t)(d / bd), nbc = (size_t)(c / bc);
    for (int j = 0; j < c; ++j) {
        double gate = 0.0, up = 0.0;
        for (size_t b = 0; b < nbd; ++b) {          /* i in index order, block by block */
            const int eg = e2[(size_t)j * nbd + b], eu = e1[(size_t)j * nbd + b];
            for (int i = (int)b * bd; i < ((int)b + 1) * bd; ++i) {
                gate += aq[i] * wq(w2, base12 + (size_t)j * d + i, wdt, eg);
                up += aq[i] * wq(w1, base12 + (size_t)j * d + i, wdt, eu);
            }
        }
        h[j] = oracle_round(silu(gate) * up, storage);
        hq[j] = h[j];
    }
    quant_blocks(hq, c, bc, NULL, NULL);
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (size_t b = 0; b < nbc; ++b) {          /* jj in index order, block by block */
            const int ed = e3[(size_t)i * nbc + b];
            for (int jj = (int)b * bc; jj < ((int)b + 1) * bc; ++jj) {
                size_t off = base3 + (size_t)(jj / cw) * d * cw + (size_t)i * cw + (size_t)(jj % cw);
                acc += hq[jj] * wq(w3, off, wdt, ed);
            }
        }
        y[i] = acc;
    }
}

/* Exponents of one block's FP8 expert weights, one per row (row scales) or
 * per block of 32 along the row (block scales): routed W1, W2 rows [E c]
 * (along d) and W3 rows [E d] (along c); the shared experts' gate/up rows
 * [n_s c_s] and the rows of their concatenated down projection [d] (along the
 * n_s c_s concatenated columns).  Each array holds rows x (row length / block). */
typedef struct { int32_t *e1, *e2, *e3, *e1s, *e2s, *e3s; } fp8_exps;

static void fp8_exps_free(fp8_exps* x) {
    free(x->e1); free(x->e2); free(x->e3); free(x->e1s); free(x->e2s); free(x->e3s);
}

static int fp8_exps_make(const oracle_cfg* cfg, const void* w1, const void* w2, const void* w3,
                         const void* w1s, const void* w2s, const void* w3s, fp8_exps* x) {
    const int d = cfg->d, E = cfg->E, c = cfg->c, ns = cfg->n_shared, cs = cfg->c_shared;
    const int wdt = cfg->in_dtype;
    const int bd = fp8_blk(cfg, d), bc = fp8_blk(cfg, c), bcs = fp8_blk(cfg, ns * cs);
    memset(x, 0, sizeof *x);
    if (d % bd || c % bc || (ns > 0 && (ns * cs) % bcs)) return -1;
    const size_t nbd = (size_t)(d / bd), nbc = (size_t)(c / bc);
    x->e1 = (int32_t*)malloc(sizeof(int32_t) * (size_t)E * c * nbd);
    x->e2 = (int32_t*)malloc(sizeof(int32_t) * (size_t)E * c * nbd);
    x->e3 = (int32_t*)malloc(sizeof(int32_t) * (size_t)E * d * nbc);
    if (!x->e1 || !x->e2 || !x->e3) return -2;
    weight_block_exps(w1, wdt, (size_t)E * c, d, bd, x->e1);
    weight_block_exps(w2, wdt, (size_t)E * c, d, bd, x->e2);
    weight_block_exps(w3, wdt, (size_t)E * d, c, bc, x->e3);
    const size_t nbs = ns > 0 ? (size_t)(ns * cs / bcs) : 0;
    if (ns > 0 && w1s) {
        x->e1s = (int32_t*)malloc(sizeof(int32_t) * (size_t)ns * cs * nbd);
        x->e2s = (int32_t*)malloc(sizeof(int32_t) * (size_t)ns * cs * nbd);
        x->e3s = (int32_t*)malloc(sizeof(int32_t) * (size_t)d * nbs);
        if (!x->e1s || !x->e2s || !x->e3s) return -2;
        weight_block_exps(w1s, wdt, (size_t)ns * cs, d, bd, x->e1s);
        weight_block_exps(w2s, wdt, (size_t)ns * cs, d, bd, x->e2s);
        /* row i of the concatenated down projection, column jj = sh c_s + j */
        for (int i = 0; i < d; ++i) {
            for (size_t b = 0; b < nbs; ++b) {
                double amax = 0.0;
                for (int jj = (int)b * bcs; jj < ((int)b + 1) * bcs; ++jj) {
                    const int sh = jj / cs, j = jj % cs;
                    double v = fabs(elem(w3s, (size_t)sh * d * cs + (size_t)i * cs + j, wdt));
                    if (v > amax) amax = v;
                }
                x->e3s[(size_t)i * nbs + b] = fp8_row_exp(amax);
            }
        }
    }
    if (wdt == ORACLE_BF16) {
        wq_tables_for(x->e1, (size_t)E * c * nbd);
        wq_tables_for(x->e2, (size_t)E * c * nbd);
        wq_tables_for(x->e3, (size_t)E * d * nbc);
        if (x->e1s) {
            wq_tables_for(x->e1s, (size_t)ns * cs * nbd);
            wq_tables_for(x->e2s, (size_t)ns * cs * nbd);
            wq_tables_for(x->e3s, (size_t)d * nbs);
        }
    }
    return 0;
}

int oracle_expert_rows(const oracle_cfg* cfg, int n_rows, const void* a, int a_dtype,
                       const int32_t* expert, const void* w1, const void* w2, const void* w3,
                       double* h_out, double* y_out) {
    const int d = cfg->d, c = cfg->c;
    int bad = 0;
    fp8_exps fx;
    memset(&fx, 0, sizeof fx);
    if (cfg->fp8 && fp8_exps_make(cfg, w1, w2, w3, NULL, NULL, NULL, &fx)) {
        fp8_exps_free(&fx);
        return -2;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < n_rows; ++r) {
        double* arow = (double*)malloc(sizeof(double) * (size_t)d);
        double* h = (double*)malloc(sizeof(double) * (size_t)c);
        double* hq = (double*)malloc(sizeof(double) * (size_t)c);
        if (!arow || !h || !hq) { bad = 1; free(arow); free(h); free(hq); continue; }
        for (int i = 0; i < d; ++i) arow[i] = elem(a, (size_t)r * d + i, a_dtype);
        size_t e = (size_t)expert[r];
        if (cfg->fp8) {
            const int bd = fp8_blk(cfg, d), bc = fp8_blk(cfg, c);
            quant_blocks(arow, d, bd, NULL, NULL);
            mlp_row_fp8(d, c, c, bd, bc, arow, w1, w2, e * c * d, fx.e1 + e * c * (d / bd), fx.e2 + e * c * (d / bd),
                        w3, e * d * c, fx.e3 + e * d * (c / bc), cfg->in_dtype, cfg->storage, h, hq,
                        y_out + (size_t)r * d);
        } else {
            mlp_row(d, c, arow, w1, e * c * d, w2, e * c * d, w3, e * d * c, cfg->in_dtype,
                    cfg->storage, h, y_out + (size_t)r * d);
        }
        free(hq);
        for (int i = 0; i < d; ++i) y_out[(size_t)r * d + i] = oracle_round(y_out[(size_t)r * d + i], cfg->storage);
        if (h_out) memcpy(h_out + (size_t)r * c, h, sizeof(double) * (size_t)c);
        free(arow);
        free(h);
    }
    fp8_exps_free(&fx);
    return bad ? -2 : 0;
}

/* ------------------------------------------------------------------- block */

/* Stand-in attention sub-block: a per-token dense map A(a) = a W_att^T,
 * W_att [d, d] (one GEMM, keeping token rows independent).  It stands in for
 * the attention of the attention/MoE wiring of §3; it is not attention. */
int oracle_attn_standin(const oracle_cfg* cfg, int n_tok, const double* a, const void* w_att, double* out) {
    const int d = cfg->d;
    if (!w_att) return -1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < n_tok; ++t) {
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += a[(size_t)t * d + j] * elem(w_att, (size_t)i * d + j, cfg->in_dtype);
            out[(size_t)t * d + i] = acc;
        }
    }
    return 0;
}

/* One FarSkip MoE block for n_tok independent token rows.
 *   u      : block input u_k = o_{k-1}*  [n_tok, d] fp64
 *   o_prev : o_{k-1}                     [n_tok, d] fp64
 *   extra  : a further term added into the residual (the attention output
 *            of the attention wirings), or NULL
 * Computes, per token (§2.1 MoE and shared expert; §3 FarSkip, eq. 8b):
 *   R    = sum_s w_s * y_{e_s}(u)       (y_e stored, so rounded per storage)
 *   S    = sum_i MLP_shared_i(u)        (rounded once, at residual precision)
 *   o*   = o_prev + extra + S           (rounded per out_storage)
 *   o    = o_prev + extra + S + R       (rounded per out_storage)
 */
int oracle_block(const oracle_cfg* cfg, const oracle_weights* wts, int n_tok,
                 const double* u, const double* o_prev, const double* extra, int out_storage,
                 double* o_star, double* o_full,
                 int32_t* topk_idx, double* topk_w, double* logits,
                 double* R_out, double* S_out) {
    const int d = cfg->d, E = cfg->E, k = cfg->k, c = cfg->c;
    const int ns = cfg->n_shared, cs = cfg->c_shared;
    /* S only feeds the residual stream, which is carried in fp32 */
    const int resid = cfg->storage == ORACLE_STORE_BF16 ? ORACLE_STORE_F32 : cfg->storage;
    double* z = logits;
    double* zbuf = NULL;
    if (!z) {
        zbuf = (double*)malloc(sizeof(double) * (size_t)n_tok * E);
        if (!zbuf) return -2;
        z = zbuf;
    }
    int rc = oracle_router(cfg, n_tok, u, ORACLE_F64, wts->w_r, wts->bias, z, topk_idx, topk_w);
    free(zbuf);
    if (rc) return rc;
    int bad = 0;
    fp8_exps fx;
    memset(&fx, 0, sizeof fx);
    if (cfg->fp8 && fp8_exps_make(cfg, wts->w1, wts->w2, wts->w3, wts->w1s, wts->w2s, wts->w3s, &fx)) {
        fp8_exps_free(&fx);
        return -2;
    }
    int cmax = c > cs ? c : cs;
    if (cfg->fp8 && ns * cs > cmax) cmax = ns * cs;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < n_tok; ++t) {
        double* h = (double*)malloc(sizeof(double) * (size_t)(cmax > 0 ? cmax : 1));
        double* hq = (double*)malloc(sizeof(double) * (size_t)(cmax > 0 ? cmax : 1));
        double* aq = (double*)malloc(sizeof(double) * (size_t)d);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        double* R = (double*)calloc((size_t)d, sizeof(double));
        double* S = (double*)calloc((size_t)d, sizeof(double));
        if (!h || !hq || !aq || !y || !R || !S) {
            bad = 1; free(h); free(hq); free(aq); free(y); free(R); free(S); continue;
        }
        const double* a = u + (size_t)t * d;
        if (cfg->fp8) {     /* the token row quantised once for all of its experts */
            memcpy(aq, a, sizeof(double) * (size_t)d);
            quant_blocks(aq, d, fp8_blk(cfg, d), NULL, NULL);
        }
        /* routed experts: Combine = gate-weighted sum of the k expert outputs */
        for (int s = 0; s < k; ++s) {
            size_t e = (size_t)topk_idx[(size_t)t * k + s];
            double w = topk_w[(size_t)t * k + s];
            if (cfg->fp8)
                mlp_row_fp8(d, c, c, fp8_blk(cfg, d), fp8_blk(cfg, c), aq, wts->w1, wts->w2, e * c * d,
                            fx.e1 + e * c * (d / fp8_blk(cfg, d)), fx.e2 + e * c * (d / fp8_blk(cfg, d)),
                            wts->w3, e * d * c, fx.e3 + e * d * (c / fp8_blk(cfg, c)), cfg->in_dtype,
                            cfg->storage, h, hq, y);
            else
                mlp_row(d, c, a, wts->w1, e * c * d, wts->w2, e * c * d, wts->w3, e * d * c,
                        cfg->in_dtype, cfg->storage, h, y);
            for (int i = 0; i < d; ++i) R[i] += w * oracle_round(y[i], cfg->storage);
        }
        /* shared experts: every token, gate weight 1 */
        if (cfg->fp8 && ns > 0) {
            mlp_row_fp8(d, ns * cs, cs, fp8_blk(cfg, d), fp8_blk(cfg, ns * cs), aq, wts->w1s, wts->w2s, 0, fx.e1s,
                        fx.e2s, wts->w3s, 0, fx.e3s, cfg->in_dtype, cfg->storage, h, hq, y);
            for (int i = 0; i < d; ++i) S[i] = y[i];    /* one MLP over the concatenated width */
        } else {
            for (int sh = 0; sh < ns; ++sh) {
                mlp_row(d, cs, a, wts->w1s, (size_t)sh * cs * d, wts->w2s, (size_t)sh * cs * d,
                        wts->w3s, (size_t)sh * d * cs, cfg->in_dtype, cfg->storage, h, y);
                for (int i = 0; i < d; ++i) S[i] += y[i];
            }
        }
        for (int i = 0; i < d; ++i) {
            double sv = oracle_round(S[i], resid);
            double op = o_prev[(size_t)t * d + i] + (extra ? extra[(size_t)t * d + i] : 0.0);
            o_star[(size_t)t * d + i] = oracle_round(op + sv, out_storage);
            o_full[(size_t)t * d + i] = oracle_round(op + sv + R[i], out_storage);
            if (R_out) R_out[(size_t)t * d + i] = R[i];
            if (S_out) S_out[(size_t)t * d + i] = sv;
        }
        free(h); free(hq); free(aq); free(y); free(R); free(S);
    }
    fp8_exps_free(&fx);
    return bad ? -2 : 0;
}

/* ------------------------------------------------------------------- stack */

/* L FarSkip blocks (§3, FarSkip equation and eq. 8a/8b).  With u_k the input of
 * block k (= o_{k-1}* in the page's notation) and o_0 = u_1 = x:
 *   block k produces o_k* = o_{k-1} + S_k and o_k = o_{k-1} + S_k + R_k;
 *   the next input is
 *     ORACLE_WIRE_PARTIAL  : u_{k+1} = o_k*          (eq. 8b, f* = shared expert)
 *     ORACLE_WIRE_OUTDATED : u_{k+1} = o_{k-1}       (eq. 8a)
 *     ORACLE_WIRE_DISABLED : u_{k+1} = o_k           (the plain residual recurrence)
 * Layers with a stand-in attention sub-block A_k (w_att) before the MoE:
 *     ORACLE_WIRE_ATTN_FARSKIP (§3, attention/MoE wiring):
 *         attn-in_k = o_{k-2} + attn-out_{k-1} + shared-out_{k-1}   (partial, 8b)
 *         mlp-in_k  = attn-in_k + routed-out_{k-1} = o_{k-1}         (outdated, 8a)
 *         o_k = o_{k-1} + A_k(attn-in_k) + S_k(mlp-in_k) + R_k(mlp-in_k);
 *         o_k* = o_k - R_k is the next attention input, o_k the next MoE input
 *     ORACLE_WIRE_ATTN_PLAIN (the ordinary layer): h_k = o_{k-1} + A_k(o_{k-1}),
 *         o_k = h_k + S_k(h_k) + R_k(h_k), o_k* = h_k + S_k
 * Storage (when not exact): o_k, o_k* are rounded to fp32 (the residual
 * stream) and u_{k+1} to the storage type; the fp32-storage configuration
 * rounds everything to fp32.
 * Outputs o_L and o_L*; per-block routing, R/S, the block inputs u_k (U_all)
 * and o_{k-1} (P_all) and the block outputs o_k (O_all) and o_k* (OS_all) when
 * the pointers are set ([L, n_tok, ...], block-major); with the attention
 * wirings U_all holds the MoE inputs, A_all the attention inputs, and P_all the
 * residual o_{k-1} entering the layer.  The attention output is carried at
 * residual precision; its input, like every block input, is rounded to the
 * storage type.
 * Token rows are independent, so any subset of the rows of x can be passed. */
int oracle_stack(const oracle_cfg* cfg, const oracle_weights* wts, int L, int wiring,
                 int n_tok, const void* x, int x_dtype,
                 double* o_last, double* o_last_star,
                 int32_t* topk_idx_all, double* topk_w_all, double* logits_all,
                 double* R_all, double* S_all, double* U_all, double* P_all,
                 double* O_all, double* OS_all, double* A_all) {
    const int d = cfg->d, E = cfg->E, k = cfg->k;
    const size_t n = (size_t)n_tok * d;
    if (L < 1 || n_tok < 0) return -1;
    const int attn = wiring == ORACLE_WIRE_ATTN_FARSKIP || wiring == ORACLE_WIRE_ATTN_PLAIN;
    double* x64 = (double*)malloc(sizeof(double) * (n ? n : 1));
    double* ubuf = (double*)malloc(sizeof(double) * (n ? n : 1));
    double* abuf = (double*)malloc(sizeof(double) * (n ? n : 1));   /* attention input */
    double* att = (double*)malloc(sizeof(double) * (n ? n : 1));    /* attention output */
    double* hbuf = (double*)malloc(sizeof(double) * (n ? n : 1));   /* h_k (plain attention layer) */
    double* ring[3];
    double* star[2];
    for (int i = 0; i < 3; ++i) ring[i] = (double*)malloc(sizeof(double) * (n ? n : 1));
    for (int i = 0; i < 2; ++i) star[i] = (double*)malloc(sizeof(double) * (n ? n : 1));
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_tok ? n_tok : 1) * k);
    double* w = (double*)malloc(sizeof(double) * (size_t)(n_tok ? n_tok : 1) * k);
    int rc = 0;
    if (!x64 || !ubuf || !abuf || !att || !hbuf || !ring[0] || !ring[1] || !ring[2] || !star[0] || !star[1] ||
        !idx || !w)
        rc = -2;
    const int resid = cfg->storage == ORACLE_STORE_BF16 ? ORACLE_STORE_F32 : cfg->storage;
    if (!rc) {
        for (size_t i = 0; i < n; ++i) x64[i] = elem(x, i, x_dtype);
        const double* o_km1 = x64;  /* o_{k-1} */
        const double* u = x64;      /* u_k (the MoE input) */
        const double* a_in = x64;   /* attention input (attention wirings) */
        for (int b = 1; b <= L && !rc; ++b) {
            double* o_k = ring[b % 3];
            double* os_k = star[b % 2];
            const oracle_weights* wb = wts + (b - 1);
            const double* extra = NULL;
            const double* base = o_km1;
            if (attn) {
                if (wiring == ORACLE_WIRE_ATTN_PLAIN) {
                    if (b > 1) {
                        for (size_t i = 0; i < n; ++i) abuf[i] = oracle_round(o_km1[i], cfg->storage);
                        a_in = abuf;
                    }
                }
                rc = oracle_attn_standin(cfg, n_tok, a_in, wb->w_att, att);
                if (rc) break;
                for (size_t i = 0; i < n; ++i) att[i] = oracle_round(att[i], resid);
                if (wiring == ORACLE_WIRE_ATTN_PLAIN) {
                    for (size_t i = 0; i < n; ++i) hbuf[i] = oracle_round(o_km1[i] + att[i], resid);
                    for (size_t i = 0; i < n; ++i) ubuf[i] = oracle_round(hbuf[i], cfg->storage);
                    u = ubuf;
                    base = hbuf;
                } else {
                    extra = att;
                }
                if (A_all) memcpy(A_all + (size_t)(b - 1) * n, a_in, sizeof(double) * n);
            }
            if (U_all) memcpy(U_all + (size_t)(b - 1) * n, u, sizeof(double) * n);
            if (P_all) memcpy(P_all + (size_t)(b - 1) * n, o_km1, sizeof(double) * n);
            rc = oracle_block(cfg, wb, n_tok, u, base, extra, resid, os_k, o_k, idx, w,
                              logits_all ? logits_all + (size_t)(b - 1) * n_tok * E : NULL,
                              R_all ? R_all + (size_t)(b - 1) * n : NULL,
                              S_all ? S_all + (size_t)(b - 1) * n : NULL);
            if (topk_idx_all) memcpy(topk_idx_all + (size_t)(b - 1) * n_tok * k, idx, sizeof(int32_t) * (size_t)n_tok * k);
            if (topk_w_all) memcpy(topk_w_all + (size_t)(b - 1) * n_tok * k, w, sizeof(double) * (size_t)n_tok * k);
            if (O_all) memcpy(O_all + (size_t)(b - 1) * n, o_k, sizeof(double) * n);
            if (OS_all) memcpy(OS_all + (size_t)(b - 1) * n, os_k, sizeof(double) * n);
            if (b == L) {
                memcpy(o_last, o_k, sizeof(double) * n);
                memcpy(o_last_star, os_k, sizeof(double) * n);
            }
            if (wiring == ORACLE_WIRE_ATTN_FARSKIP) {
                /* next attention input o_k* = o_k - R_k, next MoE input o_k */
                for (size_t i = 0; i < n; ++i) abuf[i] = oracle_round(os_k[i], cfg->storage);
                for (size_t i = 0; i < n; ++i) ubuf[i] = oracle_round(o_k[i], cfg->storage);
                a_in = abuf;
                u = ubuf;
            } else if (wiring != ORACLE_WIRE_ATTN_PLAIN) {
                const double* nxt;
                if (wiring == ORACLE_WIRE_PARTIAL) nxt = os_k;
                else if (wiring == ORACLE_WIRE_OUTDATED) nxt = o_km1;
                else nxt = o_k;
                for (size_t i = 0; i < n; ++i) ubuf[i] = oracle_round(nxt[i], cfg->storage);
                u = ubuf;
            }
            o_km1 = o_k;
        }
    }
    free(x64);
    free(ubuf);
    free(abuf);
    free(att);
    free(hbuf);
    for (int i = 0; i < 3; ++i) free(ring[i]);
    for (int i = 0; i < 2; ++i) free(star[i]);
    free(idx);
    free(w);
    return rc;
}

/* ---------------------------------------------------------------- dispatch */

/* Local Dispatch (§2.1: tokens grouped by expert, then permuted).  A plain
 * counting sort of the (token, slot) pairs by expert, stable in token order:
 *   counts[e]   = #{(t, s) : idx[t, s] = e}
 *   offsets[e]  = sum_{e' < e} counts[e'],  offsets[E] = T k
 *   pos[t k + s]= the row of (t, s) in the permuted order
 *   perm_src[p] = the token whose row sits at permuted row p
 * Returns -1 if an index is out of range. */
int oracle_dispatch(int T, int k, int E, const int32_t* topk_idx,
                    int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src) {
    if (T < 0 || k <= 0 || E <= 0) return -1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t i = 0; i < (size_t)T * k; ++i) {
        int e = topk_idx[i];
        if (e < 0 || e >= E) return -1;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    if (!cursor) return -2;
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int t = 0; t < T; ++t) {
        for (int s = 0; s < k; ++s) {
            int e = topk_idx[(size_t)t * k + s];
            int p = cursor[e]++;
            pos[(size_t)t * k + s] = p;
            perm_src[p] = t;
        }
    }
    free(cursor);
    return 0;
}

/* ----------------------------------------------------------------- combine */

/* Local Combine fused with the FarSkip update (§2.1 Combine: aggregate and sum
 * the routed outputs; §3 eq. 8b):
 *   R[t]  = sum_{s<k} w[t, s] * y_perm[pos[t, s]]
 *   o*[t] = o_prev[t] + S[t]          (S optional: zero when NULL)
 *   o[t]  = o_prev[t] + S[t] + R[t]
 * y_perm, o_prev and S are given in `in_dtype`; outputs are rounded per storage. */
int oracle_combine(int T, int k, int d, int in_dtype, int storage,
                   const void* y_perm, const int32_t* pos, const float* topk_w,
                   const void* o_prev, const void* shared_out,
                   double* o_star, double* o_full) {
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < d; ++i) {
            double r = 0.0;
            for (int s = 0; s < k; ++s) {
                size_t p = (size_t)pos[(size_t)t * k + s];
                r += (double)topk_w[(size_t)t * k + s] * elem(y_perm, p * d + i, in_dtype);
            }
            double op = elem(o_prev, (size_t)t * d + i, in_dtype);
            double sv = shared_out ? elem(shared_out, (size_t)t * d + i, in_dtype) : 0.0;
            o_star[(size_t)t * d + i] = oracle_round(op + sv, storage);
            o_full[(size_t)t * d + i] = oracle_round(op + sv + r, storage);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- backward */

/* Training form of one block (the pages train FarSkip models with Megatron-LM
 * but print no gradient formulas; these are the derivatives of the forward
 * definitions above).  With storage != ORACLE_EXACT the backward reads what the
 * forward stored -- each expert row's gate/up pre-activations g, a, its hidden
 * h and output y, rounded per storage -- and rounds its own stored operands the
 * same way: the routed output gradient dy = w dR, the pre-activation gradients
 * dg, da, each (token, slot)'s input gradient dx, the shared output gradient
 * dS and the router logit gradient dz.  Sums are fp64.  Top-k selection is
 * piecewise constant (no gradient); the router bias is not a parameter.
 *
 * Per token, with o = o_prev + S + R and o* = o_prev + S:
 *   dR = dO,  dS = dO + dOs,  do_prev = dO + dOs
 *   dw_s = <dR, y_s>,  dy_s = w_s dR
 *   dh   = dy_s W3_e                 dh[j] = sum_i dy[i] W3[i, j]
 *   dg   = dh a SiLU'(g),  da = dh SiLU(g),  SiLU'(g) = sig(g) (1 + g (1 - sig(g)))
 *   dx_s = dg W2_e + da W1_e         dx[i] = sum_j dg[j] W2[j, i] + da[j] W1[j, i]
 *   dW3_e += dy_s h^T,  dW2_e += dg u^T,  dW1_e += da u^T
 *   shared experts: the same with dS for dy and gate weight 1
 *   dz = gate-rule derivative of w applied to dw;  dW_R += dz u^T
 *   du = sum_s dx_s + dx_shared + dz W_R
 */

/* dz[0..E) from dw[0..k) for the gate rules of oracle_router (z = the logits
 * with the bias, e = the chosen experts, w = their gate weights). */
static void gate_backward(int gate, int E, int k, const double* z, const int32_t* e, const double* w,
                          const double* dw, double* dz) {
    for (int j = 0; j < E; ++j) dz[j] = 0.0;
    double c = 0.0;                       /* sum_s dw_s w_s */
    for (int s = 0; s < k; ++s) c += dw[s] * w[s];
    if (gate == ORACLE_GATE_SOFTMAX) {
        /* w_s = p_{e_s}, p = softmax(z) over all E: dz_j = sum_s dw_s p_{e_s} (delta - p_j) */
        double zmax = z[e[0]], den = 0.0;
        for (int j = 0; j < E; ++j) den += exp(z[j] - zmax);
        for (int j = 0; j < E; ++j) dz[j] = -c * exp(z[j] - zmax) / den;
        for (int s = 0; s < k; ++s) dz[e[s]] += dw[s] * w[s];
    } else if (gate == ORACLE_GATE_SOFTMAX_RENORM) {
        /* w_s = softmax over the chosen: dz_{e_r} = w_r (dw_r - c) */
        for (int r = 0; r < k; ++r) dz[e[r]] = w[r] * (dw[r] - c);
    } else if (gate == ORACLE_GATE_SIGMOID) {
        for (int s = 0; s < k; ++s) {
            double sg = sigmoid(z[e[s]]);
            dz[e[s]] = dw[s] * sg * (1.0 - sg);
        }
    } else {
        /* w_s = sig_s / sum_r sig_r: dsig_r = (dw_r - c) / sum, dz_{e_r} = dsig_r sig_r (1 - sig_r) */
        double den = 0.0;
        for (int s = 0; s < k; ++s) den += sigmoid(z[e[s]]);
        for (int r = 0; r < k; ++r) {
            double sg = sigmoid(z[e[r]]);
            dz[e[r]] = (dw[r] - c) / den * sg * (1.0 - sg);
        }
    }
}

static double silu_grad(double g) {
    double sg = sigmoid(g);
    return sg * (1.0 + g * (1.0 - sg));
}

/* One expert row forward and its backward for the row's output gradient dy
 * (already the stored, rounded one): fills g, a (stored), h (stored), y
 * (stored) when fwd, then dh, dg, da (stored) and dx (unrounded).  W1, W2
 * [c, d] from element base12 and W3 element (i, jj) at
 * base3 + (jj / cw) d cw + i cw + jj % cw (cw = c for a routed expert; the
 * shared experts side by side). */
static void mlp_row_fwd(int d, int c, int cw, const double* x, const void* w1, const void* w2, size_t base12,
                        const void* w3, size_t base3, int wdt, int storage, double* g, double* a, double* h,
                        double* y) {
    for (int j = 0; j < c; ++j) {
        double gate = 0.0, up = 0.0;
        for (int i = 0; i < d; ++i) {
            gate += x[i] * elem(w2, base12 + (size_t)j * d + i, wdt);
            up += x[i] * elem(w1, base12 + (size_t)j * d + i, wdt);
        }
        h[j] = oracle_round(silu(gate) * up, storage);
        g[j] = oracle_round(gate, storage);
        a[j] = oracle_round(up, storage);
    }
    if (y) {
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int jj = 0; jj < c; ++jj)
                acc += h[jj] * elem(w3, base3 + (size_t)(jj / cw) * d * cw + (size_t)i * cw + (size_t)(jj % cw), wdt);
            y[i] = oracle_round(acc, storage);
        }
    }
}

static void mlp_row_bwd(int d, int c, int cw, const double* dy, const double* g, const double* a,
                        const void* w1, const void* w2, size_t base12, const void* w3, size_t base3, int wdt,
                        int storage, double* dg, double* da, double* dx) {
    for (int jj = 0; jj < c; ++jj) {
        double dh = 0.0;
        for (int i = 0; i < d; ++i)
            dh += dy[i] * elem(w3, base3 + (size_t)(jj / cw) * d * cw + (size_t)i * cw + (size_t)(jj % cw), wdt);
        dg[jj] = oracle_round(dh * a[jj] * silu_grad(g[jj]), storage);
        da[jj] = oracle_round(dh * silu(g[jj]), storage);
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < c; ++j)
            acc += dg[j] * elem(w2, base12 + (size_t)j * d + i, wdt) + da[j] * elem(w1, base12 + (size_t)j * d + i, wdt);
        dx[i] = acc;
    }
}

int oracle_block_backward(const oracle_cfg* cfg, const oracle_weights* wts, int n_tok,
                          const double* u, const double* dO, const double* dOs,
                          double* du, double* do_prev, double* dw_out,
                          double* dW_R, double* dW1, double* dW2, double* dW3,
                          double* dW1s, double* dW2s, double* dW3s) {
    const int d = cfg->d, E = cfg->E, k = cfg->k, c = cfg->c;
    const int ns = cfg->n_shared, cs = cfg->c_shared, cw = ns * cs;
    const int st = cfg->storage;
    const int wdt = cfg->in_dtype;
    if (cfg->fp8 || n_tok < 0) return -1;
    const size_t nk = (size_t)n_tok * k;
    double* z = (double*)malloc(sizeof(double) * ((size_t)n_tok * E + 1));
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (nk + 1));
    double* w = (double*)malloc(sizeof(double) * (nk + 1));
    /* per (token, slot): dy, h, dg, da; per token: dS, h_s, dg_s, da_s, dz */
    double* r_dy = (double*)malloc(sizeof(double) * (nk * d + 1));
    double* r_h = (double*)malloc(sizeof(double) * (nk * c + 1));
    double* r_dg = (double*)malloc(sizeof(double) * (nk * c + 1));
    double* r_da = (double*)malloc(sizeof(double) * (nk * c + 1));
    double* s_dS = (double*)malloc(sizeof(double) * ((size_t)n_tok * d + 1));
    double* s_h = (double*)malloc(sizeof(double) * ((size_t)n_tok * (cw ? cw : 1)));
    double* s_dg = (double*)malloc(sizeof(double) * ((size_t)n_tok * (cw ? cw : 1)));
    double* s_da = (double*)malloc(sizeof(double) * ((size_t)n_tok * (cw ? cw : 1)));
    double* r_dz = (double*)malloc(sizeof(double) * ((size_t)n_tok * E + 1));
    int rc = 0;
    if (!z || !idx || !w || !r_dy || !r_h || !r_dg || !r_da || !s_dS || !s_h || !s_dg || !s_da || !r_dz) rc = -2;
    if (!rc) rc = oracle_router(cfg, n_tok, u, ORACLE_F64, wts->w_r, wts->bias, z, idx, w);
    int bad = 0;
    if (!rc) {
        const int cmax = c > cw ? c : cw;
#pragma omp parallel for schedule(dynamic, 1)
        for (int t = 0; t < n_tok; ++t) {
            double* g = (double*)malloc(sizeof(double) * (size_t)cmax);
            double* a = (double*)malloc(sizeof(double) * (size_t)cmax);
            double* y = (double*)malloc(sizeof(double) * (size_t)d);
            double* dx = (double*)malloc(sizeof(double) * (size_t)d);
            double* dw = (double*)malloc(sizeof(double) * (size_t)k);
            if (!g || !a || !y || !dx || !dw) { bad = 1; free(g); free(a); free(y); free(dx); free(dw); continue; }
            const double* x = u + (size_t)t * d;
            const double* dR = dO + (size_t)t * d;
            double* dut = du + (size_t)t * d;
            for (int i = 0; i < d; ++i) {
                double dsv = dO[(size_t)t * d + i] + (dOs ? dOs[(size_t)t * d + i] : 0.0);
                do_prev[(size_t)t * d + i] = dsv;
                s_dS[(size_t)t * d + i] = oracle_round(dsv, st);
                dut[i] = 0.0;
            }
            /* routed experts */
            for (int s = 0; s < k; ++s) {
                const size_t ts = (size_t)t * k + s;
                const size_t e = (size_t)idx[ts];
                double* h = r_h + ts * c;
                mlp_row_fwd(d, c, c, x, wts->w1, wts->w2, e * c * d, wts->w3, e * d * c, wdt, st, g, a, h, y);
                double dws = 0.0;
                for (int i = 0; i < d; ++i) dws += dR[i] * y[i];
                dw[s] = dws;
                double* dy = r_dy + ts * d;
                for (int i = 0; i < d; ++i) dy[i] = oracle_round(w[ts] * dR[i], st);
                mlp_row_bwd(d, c, c, dy, g, a, wts->w1, wts->w2, e * c * d, wts->w3, e * d * c, wdt, st,
                            r_dg + ts * c, r_da + ts * c, dx);
                for (int i = 0; i < d; ++i) dut[i] += oracle_round(dx[i], st);
            }
            if (dw_out) memcpy(dw_out + (size_t)t * k, dw, sizeof(double) * (size_t)k);
            /* shared experts: one MLP over the concatenated width */
            if (ns > 0) {
                double* hs = s_h + (size_t)t * cw;
                mlp_row_fwd(d, cw, cs, x, wts->w1s, wts->w2s, 0, wts->w3s, 0, wdt, st, g, a, hs, NULL);
                mlp_row_bwd(d, cw, cs, s_dS + (size_t)t * d, g, a, wts->w1s, wts->w2s, 0, wts->w3s, 0, wdt, st,
                            s_dg + (size_t)t * cw, s_da + (size_t)t * cw, dx);
                for (int i = 0; i < d; ++i) dut[i] += dx[i];
            }
            /* router */
            double* dz = r_dz + (size_t)t * E;
            gate_backward(cfg->gate, E, k, z + (size_t)t * E, idx + (size_t)t * k, w + (size_t)t * k, dw, dz);
            for (int j = 0; j < E; ++j) dz[j] = oracle_round(dz[j], st);
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int j = 0; j < E; ++j) acc += dz[j] * elem(wts->w_r, (size_t)j * d + i, wdt);
                dut[i] += acc;
            }
            free(g); free(a); free(y); free(dx); free(dw);
        }
    }
    if (bad) rc = -2;
    if (!rc && dW1 && dW2 && dW3 && dW_R) {
        /* weight gradients: sums over the (token, slot) pairs routed to each expert */
#pragma omp parallel for schedule(dynamic, 1)
        for (int e = 0; e < E; ++e) {
            for (size_t q = 0; q < (size_t)d * c; ++q) dW3[(size_t)e * d * c + q] = 0.0;
            for (size_t q = 0; q < (size_t)c * d; ++q) {
                dW1[(size_t)e * c * d + q] = 0.0;
                dW2[(size_t)e * c * d + q] = 0.0;
            }
            for (size_t ts = 0; ts < nk; ++ts) {
                if (idx[ts] != e) continue;
                const double* x = u + (ts / k) * d;
                const double* dy = r_dy + ts * d;
                const double* h = r_h + ts * c;
                const double* dg = r_dg + ts * c;
                const double* da = r_da + ts * c;
                for (int i = 0; i < d; ++i)
                    for (int j = 0; j < c; ++j) dW3[((size_t)e * d + i) * c + j] += dy[i] * h[j];
                for (int j = 0; j < c; ++j)
                    for (int i = 0; i < d; ++i) {
                        dW2[((size_t)e * c + j) * d + i] += dg[j] * x[i];
                        dW1[((size_t)e * c + j) * d + i] += da[j] * x[i];
                    }
            }
            for (int i = 0; i < d; ++i) {
                double* row = dW_R + (size_t)e * d;
                row[i] = 0.0;
                for (int t = 0; t < n_tok; ++t) row[i] += r_dz[(size_t)t * E + e] * u[(size_t)t * d + i];
            }
        }
        if (ns > 0 && dW1s && dW2s && dW3s) {
#pragma omp parallel for schedule(static)
            for (int jj = 0; jj < cw; ++jj) {
                const int sh = jj / cs, j = jj % cs;
                for (int i = 0; i < d; ++i) {
                    double a3 = 0.0, a1 = 0.0, a2 = 0.0;
                    for (int t = 0; t < n_tok; ++t) {
                        a3 += s_dS[(size_t)t * d + i] * s_h[(size_t)t * cw + jj];
                        a2 += s_dg[(size_t)t * cw + jj] * u[(size_t)t * d + i];
                        a1 += s_da[(size_t)t * cw + jj] * u[(size_t)t * d + i];
                    }
                    dW3s[((size_t)sh * d + i) * cs + j] = a3;
                    dW2s[((size_t)sh * cs + j) * d + i] = a2;
                    dW1s[((size_t)sh * cs + j) * d + i] = a1;
                }
            }
        }
    }
    free(z); free(idx); free(w); free(r_dy); free(r_h); free(r_dg); free(r_da);
    free(s_dS); free(s_h); free(s_dg); free(s_da); free(r_dz);
    return rc;
}

/* Backward of oracle_stack for the MoE wirings (PARTIAL, OUTDATED, DISABLED):
 * dOL, dOLs are the gradients of o_L and o_L* (dOLs may be NULL).  Blocks are
 * visited from L down to 1; block k's do_prev flows to o_{k-1}, and its du to
 * where u_k came from -- o_{k-1}* (partial), o_{k-2} (outdated) or o_{k-1}
 * (disabled), x for k = 1 -- through the storage rounding of u_k as the
 * identity.  Weight gradients are [L, ...] block-major; with dW_R NULL none
 * are computed (the input gradient alone). */
int oracle_stack_backward(const oracle_cfg* cfg, const oracle_weights* wts, int L, int wiring,
                          int n_tok, const void* x, int x_dtype, const double* dOL, const double* dOLs,
                          double* dx, double* dW_R, double* dW1, double* dW2, double* dW3,
                          double* dW1s, double* dW2s, double* dW3s) {
    const int d = cfg->d, E = cfg->E, k = cfg->k, c = cfg->c, ns = cfg->n_shared, cs = cfg->c_shared;
    if (L < 1 || n_tok < 0) return -1;
    if (wiring != ORACLE_WIRE_PARTIAL && wiring != ORACLE_WIRE_OUTDATED && wiring != ORACLE_WIRE_DISABLED) return -1;
    const size_t n = (size_t)n_tok * d;
    double* U = (double*)malloc(sizeof(double) * (n * L + 1));
    double* oL = (double*)malloc(sizeof(double) * (n + 1));
    double* oLs = (double*)malloc(sizeof(double) * (n + 1));
    double* go = (double*)calloc(n * (L + 1) + 1, sizeof(double));    /* gradients of o_0 .. o_L */
    double* gos = (double*)calloc(n * (L + 1) + 1, sizeof(double));   /* gradients of o_0* .. o_L* */
    double* du = (double*)malloc(sizeof(double) * (n + 1));
    double* dp = (double*)malloc(sizeof(double) * (n + 1));
    int rc = (!U || !oL || !oLs || !go || !gos || !du || !dp) ? -2 : 0;
    if (!rc)
        rc = oracle_stack(cfg, wts, L, wiring, n_tok, x, x_dtype, oL, oLs, NULL, NULL, NULL, NULL, NULL, U, NULL,
                          NULL, NULL, NULL);
    if (!rc) {
        memcpy(go + n * L, dOL, sizeof(double) * n);
        if (dOLs) memcpy(gos + n * L, dOLs, sizeof(double) * n);
        for (size_t i = 0; i < n; ++i) dx[i] = 0.0;
        for (int b = L; b >= 1 && !rc; --b) {
            const size_t wo = (size_t)(b - 1);
            const int gw = dW_R != NULL;    /* weight gradients wanted */
            rc = oracle_block_backward(cfg, wts + (b - 1), n_tok, U + (size_t)(b - 1) * n, go + n * b, gos + n * b,
                                       du, dp, NULL, gw ? dW_R + wo * E * d : NULL, gw ? dW1 + wo * E * c * d : NULL,
                                       gw ? dW2 + wo * E * c * d : NULL, gw ? dW3 + wo * E * d * c : NULL,
                                       gw && ns ? dW1s + wo * ns * cs * d : NULL,
                                       gw && ns ? dW2s + wo * ns * cs * d : NULL,
                                       gw && ns ? dW3s + wo * ns * d * cs : NULL);
            if (rc) break;
            double* g_prev = go + n * (b - 1);                     /* o_{b-1} */
            for (size_t i = 0; i < n; ++i) g_prev[i] += dp[i];
            double* target;
            if (b == 1) target = dx;                               /* u_1 = x */
            else if (wiring == ORACLE_WIRE_PARTIAL) target = gos + n * (b - 1);   /* u_b = o_{b-1}* */
            else if (wiring == ORACLE_WIRE_OUTDATED) target = go + n * (b - 2);   /* u_b = o_{b-2} */
            else target = go + n * (b - 1);                                       /* u_b = o_{b-1} */
            for (size_t i = 0; i < n; ++i) target[i] += du[i];
        }
        for (size_t i = 0; i < n; ++i) dx[i] += go[i];             /* o_0 = x */
    }
    free(U); free(oL); free(oLs); free(go); free(gos); free(du); free(dp);
    return rc;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
