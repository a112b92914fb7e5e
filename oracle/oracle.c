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

int oracle_expert_rows(const oracle_cfg* cfg, int n_rows, const void* a, int a_dtype,
                       const int32_t* expert, const void* w1, const void* w2, const void* w3,
                       double* h_out, double* y_out) {
    const int d = cfg->d, c = cfg->c;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int r = 0; r < n_rows; ++r) {
        double* arow = (double*)malloc(sizeof(double) * (size_t)d);
        double* h = (double*)malloc(sizeof(double) * (size_t)c);
        if (!arow || !h) { bad = 1; free(arow); free(h); continue; }
        for (int i = 0; i < d; ++i) arow[i] = elem(a, (size_t)r * d + i, a_dtype);
        size_t e = (size_t)expert[r];
        mlp_row(d, c, arow, w1, e * c * d, w2, e * c * d, w3, e * d * c, cfg->in_dtype,
                cfg->storage, h, y_out + (size_t)r * d);
        for (int i = 0; i < d; ++i) y_out[(size_t)r * d + i] = oracle_round(y_out[(size_t)r * d + i], cfg->storage);
        if (h_out) memcpy(h_out + (size_t)r * c, h, sizeof(double) * (size_t)c);
        free(arow);
        free(h);
    }
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
    const int cmax = c > cs ? c : cs;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < n_tok; ++t) {
        double* h = (double*)malloc(sizeof(double) * (size_t)(cmax > 0 ? cmax : 1));
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        double* R = (double*)calloc((size_t)d, sizeof(double));
        double* S = (double*)calloc((size_t)d, sizeof(double));
        if (!h || !y || !R || !S) { bad = 1; free(h); free(y); free(R); free(S); continue; }
        const double* a = u + (size_t)t * d;
        /* routed experts: Combine = gate-weighted sum of the k expert outputs */
        for (int s = 0; s < k; ++s) {
            size_t e = (size_t)topk_idx[(size_t)t * k + s];
            double w = topk_w[(size_t)t * k + s];
            mlp_row(d, c, a, wts->w1, e * c * d, wts->w2, e * c * d, wts->w3, e * d * c,
                    cfg->in_dtype, cfg->storage, h, y);
            for (int i = 0; i < d; ++i) R[i] += w * oracle_round(y[i], cfg->storage);
        }
        /* shared experts: every token, gate weight 1 */
        for (int sh = 0; sh < ns; ++sh) {
            mlp_row(d, cs, a, wts->w1s, (size_t)sh * cs * d, wts->w2s, (size_t)sh * cs * d,
                    wts->w3s, (size_t)sh * d * cs, cfg->in_dtype, cfg->storage, h, y);
            for (int i = 0; i < d; ++i) S[i] += y[i];
        }
        for (int i = 0; i < d; ++i) {
            double sv = oracle_round(S[i], resid);
            double op = o_prev[(size_t)t * d + i] + (extra ? extra[(size_t)t * d + i] : 0.0);
            o_star[(size_t)t * d + i] = oracle_round(op + sv, out_storage);
            o_full[(size_t)t * d + i] = oracle_round(op + sv + R[i], out_storage);
            if (R_out) R_out[(size_t)t * d + i] = R[i];
            if (S_out) S_out[(size_t)t * d + i] = sv;
        }
        free(h); free(y); free(R); free(S);
    }
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

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
