/*
 * oracle.h -- C interface of the CPU oracle (test infrastructure only; see oracle.c).
 * Nothing here is shared with the CUDA library.
 */
#ifndef FARSKIP_ORACLE_H
#define FARSKIP_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of the arrays handed in */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };
/* storage rounding applied to the tensors a layer writes out */
enum { ORACLE_EXACT = 0, ORACLE_STORE_BF16 = 1, ORACLE_STORE_F32 = 2 };
/* gate rules s() */
enum { ORACLE_GATE_SOFTMAX = 0, ORACLE_GATE_SOFTMAX_RENORM = 1,
       ORACLE_GATE_SIGMOID = 2, ORACLE_GATE_SIGMOID_NORM = 3 };
/* input wiring of block k+1 */
enum { ORACLE_WIRE_PARTIAL = 0, ORACLE_WIRE_OUTDATED = 1, ORACLE_WIRE_DISABLED = 2,
       ORACLE_WIRE_ATTN_FARSKIP = 3, ORACLE_WIRE_ATTN_PLAIN = 4 };

typedef struct {
    int d, E, k, c;          /* model dim, routed experts, top-k, expert width */
    int n_shared, c_shared;  /* shared experts and their width (n_shared may be 0) */
    int gate;                /* ORACLE_GATE_* */
    int in_dtype;            /* element type of the weights: ORACLE_F32 / BF16 / F64 */
    int storage;             /* ORACLE_EXACT / STORE_BF16 / STORE_F32 */
    int fp8;                 /* expert GEMM operands in FP8 E4M3: 1 with per-row scales, 2 with one scale
                                per block of 32 along the contraction (MX); see oracle.c */
} oracle_cfg;

typedef struct {
    const void* w_r;   /* [E, d] router */
    const float* bias; /* [E] or NULL */
    const void* w1;    /* [E, c, d] up   (W1 in the page's MLP equation) */
    const void* w2;    /* [E, c, d] gate (W2, under g = SiLU) */
    const void* w3;    /* [E, d, c] down */
    const void* w1s;   /* [n_shared, c_shared, d] */
    const void* w2s;   /* [n_shared, c_shared, d] */
    const void* w3s;   /* [n_shared, d, c_shared] */
    const void* w_att; /* [d, d] stand-in attention A(a) = a W_att^T (attention wirings), or NULL */
} oracle_weights;

double oracle_round(double x, int storage);
double oracle_e4m3(double x);
int oracle_e4m3_array(int64_t n, const double* x, double* out, uint8_t* codes);
int oracle_quant_rows(int rows, int cols, const void* x, int x_dtype,
                      uint8_t* codes, int32_t* exps, double* deq);
int oracle_quant_blocks(int rows, int cols, int blk, const void* x, int x_dtype,
                        uint8_t* codes, int32_t* exps, double* deq);
int oracle_router(const oracle_cfg* cfg, int n_tok, const void* u, int u_dtype,
                  const void* w_r, const float* bias,
                  double* logits, int32_t* topk_idx, double* topk_w);
int oracle_expert_rows(const oracle_cfg* cfg, int n_rows, const void* a, int a_dtype,
                       const int32_t* expert, const void* w1, const void* w2, const void* w3,
                       double* h_out, double* y_out);
int oracle_block(const oracle_cfg* cfg, const oracle_weights* wts, int n_tok,
                 const double* u, const double* o_prev, const double* extra, int out_storage,
                 double* o_star, double* o_full,
                 int32_t* topk_idx, double* topk_w, double* logits,
                 double* R_out, double* S_out);
int oracle_stack(const oracle_cfg* cfg, const oracle_weights* wts, int L, int wiring,
                 int n_tok, const void* x, int x_dtype,
                 double* o_last, double* o_last_star,
                 int32_t* topk_idx_all, double* topk_w_all, double* logits_all,
                 double* R_all, double* S_all, double* U_all, double* P_all,
                 double* O_all, double* OS_all, double* A_all);
int oracle_attn_standin(const oracle_cfg* cfg, int n_tok, const double* a, const void* w_att, double* out);
int oracle_dispatch(int T, int k, int E, const int32_t* topk_idx,
                    int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src);
int oracle_combine(int T, int k, int d, int in_dtype, int storage,
                   const void* y_perm, const int32_t* pos, const float* topk_w,
                   const void* o_prev, const void* shared_out,
                   double* o_star, double* o_full);
int oracle_block_backward(const oracle_cfg* cfg, const oracle_weights* wts, int n_tok,
                          const double* u, const double* dO, const double* dOs,
                          double* du, double* do_prev, double* dw_out,
                          double* dW_R, double* dW1, double* dW2, double* dW3,
                          double* dW1s, double* dW2s, double* dW3s);
int oracle_stack_backward(const oracle_cfg* cfg, const oracle_weights* wts, int L, int wiring,
                          int n_tok, const void* x, int x_dtype, const double* dOL, const double* dOLs,
                          double* dx, double* dW_R, double* dW1, double* dW2, double* dW3,
                          double* dW1s, double* dW2s, double* dW3s);
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
