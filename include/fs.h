/*
 * fs.h -- C ABI of libfs, the GB300 (sm_103a) FarSkip-Collective MoE layer library.
 *
 * What is computed ("FarSkip-Collective: Unhobbling Blocking Communication in
 * Mixture of Experts Models", papercache.org summary):
 *   §2.1 MLP equation   MLP(A) = sigma(A W1^T . g(A W2^T)) W3^T, read as
 *                       (SiLU(A W2^T) * (A W1^T)) W3^T  (W1 = up, W2 = gate, W3 = down)
 *   §2.1 MoE equation   MoE(A) = sum_j G(A)_j MLP^j(A),  G(A) = s(A W_R^T)
 *   §2.1 Dispatch / Combine: on one GPU a local stable permutation of token rows
 *                       by expert and the gate-weighted sum back to token order;
 *                       a shared expert processes every token
 *   §3 FarSkip equation o_k = o_0 + f_1(o_0) + f_2(o_1*) + ... + f_k(o_{k-1}*)
 *   §3 eq. (8a)/(8b)    o_k* = o_{k-1} (outdated) | o_{k-1} + f_k*(o_{k-1}*) (partial),
 *                       f_k* = the shared-expert part of block k
 *
 * Conventions for every entry point:
 *   - All pointers except `desc`/`blocks` are DEVICE pointers owned by the caller.
 *     The library never allocates, frees or synchronises; every call is
 *     asynchronous on `stream` (a cudaStream_t, NULL = the legacy default stream).
 *   - Argument errors return before any launch and leave outputs untouched.
 *     A failed launch returns FS_ERR_CUDA.  No exception crosses the ABI.
 *   - Device-side faults that the kernels detect (an expert index out of range,
 *     inconsistent offsets, a pipeline wait that ran out of time) never trap:
 *     the kernel records a code in the library's device error word and skips
 *     the work; fs_get_error() reads and clears it.
 *   - Row-major layouts throughout.  Activations are [rows, d] in the
 *     activation type: bf16 for FS_BF16, FS_FP8 and FS_MXFP8, fp32 for FS_F32 (the
 *     FP8 paths' E4M3 operands live inside the expert steps, see FS_FP8); gate weights and
 *     logits are fp32; indices int32.
 *   - Pointers must be 16-byte aligned; d and c must be multiples of 64;
 *     n_shared * c_shared must be a multiple of 64 (FS_FP8, FS_MXFP8: d, c and c_shared
 *     multiples of 128).  Otherwise FS_ERR_UNSUPPORTED.
 *   - Workspace: `ws` is caller-owned device scratch of at least
 *     fs_workspace_bytes(desc, L) bytes (L = 0 for the single-step calls),
 *     256-byte aligned.  Contents need not be initialised.
 *   - Environment, read once per process: FS_TC_VARIANT=pair runs the bf16 and
 *     FP8 tensor-core GEMMs on the CTA-pair kernel (256-row tiles over two SMs),
 *     pair_down / pair_up only the experts' down / gate/up projections; unset,
 *     the single-CTA kernel (the faster one under this GPU's power cap).  Every
 *     variant gives results within the same bounds of the definition; the
 *     gathered-row GEMM (fs_grouped_swiglu_gather) has no pair form and answers
 *     FS_ERR_UNSUPPORTED under FS_TC_VARIANT=pair.
 */
#ifndef FARSKIP_FS_H
#define FARSKIP_FS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FS_OK = 0,
    FS_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, k > E, bad enum */
    FS_ERR_UNSUPPORTED = 2,   /* shape/alignment outside what the kernels handle */
    FS_ERR_WORKSPACE = 3,     /* ws too small or misaligned */
    FS_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
    FS_ERR_DEVICE_STATE = 5   /* fs_get_error: a kernel recorded a device-side fault */
} fs_status;

/* FS_FP8: the FP8 expert path (the pages run inference with FP8 quantisation
 * and fused MoE forward kernels; experimental setup, software configuration).
 * Activations, the router, Combine and the residual stream are as for FS_BF16;
 * the operands of the expert GEMMs (routed and shared) are FP8 E4M3 with one
 * power-of-two scale per row along the contraction: per token for the block
 * input (quantised once by Dispatch), per row of the stored bf16 hidden h, per
 * output channel for the weights.  The scale of a row x is 2^e with e the
 * smallest integer such that max |x_i| 2^-e <= 448; the code of x_i is
 * x_i 2^-e rounded to E4M3 (nearest, ties to even, saturating at 448).  The
 * tensor cores take the E4M3 codes (kind::f8f6f4, fp32 accumulate) and the
 * GEMM epilogue multiplies by the two row scales.
 *
 * FS_MXFP8: the same expert path with block scales (the MX formats): every
 * operand row along the contraction is cut into blocks of 32 elements and each
 * block gets its own power-of-two scale by the rule above (clamped to 2^-127 ..
 * 2^127), stored as a UE8M0 byte (exponent + 127).  The tensor cores apply
 * both operands' block scales inside the contraction (kind::mxf8f6f4 with
 * block_scale).  The stored bf16 hidden h is quantised in blocks of 32 by the
 * gate/up GEMM itself.  Dispatch pads each expert's segment to a multiple of
 * 128 rows (see fs_dispatch).  d, c, c_shared multiples of 128. */
typedef enum { FS_BF16 = 0, FS_F32 = 1, FS_FP8 = 2, FS_MXFP8 = 3 } fs_dtype;

/* Gate rule s() applied to the top-k logits z (after the optional bias):
 *   SOFTMAX         w_s = exp(z_s) / sum over ALL experts of exp(z_j)
 *   SOFTMAX_RENORM  w_s = exp(z_s) / sum over the k chosen of exp(z_s')
 *   SIGMOID         w_s = sigmoid(z_s)
 *   SIGMOID_NORM    w_s = sigmoid(z_s) / sum over the k chosen of sigmoid(z_s')
 * Selection: the k largest z, descending, ties to the lower expert index. */
typedef enum {
    FS_GATE_SOFTMAX = 0,
    FS_GATE_SOFTMAX_RENORM = 1,
    FS_GATE_SIGMOID = 2,
    FS_GATE_SIGMOID_NORM = 3
} fs_gate;

/* Input of block k+1 (§3, eq. 8a/8b): PARTIAL u = o_k* = o_{k-1} + S_k,
 * OUTDATED u = o_{k-1}, DISABLED u = o_k (plain residual recurrence). */
typedef enum {
    FS_WIRE_PARTIAL = 0,
    FS_WIRE_OUTDATED = 1,
    FS_WIRE_DISABLED = 2,
    /* Layers with a stand-in attention sub-block A_k(a) = a W_att^T before the MoE
     * (fs_block_weights.w_att), wired as in §3's attention/MoE wiring:
     *   attn-in_k = o_{k-2} + attn-out_{k-1} + shared-out_{k-1}
     *   mlp-in_k  = attn-in_k + routed-out_{k-1} = o_{k-1}
     *   o_k = o_{k-1} + A_k(attn-in_k) + S_k(mlp-in_k) + R_k(mlp-in_k), o_k* = o_k - R_k */
    FS_WIRE_ATTN_FARSKIP = 3,
    /* the ordinary layer: h_k = o_{k-1} + A_k(o_{k-1}), o_k = h_k + S_k(h_k) + R_k(h_k),
     * o_k* = h_k + S_k */
    FS_WIRE_ATTN_PLAIN = 4
} fs_wiring;

/* One MoE layer: T tokens of width d, E routed experts of width c, top-k,
 * n_shared shared experts of width c_shared (0 = none), activation dtype, gate.
 * Every call validates it first: T, d, E, k, c >= 1, k <= E, n_shared >= 0 and
 * c_shared >= 1 when n_shared > 0, else FS_ERR_INVALID_ARG (an empty batch,
 * T = 0, is such an error: the caller skips the call); d, c, c_shared multiples
 * of 64 (128 for FS_FP8 and FS_MXFP8), E <= 512, k <= 16 and T k < 2^31 - 1024
 * (FS_MXFP8: T k + 127 E + 128 < 2^31 - 1024), else FS_ERR_UNSUPPORTED. */
typedef struct {
    int32_t T, d, E, k, c, n_shared, c_shared;
    int32_t dtype;   /* fs_dtype */
    int32_t gate;    /* fs_gate */
} fs_layer_desc;

/* One block's weights in the library's packed layouts (fs_pack_w13, fs_pack_w3,
 * fs_pack_w3_shared).  Element type: the router weight in the activation type,
 * the expert weights in desc->dtype's packed layout (FP8 / MX packs for FS_FP8 /
 * FS_MXFP8). */
typedef struct {
    const void* w_r;        /* [E, d] router (W_R), row-major */
    const float* bias;      /* [E] router bias added to the logits, or NULL */
    const void* w13;        /* packed gate/up: fs_pack_w13(E, c, d) */
    const void* w3;         /* packed down: fs_pack_w3(E, d, c) */
    const void* w13_shared; /* fs_pack_w13(1, n_shared c_shared, d) of the shared experts, NULL when n_shared = 0 */
    const void* w3_shared;  /* fs_pack_w3_shared(n_shared, c_shared, d) */
    const void* w_att;      /* [d, d] stand-in attention weight, row-major (attention wirings only), or NULL */
} fs_block_weights;

/* Bytes of workspace needed by the single-step calls (L = 0) or by
 * fs_farskip_stack with L blocks (L >= 1) and the MoE wirings (PARTIAL,
 * OUTDATED, DISABLED).  Returns 0 for an invalid desc. */
size_t fs_workspace_bytes(const fs_layer_desc* desc, int L);

/* Workspace of fs_farskip_stack with the attention wirings (FS_WIRE_ATTN_*):
 * fs_workspace_bytes(desc, L) plus the attention buffers.  0 if invalid. */
size_t fs_workspace_bytes_attn(const fs_layer_desc* desc, int L);

/* Packed weight layouts.  A weight matrix [G, N, K] (N output rows, K the
 * contracted dimension, K-contiguous as the page writes W1, W2 [c, d] and
 * W3 [d, c]) is stored
 *   bf16: tiled, [G][ceil(N/256)][K/64][256][64]: every 256-row x 64-column
 *         tile the tensor-core GEMM loads is one contiguous 32 KB block
 *         (rows past N are zero), so weight streaming reads HBM sequentially;
 *   fp32: row-major [G, N, K];
 *   FP8:  E4M3 codes tiled as [G][ceil(N/256)][K/128][256][128] (32 KB blocks,
 *         rows past N zero), then the G N fp32 row scales (output channel n of
 *         group g at index g N + n).  The pack functions take the bf16 weights
 *         and quantise each output-channel row (FS_FP8 in fs_dtype);
 *   MXFP8: the codes tiled as for FP8 (rows past N zero), then the UE8M0
 *         block scales as [G][ceil(N/256)][K/128][1024]: for a 256-row tile and
 *         128 elements of K, byte (r / 128) 512 + (r % 32) 16 + ((r % 128) / 32) 4 + b
 *         holds the scale of tile row r, block b (0..3) of those 128 elements
 *         (rows past N: 127, a unit scale).
 * fs_packed_bytes gives the size (0 for invalid arguments; K % 64 == 0, FP8:
 * K % 128 == 0, MXFP8: K and N multiples of 128). */
size_t fs_packed_bytes(int32_t G, int32_t N, int32_t K, int32_t dtype);

/* Gate/up: the page's W1 (up) and W2 (gate), each [G, c, d], as one packed
 * [G, N = 2c, K = d] matrix whose rows interleave gate and up: for each block
 * of 64 expert columns b, packed rows [128b, 128b+64) are W2 rows [64b, 64b+64)
 * and rows [128b+64, 128b+128) are W1 rows, so the SwiGLU epilogue finds gate
 * and up of one column in the same tile.  c % 64 == 0, d % 64 == 0.  w13 holds
 * fs_packed_bytes(G, 2c, d, dtype) bytes. */
fs_status fs_pack_w13(int32_t G, int32_t c, int32_t d, int32_t dtype,
                      const void* w1, const void* w2, void* w13, void* stream);

/* Down: the page's W3 [G, d, c] as a packed [G, N = d, K = c] matrix
 * (fs_packed_bytes(G, d, c, dtype) bytes). */
fs_status fs_pack_w3(int32_t G, int32_t d, int32_t c, int32_t dtype, const void* w3, void* w3p,
                     void* stream);

/* Shared experts: n_shared down projections, each [d, c_shared], side by side
 * along the expert width, w3cat[i, s c_shared + j] = w3s[s, i, j], packed as a
 * [1, N = d, K = n_shared c_shared] matrix (fs_packed_bytes(1, d, n_shared
 * c_shared, dtype) bytes).  By the TP-slicing identity of §2.1 the sum of the
 * shared experts equals one MLP over the concatenated width; their gate/up
 * weights [n_shared, c_shared, d] are already concatenated in memory and are
 * packed with fs_pack_w13(G = 1, c = n_shared c_shared).  c_shared % 64 == 0. */
fs_status fs_pack_w3_shared(int32_t n_shared, int32_t c_shared, int32_t d, int32_t dtype,
                            const void* w3s, void* w3cat, void* stream);

/* FP8 row-scaled matrix [rows, cols] (the FS_FP8 activations x_perm and the
 * output of fs_quantize_rows_fp8): rows * cols E4M3 codes, row-major, then
 * from byte offset rows * cols rounded up to a multiple of 256 the rows fp32
 * scales; element (r, i) = value(code[r, i]) * scale[r].  Its size in bytes,
 * or 0 for rows < 1 or cols < 1. */
size_t fs_fp8_rows_bytes(int64_t rows, int32_t cols);

/* Quantise bf16 rows x [rows, cols] to the FP8 row-scaled matrix q (see
 * FS_FP8): the quantisation of the hidden between the two expert GEMMs.
 * cols % 128 == 0. */
fs_status fs_quantize_rows_fp8(int64_t rows, int32_t cols, const void* x, void* q, void* stream);

/* MX matrix [rows, cols] (the FS_MXFP8 activations: x_perm, the shared
 * experts' quantised input, the hidden): with rows128 = rows rounded up to a
 * multiple of 128, rows128 * cols E4M3 codes row-major, then from byte offset
 * rows128 * cols rounded up to a multiple of 256 the UE8M0 block scales in
 * 512-byte chunks [rows128 / 128][cols / 128][512]: byte
 * (r % 32) 16 + ((r % 128) / 32) 4 + b of chunk (r / 128, j) holds the scale of
 * row r, block b (0..3) of columns [128 j, 128 j + 128); element (r, i) =
 * value(code[r, i]) 2^(scale byte - 127).  Its size in bytes, or 0 for
 * rows < 1 or cols not a positive multiple of 128. */
size_t fs_mx_rows_bytes(int64_t rows, int32_t cols);

/* Quantise bf16 rows x [rows, cols] to the MX matrix q (blocks of 32 along
 * each row; the rows up to rows128 get zero codes and unit scales).
 * cols % 128 == 0. */
fs_status fs_quantize_rows_mx(int64_t rows, int32_t cols, const void* x, void* q, void* stream);

/* Rows of fs_dispatch's x_perm and of fs_grouped_swiglu's y_perm for desc:
 * T k, or for FS_MXFP8 (128-row aligned expert segments) T k + 127 E rounded
 * up to a multiple of 128.  0 for an invalid desc. */
int64_t fs_dispatch_rows(const fs_layer_desc* desc);

/* Router (§2.1, G(A) = s(A W_R^T)): logits z = u W_R^T + bias (fp32 accumulate;
 * bf16 operands on the tensor cores for FS_BF16, fp32 FMA for FS_F32), then the
 * top-k selection and gate weights of desc->gate.
 *   u [T, d], w_r [E, d], bias [E] fp32 or NULL
 *   -> topk_idx [T, k] int32 (slot order = descending z), topk_w [T, k] fp32,
 *      logits [T, E] fp32 (z without the bias; NULL = kept in ws only).
 * Needs ws of fs_workspace_bytes(desc, 0) bytes.  E <= 512, k <= 16. */
fs_status fs_router_topk(const fs_layer_desc* desc, const void* u, const void* w_r,
                         const float* bias, int32_t* topk_idx, float* topk_w, float* logits,
                         void* ws, size_t ws_bytes, void* stream);

/* Dispatch (§2.1, local form): stable counting sort of the (token, slot) pairs
 * by expert, in token order within each expert, and the permuted copy of u.
 *   topk_idx [T, k], u [T, d]
 *   -> counts [E], offsets [E+1] (exclusive prefix, offsets[E] = T k),
 *      pos [T k] (pos[t k + s] = permuted row of (t, s)),
 *      perm_src [T k] (perm_src[p] = token of permuted row p),
 *      x_perm [T k, d] (x_perm[p] = u[perm_src[p]]); x_perm NULL = no row copy
 *      (for fs_grouped_swiglu_gather, which gathers the rows itself).
 * An index outside [0, E) sets the device error word (reported by
 * fs_get_error) and that pair is dropped.  FS_FP8: u is bf16 and x_perm is an
 * FP8 row-scaled matrix [T k, d] (fs_fp8_rows_bytes(T k, d) bytes): each token
 * row is quantised once and its codes and scale go to all of its k rows.
 * FS_MXFP8: each expert's segment starts at a multiple of 128 rows: offsets[e]
 * is the exclusive prefix sum of the counts rounded up to 128 (offsets[E] the
 * padded total), expert e's rows are [offsets[e], offsets[e] + counts[e]) and
 * the rows up to offsets[e+1] are padding with unspecified contents; x_perm is
 * an MX matrix of fs_dispatch_rows(desc) rows (fs_mx_rows_bytes bytes), each
 * token row quantised once in blocks of 32, and perm_src has
 * fs_dispatch_rows(desc) entries (those of padding rows unspecified). */
fs_status fs_dispatch(const fs_layer_desc* desc, const int32_t* topk_idx, const void* u,
                      int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src,
                      void* x_perm, void* ws, size_t ws_bytes, void* stream);

/* fs_dispatch without a workspace.  The paper has no counterpart: this exists
 * for callers that cannot hand the library device scratch memory -- for example
 * a plugin or custom-op interface that passes only input and output buffers,
 * or code that must not call cudaMalloc/cudaFree (which can synchronise the
 * device) on its execution path.  Same arguments and results as fs_dispatch,
 * minus ws/ws_bytes (x_perm NULL = no row copy, as there).  Its scratch (the
 * per-chunk expert histogram) is a fixed 256 KiB device array inside the
 * library, present on every GPU that loads the library until the process
 * exits; it holds ceil(T / 1024) * E <= 65536 ints (e.g. T <= 131072 tokens
 * with E <= 512 experts, T <= 262144 with E <= 256).  Larger shapes return
 * FS_ERR_WORKSPACE before any launch (fs_last_cuda_error gives the sizes).
 * Nothing in the scratch needs to start at zero: each call overwrites every
 * entry it reads.  All calls share the one array, so calls that overlap on the
 * GPU (several streams, or several host threads) race and must be serialised
 * by the caller.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current) and keeps it for
 * the life of the process; make that first call before any stream capture,
 * and do not keep using the library after cudaDeviceReset on that device (the
 * kept address, like the library's error word and events, belongs to the
 * context that was reset).  Allocates nothing. */
fs_status fs_dispatch_noalloc(const fs_layer_desc* desc, const int32_t* topk_idx, const void* u,
                              int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src,
                              void* x_perm, void* stream);

/* Routed experts (§2.1 MLP and MoE equations), grouped by expert: for every
 * expert e and every row p in [offsets[e], offsets[e+1]):
 *   h = SiLU(x W2_e^T) * (x W1_e^T)  (fp32 accumulate, stored bf16/fp32 in ws)
 *   y_perm[p] = h W3_e^T             (fp32 accumulate, stored in the activation type)
 *   x_perm [T k, d], offsets [E+1] (device; the host never reads them),
 *   w13 = fs_pack_w13(E, c, d), w3 = fs_pack_w3(E, d, c) -> y_perm [T k, d].
 * bf16: persistent tcgen05/TMEM grouped GEMMs fed by TMA; fp32: fp32 FMA.
 * FS_FP8: x_perm is fs_dispatch's FP8 row-scaled matrix, the weights are the
 * FP8 packs; h is stored bf16, quantised per row (fs_quantize_rows_fp8) and
 * fed to the down GEMM as E4M3; y_perm is bf16.  FS_MXFP8: x_perm is
 * fs_dispatch's MX matrix, offsets its padded offsets, the weights the MXFP8
 * packs; every row of each padded segment is computed (padding rows give
 * unspecified y), h is rounded to bf16 and quantised in blocks of 32 by the
 * gate/up GEMM's epilogue; y_perm has fs_dispatch_rows(desc) rows. */
fs_status fs_grouped_swiglu(const fs_layer_desc* desc, const void* x_perm, const int32_t* offsets,
                            const void* w13, const void* w3, void* y_perm,
                            void* ws, size_t ws_bytes, void* stream);

/* fs_grouped_swiglu with the Dispatch row copy fused into the first GEMM: row
 * p of the routed-expert input is read straight from u[perm_src[p]] by the
 * GEMM's operand loads (TMA tile::gather4 on the tensor cores), so x_perm is
 * never written or read.  u [T, d], perm_src [T k] (fs_dispatch's output),
 * offsets [E+1] -> y_perm [T k, d].  Results are bit-identical to
 * fs_dispatch + fs_grouped_swiglu.  FS_ERR_UNSUPPORTED with the CTA-pair GEMM
 * variant and for FS_FP8 and FS_MXFP8. */
fs_status fs_grouped_swiglu_gather(const fs_layer_desc* desc, const void* u, const int32_t* perm_src,
                                   const int32_t* offsets, const void* w13, const void* w3,
                                   void* y_perm, void* ws, size_t ws_bytes, void* stream);

/* Shared expert(s) (§2.1): S = sum_i MLP_shared_i(u) over all T tokens, as one
 * MLP of width n_shared c_shared.  u [T, d] -> s_out [T, d] in fp32 (S is only
 * ever added into the residual stream, so it keeps fp32 accumulator precision).
 * FS_FP8: u is bf16 and is quantised per token in ws; the weights are FP8 packs.
 * FS_MXFP8: u is quantised in blocks of 32 in ws; the weights are MX packs. */
fs_status fs_shared_expert(const fs_layer_desc* desc, const void* u, const void* w13_shared,
                           const void* w3_shared, void* s_out, void* ws, size_t ws_bytes,
                           void* stream);

/* Combine (§2.1, local form) fused with the FarSkip update (§3, eq. 8a/8b):
 *   R[t]  = sum_{s<k} topk_w[t, s] * y_perm[pos[t k + s]]   (fp32, slot order)
 *   o_partial[t] = o_prev[t] + S[t] + extra[t]               (o_k*)
 *   o_full[t]    = o_prev[t] + S[t] + extra[t] + R[t]        (o_k)
 *   u_next[t]    = the next block's input per `wiring`: o_k* (PARTIAL),
 *                  o_prev (OUTDATED) or o_k (DISABLED)
 *   u_full[t]    = o_k
 * All sums in fp32, each output rounded once.  y_perm, u_next and u_full have
 * the activation type; shared_out (fs_shared_expert's output) and
 * extra (e.g. fs_attn_standin's output) are fp32; the residual stream o_prev
 * (prev_dtype) and o_partial / o_full (out_dtype) are FS_BF16 or FS_F32 each,
 * so a stack can carry its residual in fp32.  shared_out NULL = no shared
 * expert; extra NULL = no extra term; o_partial, u_next, u_full NULL = not
 * written (wiring is then ignored). */
fs_status fs_combine(const fs_layer_desc* desc, const void* y_perm, const int32_t* pos,
                     const float* topk_w, const void* o_prev, int32_t prev_dtype,
                     const void* shared_out, const float* extra, void* o_partial, void* o_full,
                     int32_t out_dtype, void* u_next, int32_t wiring, void* u_full, void* stream);

/* The shared experts (§2.1) with Combine and the FarSkip update (§3, eq. 8a/8b)
 * in one pass: fs_shared_expert followed by fs_combine, with the combine done
 * in the epilogue of the shared experts' down projection, so the fp32 shared
 * output S never goes to memory and the memory-bound combine overlaps that
 * projection's tensor-core work.  Results are bit-identical to
 *   fs_shared_expert(desc, u, w13_shared, w3_shared, S, ...);
 *   fs_combine(desc, y_perm, pos, topk_w, o_prev, prev_dtype, S, NULL,
 *              o_partial, o_full, out_dtype, u_next, wiring, NULL, ...).
 * u [T, d] (the shared experts' input), y_perm, pos, topk_w as for fs_combine
 * (the routed experts' outputs must be complete when the call's work runs),
 * o_prev [T, d] in prev_dtype -> o_partial (NULL = not written), o_full in
 * out_dtype, u_next (NULL = not written) per wiring.  FS_BF16 or FS_FP8 with
 * n_shared >= 1 and k <= 8, else FS_ERR_UNSUPPORTED (n_shared = 0:
 * FS_ERR_INVALID_ARG).  Needs ws of fs_workspace_bytes(desc, 0) bytes.
 * (fs_farskip_stack keeps the two separate calls: at DeepSeek-V3's shapes this
 * fused pass measured slower than them.) */
fs_status fs_shared_expert_combine(const fs_layer_desc* desc, const void* u, const void* w13_shared,
                                   const void* w3_shared, const void* y_perm, const int32_t* pos,
                                   const float* topk_w, const void* o_prev, int32_t prev_dtype, void* o_partial,
                                   void* o_full, int32_t out_dtype, void* u_next, int32_t wiring, void* ws,
                                   size_t ws_bytes, void* stream);

/* Stand-in attention sub-block for the attention wirings: out = a W_att^T
 * (a per-token dense GEMM on the tensor cores for bf16, fp32 FMA for fp32).
 * It stands in for attention (which mixes tokens) so the §3 attention/MoE
 * wiring can be run; it is not attention.  a [T, d] (activation type),
 * w_att [d, d] -> out [T, d] fp32.  Needs ws of fs_workspace_bytes(desc, 0). */
fs_status fs_attn_standin(const fs_layer_desc* desc, const void* a, const void* w_att, float* out,
                          void* ws, size_t ws_bytes, void* stream);

/* L FarSkip blocks (§3): o_0 = u_1 = x; block k runs router, dispatch, routed
 * experts, shared expert and combine on u_k and o_{k-1}, producing
 * o_k* = o_{k-1} + S_k and o_k = o_k* + R_k; u_{k+1} follows `wiring`.
 * Between blocks the residual stream o_k, o_k* is kept in fp32 (in ws) and
 * u_{k+1} is its rounding to the activation type (the GEMM operand).  The
 * attention wirings (FS_WIRE_ATTN_*) run A_k from blocks[k].w_att first and
 * need fs_workspace_bytes_attn(desc, L) bytes of ws.
 *   blocks [L] (host array of device pointers), x [T, d]
 *   -> o_full = o_L, o_partial = o_L* (NULL = not written), activation type.
 * Needs ws of fs_workspace_bytes(desc, L) bytes.  Everything is enqueued on
 * `stream` with no host synchronisation. */
fs_status fs_farskip_stack(const fs_layer_desc* desc, int32_t L, int32_t wiring,
                           const fs_block_weights* blocks, const void* x,
                           void* o_full, void* o_partial, void* ws, size_t ws_bytes,
                           void* stream);

/* fs_farskip_stack on two streams, the single-GPU form of the overlap the
 * FarSkip wiring enables (§3, §4): with the partial (or outdated) wiring the
 * input of block k+1 is u_{k+1} = o_{k-1} + S_k (or o_{k-1}), which does not
 * depend on block k's routed experts.  So `stream2` runs, for every block, the
 * router, dispatch and shared expert and forms o_k* = o_{k-1} + S_k and
 * u_{k+1}, while `stream` runs the routed experts and the final
 * o_k = o_k* + R_k; block k+1's router/dispatch/shared thus run concurrently
 * with block k's routed grouped GEMMs.  Bit-identical to fs_farskip_stack.
 * wiring must be FS_WIRE_PARTIAL or FS_WIRE_OUTDATED; stream2 != stream.
 * Every dtype (FS_FP8 / FS_MXFP8: stream2's Dispatch also quantises u_k for
 * the shared experts).
 * Work queued on `stream` before the call is complete before stream2 starts,
 * and work queued on `stream` after the call sees all of the stack's results.
 * Needs ws of fs_workspace_bytes_overlap(desc, L) bytes.  The library keeps
 * three CUDA events per device for the hand-over (created on first use). */
fs_status fs_farskip_stack_overlap(const fs_layer_desc* desc, int32_t L, int32_t wiring,
                                   const fs_block_weights* blocks, const void* x,
                                   void* o_full, void* o_partial, void* ws, size_t ws_bytes,
                                   void* stream, void* stream2);
size_t fs_workspace_bytes_overlap(const fs_layer_desc* desc, int L);

/* ----------------------------------------------------------------- training
 * The backward of the MoE stack for the MoE wirings (PARTIAL, OUTDATED,
 * DISABLED), bf16 (FS_BF16) only.  The pages train FarSkip models but print no
 * gradient formulas; these are the derivatives of the forward above:
 *   per block, with o = o_prev + S + R and o* = o_prev + S:
 *     dR = dO, dS = dO + dOs, do_prev = dO + dOs
 *     routed: dw_s = <dR, y_s>, dy = w_s dR, dh = dy W3, dg = dh a SiLU'(g),
 *             da = dh SiLU(g), dx = dg W2 + da W1, dW3 += dy h^T,
 *             dW2 += dg u^T, dW1 += da u^T (u the block input)
 *     shared experts: the same with dS and gate weight 1
 *     router: dz = d(gate weights)/dz applied to dw (the gate rule of desc;
 *             top-k selection has no gradient; the bias is not a parameter),
 *             dW_R += dz u^T, du += dz W_R
 *     du = sum_s dx_s (Dispatch backward) + dx_shared + dz W_R
 *   the stack: block k's do_prev flows to o_{k-1}; its du to where u_k came
 *   from (o_{k-1}* partial, o_{k-2} outdated, o_{k-1} disabled, x for k = 1).
 * Stored backward operands are bf16 (dy, dg/da, dx per slot, dS, dz); every
 * sum is fp32; the input gradient and the weight gradients are fp32 in the
 * page's layouts.  fs_farskip_stack_train runs the forward and keeps what the
 * backward reads (u_k, logits, routing, Dispatch permutation, x_perm,
 * pre-activations, hidden, y_perm) in `saved` (fs_train_saved_bytes(desc, L) bytes, 256-byte
 * aligned); it needs ws of fs_workspace_bytes(desc, L).
 * fs_farskip_stack_backward needs ws of fs_workspace_bytes_backward(desc, L). */

/* Transposed weight packs of the input-gradient GEMMs, in the tiled bf16
 * layout (sizes: fs_packed_bytes(G, N', K', FS_BF16) with the N', K' given):
 *   fs_pack_w13t        [G, d, 2c]: element (i, q) = packed gate/up row q of W1/W2, column i
 *   fs_pack_w3t         [G, c, d]:  element (j, i) = W3[i, j]
 *   fs_pack_w3t_shared  [1, n_shared c_shared, d]: the transposed concatenated shared W3
 *   fs_pack_wrt         [1, d, E rounded up to 64]: element (i, j) = W_R[j, i] (0 for j >= E) */
fs_status fs_pack_w13t(int32_t G, int32_t c, int32_t d, const void* w1, const void* w2, void* out, void* stream);
fs_status fs_pack_w3t(int32_t G, int32_t d, int32_t c, const void* w3, void* out, void* stream);
fs_status fs_pack_w3t_shared(int32_t n_shared, int32_t c_shared, int32_t d, const void* w3s, void* out,
                             void* stream);
fs_status fs_pack_wrt(int32_t E, int32_t d, const void* w_r, void* out, void* stream);

/* One block's transposed packs (device pointers; the shared ones NULL when n_shared = 0). */
typedef struct {
    const void* w13t;
    const void* w3t;
    const void* w13t_shared;   /* fs_pack_w13t(1, n_shared c_shared, d) of the shared gate/up */
    const void* w3t_shared;
    const void* w_rt;
} fs_block_weights_t;

/* One block's weight gradients (device, fp32, page layouts: dw_r [E, d],
 * dw1, dw2 [E, c, d], dw3 [E, d, c], shared [n_shared, c_shared, d] and
 * [n_shared, d, c_shared]).  Overwritten. */
typedef struct {
    float* dw_r;
    float* dw1;
    float* dw2;
    float* dw3;
    float* dw1_shared;
    float* dw2_shared;
    float* dw3_shared;
} fs_block_grads;

size_t fs_train_saved_bytes(const fs_layer_desc* desc, int L);
size_t fs_workspace_bytes_backward(const fs_layer_desc* desc, int L);

/* fs_farskip_stack for the MoE wirings, keeping the backward's inputs in `saved`. */
fs_status fs_farskip_stack_train(const fs_layer_desc* desc, int32_t L, int32_t wiring,
                                 const fs_block_weights* blocks, const void* x, void* o_full,
                                 void* o_partial, void* saved, size_t saved_bytes, void* ws,
                                 size_t ws_bytes, void* stream);

/* Backward of the stack run by fs_farskip_stack_train (same desc, L, wiring,
 * blocks, saved): d_o, d_os [T, d] fp32 the gradients of o_L and o_L* (d_os
 * NULL = zero) -> dx [T, d] fp32 and grads[L]. */
fs_status fs_farskip_stack_backward(const fs_layer_desc* desc, int32_t L, int32_t wiring,
                                    const fs_block_weights* blocks, const fs_block_weights_t* blocks_t,
                                    const void* saved, size_t saved_bytes, const float* d_o,
                                    const float* d_os, float* dx, const fs_block_grads* grads,
                                    void* ws, size_t ws_bytes, void* stream);

/* Read and clear the device error word (synchronises the device).  FS_OK when
 * no kernel recorded a fault; FS_ERR_DEVICE_STATE otherwise, with the raw code
 * in *code when code != NULL (1 = expert index out of range, 2 = inconsistent
 * offsets, 3 = pipeline wait timed out, 4 = size beyond a kernel limit). */
fs_status fs_get_error(int32_t* code);

/* Self-test of the kernels' bounded waits: one kernel waits on a barrier that
 * nothing signals, gives up after limit_us microseconds (1 .. 2,000,000),
 * records code 3 (a wait timed out) in the device error word and returns; the
 * context stays usable.  fs_get_error then reports FS_ERR_DEVICE_STATE, 3. */
fs_status fs_selftest_wait_timeout(int32_t limit_us, void* stream);

/* Number of kernels this library has launched since it was loaded. */
uint64_t fs_launch_count(void);

/* Text of the last CUDA error behind an FS_ERR_CUDA on this host thread
 * ("" if none).  The string is owned by the library. */
const char* fs_last_cuda_error(void);

/* Human-readable name of a status. */
const char* fs_status_string(fs_status status);

#ifdef __cplusplus
}
#endif
#endif
