// kernels.h -- internal launchers of libfs (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fs {

constexpr int kMaxGroups = 1024;   // groups (experts) one grouped GEMM handles
constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 512;   // router top-k kernel limit

// EPI_DSWIGLU: the accumulator is dh (hidden columns); with the stored
// pre-activations g, a (TcExtra::aux, packed gate/up column order) it writes
// dg = dh a SiLU'(g) and da = dh SiLU(g) (bf16) at the same packed columns.
// EPI_COMBINE: one group over all T token rows (the shared experts' down
// projection); the accumulator is the shared output S of token row t, and the
// epilogue is Combine fused with the FarSkip update (CombineEpi).
enum { EPI_SWIGLU = 0, EPI_BF16 = 1, EPI_F32 = 2, EPI_DSWIGLU = 3, EPI_COMBINE = 4 };

// Combine in the epilogue of the shared experts' down projection, with the
// arithmetic of combine_kernel (fp32, rounded once per output):
//   base = o_prev[t] + S[t]; R = sum_{s<k} w[t, s] y_perm[pos[t k + s]] (slot order)
//   o_partial[t] = base (if set), o_full[t] = base + R,
//   u_next[t] = bf16 of base (u_src 0), o_prev (1) or base + R (2) (if set).
// y_perm and u_next are bf16; the residual o_prev / o_partial / o_full is bf16
// or fp32; k <= 8.
struct CombineEpi {
    const void* y_perm = nullptr;
    const int32_t* pos = nullptr;
    const float* topk_w = nullptr;
    int k = 0;
    const void* o_prev = nullptr;
    int prev_bf16 = 0;
    void* o_partial = nullptr;
    void* o_full = nullptr;
    int out_bf16 = 0;
    void* u_next = nullptr;
    int u_src = 0;
};
constexpr int kCombineEpiMaxK = 8;

// Optional epilogue inputs/outputs of launch_tc_gemm:
//   aux          EPI_SWIGLU: also store the pre-activations g, a (bf16) here
//                (training forward); EPI_DSWIGLU: read them from here
//   aux_ld       row stride of aux in elements (2c)
//   accumulate   EPI_F32: out += acc instead of out = acc
struct TcExtra {
    void* aux = nullptr;
    long long aux_ld = 0;
    int accumulate = 0;
    // EPI_F32, one group, no accumulate, no gather: the K loop split into ksplit
    // ranges, range s written to rows [s a_rows, (s + 1) a_rows) of out (partial
    // sums; the consumer adds them in order).  Ignored (1) by the CTA-pair kernel.
    int ksplit = 1;
    // EPI_COMBINE: the Combine operands and outputs (out is unused)
    const CombineEpi* combine = nullptr;
    // -1: the library-wide kernel variant; 0: single-CTA kernel; 1: CTA-pair kernel
    // (its plan must then be built with 256-row tiles)
    int variant = -1;
};

void count_launch();
int* dev_error_ptr();

// gemm_tc.cu (bf16 operands, tcgen05)
int tc_block_m();
int tc_block_m_f8();
// K splits of the router logits GEMM for T rows, N = E, K = d: enough CTAs for
// the SMs when T is small (1 when the CTA-pair kernel is selected or T is large)
int tc_router_ksplit(long long T, int E, int d);
cudaError_t launch_plan(const int* offsets, int G, int n_rows, int bm, int* plan, cudaStream_t st);
// gather_rows (nullable): GEMM row p reads row gather_rows[p] of A (p < gather_limit)
bool tc_gather_supported();
// b_blocked: B is in the tiled weight layout of pack.cu ([G][ceil(N/256)][K/64][256][64])
cudaError_t launch_tc_gemm(int epi, const void* A, long long a_rows, const void* B, int G, int N, int K,
                           const int* plan, int max_mtiles, void* out, long long ldo, int out_cols,
                           const int* gather_rows, int gather_limit, bool b_blocked, cudaStream_t st,
                           const TcExtra* ex = nullptr);
// Weight-gradient GEMM: for each group g, out_g [M, N] = sum over the group's
// rows p in [offs[g], offs[g+1]) of A[p, m] B[p, n], with A [P, lda] and B
// [P, ldb] bf16 row-major (one row per token, read in place as MN-major
// tiles), offs on the device (nullptr: G = 1, rows [0, P)); M <= lda, N <= ldb.
// fp32 out; remap 0: out [G][M][N]; remap 1 (packed gate/up rows, M = 2c):
// rows to out2 (gate, W2) and out (up, W1), each [G][c][N]; remap 2
// (concatenated shared down columns): [N / split][M][split].
cudaError_t launch_wgrad_gemm(const void* A, int lda, const void* B, int ldb, long long P, const int* offs, int G,
                              int M, int N, float* out, float* out2, int remap, int split, cudaStream_t st);
// FP8 E4M3 operands (kind::f8f6f4): A codes [a_rows, K] with a_scale[a_rows],
// B packed by quant.cu with b_scale[G N]; the epilogue multiplies the fp32
// accumulator by a_scale[row] b_scale[g N + col].  Single-CTA kernel only.
cudaError_t launch_tc_gemm_f8(int epi, const void* A, long long a_rows, const float* a_scale, const void* B,
                              const float* b_scale, int G, int N, int K, const int* plan, int max_mtiles, void* out,
                              long long ldo, int out_cols, cudaStream_t st, const CombineEpi* combine = nullptr,
                              int variant = -1);
// The forward down projections (y = h W3^T) on the CTA-pair kernel while the
// other GEMMs keep the library-wide variant (FS_TC_VARIANT=pair_down); the
// forward gate/up projections on it (FS_TC_VARIANT=pair_up).
bool tc_down_pair();
bool tc_up_pair();

// Tensor maps (gemm_tc.cu): a [rows, cols] row-major matrix of bf16 (f8: 8-bit
// codes) with a box_rows x 128-byte box and the 128-byte swizzle; the tiled
// weight layout [nblocks][256][128 bytes]; a bf16 output map for 32 x 32
// pieces (64-byte swizzle).  num_sms: SMs of the current device.
cudaError_t make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows, bool f8 = false);
cudaError_t make_map_blocked(CUtensorMap* m, const void* base, long long nblocks, int box_rows, bool f8 = false);
cudaError_t make_out_map_bf16(CUtensorMap* m, void* base, long long rows, long long cols, long long ldo);
cudaError_t num_sms(int* out);
// Raise fn's dynamic shared memory limit to `bytes` on the current device, once
// per device (the attribute belongs to each device's copy of the kernel; set[d]
// records device d).  num_sms is cached per device too.
constexpr int kMaxDevices = 64;
cudaError_t smem_attr_once(const void* fn, size_t bytes, bool (&set)[kMaxDevices]);

// gemm_mx.cu: block-scaled FP8 operands (kind::mxf8f6f4.block_scale).  A is an
// MX matrix of a_rows (a multiple of 128) rows and K columns (codes A, scale
// chunks a_sf), B MX-packed weights [G, N, K] (codes, chunks b_sf); groups
// start at multiples of 128 rows.  EPI_SWIGLU writes the hidden as an MX
// matrix (codes at out with row stride ldo bytes, chunks at h_sf; out_cols = c);
// EPI_BF16 / EPI_F32 write bf16 / fp32 rows.
cudaError_t launch_mx_gemm(int epi, const void* A, long long a_rows, const uint8_t* a_sf, const void* B,
                           const uint8_t* b_sf, int G, int N, int K, const int* plan, int max_mtiles, void* out,
                           long long ldo, int out_cols, uint8_t* h_sf, cudaStream_t st);

// mx.cu: MX packs and quantisation (layouts in mx.cuh)
size_t packed_bytes_mx(int G, int N, int K);
const uint8_t* packed_sf_mx(const void* packed, int G, int N, int K);
cudaError_t launch_pack_w13_mx(int G, int c, int d, const void* w1, const void* w2, void* w13, cudaStream_t st);
cudaError_t launch_pack_w3_mx(int G, int d, int c, const void* w3, void* w3p, cudaStream_t st);
cudaError_t launch_pack_w3_shared_mx(int ns, int cs, int d, const void* w3s, void* w3cat, cudaStream_t st);
cudaError_t launch_quant_rows_mx(const void* x, long long rows, int cols, void* q, cudaStream_t st);
cudaError_t launch_dispatch_copy_mx(const void* u, int T, int d, int k, const int32_t* pos, void* x_q,
                                    long long rows_cap, void* u_q, cudaStream_t st);

// gemm_simt.cu (fp32 operands, fp32 FMA)
int simt_block_m();
cudaError_t launch_simt_gemm(int epi, const float* A, long long a_rows, const float* B, int G, int N, int K,
                             const int* plan, int max_mtiles, float* out, long long ldo, int out_cols,
                             const int* gather_rows, int gather_limit, cudaStream_t st);

// router.cu
// logits: nsplit partial sums [nsplit][T][E] added in order (nsplit = 1: the
// logits themselves); z_out (nullable) receives the summed logits [T, E].
cudaError_t launch_topk(const float* logits, int nsplit, const float* bias, int T, int E, int k, int gate,
                        int32_t* topk_idx, float* topk_w, float* z_out, cudaStream_t st);

// dispatch.cu
constexpr int kStaticDispatchScratchInts = 65536;   // 256 KiB: fs_dispatch_noalloc's scratch
size_t dispatch_ws_bytes(int T, int E);
// qmode kQuantRow: x_perm is an FP8 row-scaled matrix [T k, d] (fp8.cuh) and u
// (bf16) is quantised per token on the way; kQuantMx: each expert's segment
// starts at a multiple of 128 rows (offsets padded) and x_perm is an MX matrix
// of rows_cap rows (mx.cuh), u quantised in blocks of 32; u_q (nullable)
// receives the quantised u [T, d] in the same form.
enum { kQuantNone = 0, kQuantRow = 1, kQuantMx = 2 };
cudaError_t launch_dispatch_noalloc(const int32_t* topk_idx, const void* u, int T, int d, int E, int k, int elem_bytes,
                                    int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src,
                                    void* x_perm, cudaStream_t st, int qmode, long long rows_cap);
cudaError_t launch_dispatch(const int32_t* topk_idx, const void* u, int T, int d, int E, int k, int elem_bytes,
                            int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src, void* x_perm,
                            int32_t* scratch, cudaStream_t st, int qmode = kQuantNone, void* u_q = nullptr,
                            long long rows_cap = 0);

// combine.cu
cudaError_t launch_combine(const void* y_perm, const int32_t* pos, const float* topk_w, const void* o_prev,
                           int prev_bf16, const void* shared_out, const float* extra, void* o_partial, void* o_full,
                           int out_bf16, void* u_next, int u_src, void* u_full, int T, int d, int k, int is_bf16,
                           cudaStream_t st);

// pack.cu -- bf16 weights are packed into the tiled layout [G][ceil(N/256)][K/64][256][64]
// (rows past N are zero); fp32 weights keep row-major layouts.
size_t packed_bytes(int G, int N, int K, int elem_bytes);
cudaError_t launch_pack_w13(int G, int c, int d, int elem_bytes, const void* w1, const void* w2, void* w13,
                            cudaStream_t st);
cudaError_t launch_pack_w3(int G, int d, int c, int elem_bytes, const void* w3, void* w3p, cudaStream_t st);
cudaError_t launch_pack_w3_shared(int ns, int cs, int d, int elem_bytes, const void* w3s, void* w3cat,
                                  cudaStream_t st);

// quant.cu -- FP8 E4M3: packed weights hold codes [G][ceil(N/256)][K/128][256][128]
// then G N fp32 row scales; launch_quant_rows writes an FP8 row-scaled matrix.
size_t packed_bytes_fp8(int G, int N, int K);
const float* packed_scales_fp8(const void* packed, int G, int N, int K);
cudaError_t launch_pack_w13_fp8(int G, int c, int d, const void* w1, const void* w2, void* w13, cudaStream_t st);
cudaError_t launch_pack_w3_fp8(int G, int d, int c, const void* w3, void* w3p, cudaStream_t st);
cudaError_t launch_pack_w3_shared_fp8(int ns, int cs, int d, const void* w3s, void* w3cat, cudaStream_t st);
cudaError_t launch_quant_rows(const void* x, long long rows, int cols, void* q, cudaStream_t st);

// backward.cu -- memory-bound steps of the MoE block's backward (do_prev and du
// are accumulated into: +=)
cudaError_t launch_combine_backward(const float* dO, const float* dOs, const void* y_perm, const int32_t* pos,
                                    const float* topk_w, int T, int d, int k, void* dy_perm, float* dw, void* dS,
                                    float* do_prev, cudaStream_t st);
cudaError_t launch_gather_sum(const void* dx_perm, const int32_t* pos, int T, int d, int k, float* du,
                              cudaStream_t st);
cudaError_t launch_gate_backward(const float* logits, const float* bias, const int32_t* idx, const float* w,
                                 const float* dw, int T, int E, int E_pad, int k, int gate, void* dz,
                                 cudaStream_t st);
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st);
cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t st);   // bytes % 16 == 0
cudaError_t launch_zero(void* dst, size_t bytes, cudaStream_t st);                    // bytes % 16 == 0
// transposed weight packs (mode 0 W13^T, 1 W3^T, 2 W3cat^T, 3 W_R^T) in the tiled layout [G][N'/256][K'/64][256][64]
cudaError_t launch_pack_t(int mode, int G, int Np, int Kp, int c, int d, int cs, int E, const void* a, const void* b,
                          void* out, cudaStream_t st);

}  // namespace fs
