// api.cu -- the C ABI of libfs: argument validation, workspace planning, the
// single-step entry points, the L-block FarSkip drivers (one stream, two
// streams), the FP8 expert path, and the training forward and backward.
//
// "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
// Models" (papercache.org summary): §2.1 (MLP, MoE, router, Dispatch, Combine,
// shared expert) and §3 (FarSkip equation, eq. 8a/8b).  Every step of the
// path runs in this library's kernels; the host side only validates, plans
// buffers inside the caller's workspace and enqueues launches.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fs.h"
#include "common.cuh"
#include "fp8.cuh"
#include "kernels.h"
#include "mx.cuh"

namespace fs {

__device__ int g_fs_dev_error;

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static thread_local char g_last_cuda[256] = "";

static int* g_err_ptr[64] = {nullptr};

int* dev_error_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fs_dev_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

// Three events per device for the two-stream stack, created on first use and
// reused (cudaStreamWaitEvent waits for the most recent record).
static cudaEvent_t g_events[64][3];
static bool g_events_ready[64] = {false};
static std::mutex g_events_mu;

static cudaError_t stack_events(cudaEvent_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_events_mu);
    if (!g_events_ready[dev]) {
        for (int i = 0; i < 3; ++i) {
            e = cudaEventCreateWithFlags(&g_events[dev][i], cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        g_events_ready[dev] = true;
    }
    *out = g_events[dev];
    return cudaSuccess;
}

static fs_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FS_OK;
    std::snprintf(g_last_cuda, sizeof g_last_cuda, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return FS_ERR_CUDA;
}

#define FS_TRY(expr)                               \
    do {                                           \
        cudaError_t e_ = (expr);                   \
        if (e_ != cudaSuccess) return cuda_status(e_); \
    } while (0)

// ------------------------------------------------------------- validation
static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static fs_status check_desc(const fs_layer_desc* d) {
    if (!d) return FS_ERR_INVALID_ARG;
    if (d->T < 1 || d->d < 1 || d->E < 1 || d->k < 1 || d->c < 1 || d->n_shared < 0) return FS_ERR_INVALID_ARG;
    if (d->k > d->E) return FS_ERR_INVALID_ARG;
    if (d->dtype != FS_BF16 && d->dtype != FS_F32 && d->dtype != FS_FP8 && d->dtype != FS_MXFP8)
        return FS_ERR_INVALID_ARG;
    if (d->gate < FS_GATE_SOFTMAX || d->gate > FS_GATE_SIGMOID_NORM) return FS_ERR_INVALID_ARG;
    if (d->n_shared > 0 && d->c_shared < 1) return FS_ERR_INVALID_ARG;
    if (d->d % 64 || d->c % 64) return FS_ERR_UNSUPPORTED;
    if (d->n_shared > 0 && d->c_shared % 64) return FS_ERR_UNSUPPORTED;
    if ((d->dtype == FS_FP8 || d->dtype == FS_MXFP8) &&
        (d->d % 128 || d->c % 128 || (d->n_shared > 0 && d->c_shared % 128)))
        return FS_ERR_UNSUPPORTED;
    if (d->E > kMaxExperts || d->k > kMaxTopK) return FS_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(d->T) * d->k;
    if (rows > 0x7fffffffLL - 1024) return FS_ERR_UNSUPPORTED;
    // MX: the 128-row-padded expert segments must fit the same bound
    if (d->dtype == FS_MXFP8 && rows + 127LL * d->E + 128 > 0x7fffffffLL - 1024) return FS_ERR_UNSUPPORTED;
    return FS_OK;
}

// Activations (GEMM inputs u_k, y_perm, u_next) are bf16 for FS_BF16, FS_FP8
// and FS_MXFP8 (whose expert operands are quantised inside the path), fp32 for
// FS_F32.
static inline int elem_bytes(const fs_layer_desc* d) { return d->dtype == FS_F32 ? 4 : 2; }
static inline int act_dtype(const fs_layer_desc* d) { return d->dtype == FS_F32 ? FS_F32 : FS_BF16; }
static inline bool is_fp8(const fs_layer_desc* d) { return d->dtype == FS_FP8; }
static inline bool is_mx(const fs_layer_desc* d) { return d->dtype == FS_MXFP8; }
static inline int qmode(const fs_layer_desc* d) { return is_fp8(d) ? kQuantRow : (is_mx(d) ? kQuantMx : kQuantNone); }
// Rows of x_perm / y_perm: T k, or with the MX path's 128-row-aligned expert
// segments T k + 127 E rounded up to 128.
static inline long long perm_rows(const fs_layer_desc* d) {
    const long long rows = static_cast<long long>(d->T) * d->k;
    return is_mx(d) ? mx_rows128(rows + 127LL * d->E) : rows;
}

// ------------------------------------------------------------- workspace
struct Layout {
    // single-step regions (L = 0)
    size_t logits, disp, plan_z, plan_r, plan_r2, h_r, hq_r, plan_s, plan_s2, h_s, hq_s, uq, plan_a, end0;
    // stack regions (L >= 1)
    size_t topk_idx, topk_w, counts, offsets, pos, perm, x_perm, y_perm, s_out, ring[3], star[2], ubuf[2], end;
    size_t att, hbuf, abuf[2], end_attn;   // attention wirings only: A_k output, h_k, attention inputs
    int nring, nstar, nu;   // fp32 o_k / o_k* and activation-type u_{k+1} buffers of blocks 1..L-1
};

static Layout layout(const fs_layer_desc* d, int L) {
    const size_t A = 256;
    const size_t es = elem_bytes(d);
    const size_t T = d->T, E = d->E, k = d->k, dm = d->d;
    const size_t rows = T * k;
    const size_t cw = static_cast<size_t>(d->n_shared) * d->c_shared;
    Layout l;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, A); return at; };
    // router logits, or for few tokens the partial sums of its K ranges
    l.logits = take(T * E * 4 * static_cast<size_t>(d->dtype == FS_F32 ? 1 : tc_router_ksplit(d->T, d->E, d->d)));
    l.disp = take(dispatch_ws_bytes(d->T, d->E));
    l.plan_z = take(4 * sizeof(int));
    l.plan_r = take(2 * (E + 1) * sizeof(int));
    l.plan_r2 = take(2 * (E + 1) * sizeof(int));    // the down projection's plan when it runs on CTA pairs
    const bool f8 = is_fp8(d), mxq = is_mx(d);
    const long long prow = perm_rows(d);
    // MX: the hidden goes straight from the gate/up epilogue into an MX matrix
    l.h_r = take(mxq ? mx_rows_bytes(prow, d->c) : rows * d->c * es);
    l.hq_r = take(f8 ? fp8_rows_bytes(static_cast<long long>(rows), d->c) : 0);   // FP8: quantised h
    l.plan_s = take(4 * sizeof(int));
    l.plan_s2 = take(4 * sizeof(int));
    l.h_s = take(mxq ? (cw ? mx_rows_bytes(static_cast<long long>(T), static_cast<int>(cw)) : 0) : T * cw * es);
    l.hq_s = take(f8 && cw ? fp8_rows_bytes(static_cast<long long>(T), static_cast<int>(cw)) : 0);
    l.uq = take(f8 && cw ? fp8_rows_bytes(static_cast<long long>(T), d->d)
                         : (mxq && cw ? mx_rows_bytes(static_cast<long long>(T), d->d) : 0));   // quantised u_k
    l.plan_a = take(4 * sizeof(int));
    l.end0 = o;
    l.topk_idx = take(rows * 4);
    l.topk_w = take(rows * 4);
    l.counts = take(E * 4);
    l.offsets = take((E + 1) * 4);
    l.pos = take(rows * 4);
    l.perm = take(static_cast<size_t>(perm_rows(d)) * 4);
    l.x_perm = take(f8 ? fp8_rows_bytes(static_cast<long long>(rows), d->d)
                       : (mxq ? mx_rows_bytes(prow, d->d) : rows * dm * es));
    l.y_perm = take(static_cast<size_t>(prow) * dm * es);
    l.s_out = take(cw ? T * dm * 4 : 0);     // S in fp32
    // The residual stream between blocks is fp32; the last block writes the
    // caller's outputs.  o_{b-2}, o_{b-1} (and o_{b-1}*) stay live while block
    // b writes, so 3 (2) slots suffice for any L.
    const int nring = L > 1 ? (L - 1 < 3 ? L - 1 : 3) : 0;
    const int nstar = L > 1 ? (L - 1 < 2 ? L - 1 : 2) : 0;
    l.nring = nring;
    l.nstar = nstar;
    l.nu = nstar;
    for (int i = 0; i < 3; ++i) l.ring[i] = i < nring ? take(T * dm * 4) : 0;
    for (int i = 0; i < 2; ++i) l.star[i] = i < nstar ? take(T * dm * 4) : 0;
    for (int i = 0; i < 2; ++i) l.ubuf[i] = i < nstar ? take(T * dm * es) : 0;
    l.end = o;
    l.att = take(T * dm * 4);
    l.hbuf = take(T * dm * 4);
    for (int i = 0; i < 2; ++i) l.abuf[i] = take(T * dm * es);
    l.end_attn = o;
    return l;
}

// Workspace of the two-stream stack: the single-step regions, then two slots
// (blocks alternate) of every per-block buffer the two streams hand over.
struct OverlapLayout {
    size_t end0;
    size_t idx[2], w[2], counts[2], offsets[2], pos[2], perm[2], x_perm[2], s_out[2], ostar[2], oring[2], ubuf[2];
    size_t y_perm, end;
};

static OverlapLayout layout_overlap(const fs_layer_desc* d, int L) {
    const size_t A = 256;
    const size_t es = elem_bytes(d);
    const size_t T = d->T, E = d->E, k = d->k, dm = d->d;
    const size_t rows = T * k;
    const long long prow = perm_rows(d);     // MX: every expert's segment padded to 128 rows
    OverlapLayout l;
    size_t o = layout(d, 0).end0;
    l.end0 = o;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, A); return at; };
    const int slots = L < 2 ? 1 : 2;
    for (int i = 0; i < 2; ++i) {
        const bool on = i < slots;
        l.idx[i] = on ? take(rows * 4) : 0;
        l.w[i] = on ? take(rows * 4) : 0;
        l.counts[i] = on ? take(E * 4) : 0;
        l.offsets[i] = on ? take((E + 1) * 4) : 0;
        l.pos[i] = on ? take(rows * 4) : 0;
        l.perm[i] = on ? take(static_cast<size_t>(prow) * 4) : 0;
        l.x_perm[i] = on ? take(is_fp8(d) ? fp8_rows_bytes(static_cast<long long>(rows), d->d)
                                          : (is_mx(d) ? mx_rows_bytes(prow, d->d) : rows * dm * es))
                         : 0;
        l.s_out[i] = on ? take(T * dm * 4) : 0;
        l.ostar[i] = on ? take(T * dm * 4) : 0;
        l.oring[i] = on ? take(T * dm * 4) : 0;
        l.ubuf[i] = on ? take(T * dm * es) : 0;
    }
    l.y_perm = take(static_cast<size_t>(prow) * dm * es);
    l.end = o;
    return l;
}

static fs_status check_ws(const fs_layer_desc* d, int L, const void* ws, size_t ws_bytes) {
    if (!ws) return FS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return FS_ERR_WORKSPACE;
    const Layout l = layout(d, L);
    if (ws_bytes < (L >= 1 ? l.end : l.end0)) return FS_ERR_WORKSPACE;
    return FS_OK;
}

template <typename T>
static T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

static inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// ------------------------------------------------------------ step bodies
static fs_status router_impl(const fs_layer_desc* d, const void* u, const void* w_r, const float* bias,
                             int32_t* idx, float* w, float* logits, void* ws, cudaStream_t st) {
    const Layout l = layout(d, 0);
    float* z = logits ? logits : at<float>(ws, l.logits);
    int* plan = at<int>(ws, l.plan_z);
    if (d->dtype != FS_F32) {
        const int bm = tc_block_m();
        FS_TRY(launch_plan(nullptr, 1, d->T, bm, plan, st));
        TcExtra ex;
        ex.ksplit = tc_router_ksplit(d->T, d->E, d->d);
        if (ex.ksplit > 1) {
            // few tokens: K ranges on more SMs, partials summed in order by the top-k kernel
            float* zp = at<float>(ws, l.logits);
            FS_TRY(launch_tc_gemm(EPI_F32, u, d->T, w_r, 1, d->E, d->d, plan, ceil_div(d->T, bm) + 1, zp, d->E,
                                  d->E, nullptr, 0, false, st, &ex));
            FS_TRY(launch_topk(zp, ex.ksplit, bias, d->T, d->E, d->k, d->gate, idx, w, logits, st));
            return FS_OK;
        }
        FS_TRY(launch_tc_gemm(EPI_F32, u, d->T, w_r, 1, d->E, d->d, plan, ceil_div(d->T, bm) + 1, z, d->E, d->E,
                              nullptr, 0, false, st));
    } else {
        const int bm = simt_block_m();
        FS_TRY(launch_plan(nullptr, 1, d->T, bm, plan, st));
        FS_TRY(launch_simt_gemm(EPI_F32, static_cast<const float*>(u), d->T, static_cast<const float*>(w_r), 1,
                                d->E, d->d, plan, ceil_div(d->T, bm) + 1, z, d->E, d->E, nullptr, 0, st));
    }
    FS_TRY(launch_topk(z, 1, bias, d->T, d->E, d->k, d->gate, idx, w, nullptr, st));
    return FS_OK;
}

// FS_FP8: x_perm is an FP8 row-scaled matrix; with u_q set the quantised u_k
// is also written there (the shared experts' operand).
static fs_status dispatch_impl(const fs_layer_desc* d, const int32_t* idx, const void* u, int32_t* counts,
                               int32_t* offsets, int32_t* pos, int32_t* perm, void* x_perm, void* ws,
                               cudaStream_t st, void* u_q = nullptr) {
    const Layout l = layout(d, 0);
    FS_TRY(launch_dispatch(idx, u, d->T, d->d, d->E, d->k, elem_bytes(d), counts, offsets, pos, perm, x_perm,
                           at<int32_t>(ws, l.disp), st, qmode(d), qmode(d) != kQuantNone ? u_q : nullptr,
                           perm_rows(d)));
    return FS_OK;
}

// Two grouped GEMMs over `rows` rows split into G groups by `offsets`
// (nullptr = one group): h = SiLU(x W2^T) * (x W1^T), then y = h W3^T, with
// y stored in the activation type (y_f32 = false) or in fp32.  With gather
// non-null, GEMM row p reads row gather[p] of x (x has x_rows rows): the
// Dispatch permutation applied inside the first GEMM's operand loads.
// FS_FP8: x is an FP8 row-scaled matrix [x_rows, d], the weights FP8 packs; h
// (bf16) is quantised per row into hq before the down GEMM.
// With cmb set (one group over the T token rows, tensor-core dtypes) the down
// projection's epilogue is Combine fused with the FarSkip update (y unused).
// plan2 (nullable): room for a second plan, used when one of the two GEMMs runs
// on the CTA-pair kernel (tc_down_pair, tc_up_pair) and the other does not.
static fs_status swiglu_impl(const fs_layer_desc* d, const void* x, long long x_rows, const int32_t* gather, int rows,
                             const int32_t* offsets, int G, int cw, const void* w13, const void* w3, void* y,
                             bool y_f32, int* plan, void* h, void* hq, cudaStream_t st, void* gu_save = nullptr,
                             const CombineEpi* cmb = nullptr, int* plan2 = nullptr) {
    // down (dp) or gate/up (up) projection on CTA pairs: its own plan of 256-row tiles
    const bool dp = plan2 && tc_down_pair() && tc_block_m() == 128;
    const bool up = plan2 && tc_up_pair() && tc_block_m() == 128 && !gather;
    const int max_mt2 = ceil_div(rows, 256) + G;
    if (is_mx(d)) {
        // x: an MX matrix of x_rows rows (a multiple of 128 or the token count);
        // groups start at multiples of 128; the hidden is written as an MX matrix
        const long long xr = mx_rows128(x_rows);
        const int max_mt = ceil_div(xr, 128) + G;
        const uint8_t* xs = static_cast<const uint8_t*>(x) + mx_sf_offset(xr, d->d);
        uint8_t* hc = static_cast<uint8_t*>(h);
        uint8_t* hs = hc + mx_sf_offset(xr, cw);
        FS_TRY(launch_plan(offsets, G, offsets ? static_cast<int>(xr) : rows, 128, plan, st));
        FS_TRY(launch_mx_gemm(EPI_SWIGLU, x, xr, xs, w13, packed_sf_mx(w13, G, 2 * cw, d->d), G, 2 * cw, d->d, plan,
                              max_mt, hc, cw, cw, hs, st));
        FS_TRY(launch_mx_gemm(y_f32 ? EPI_F32 : EPI_BF16, hc, xr, hs, w3, packed_sf_mx(w3, G, d->d, cw), G, d->d, cw,
                              plan, max_mt, y, d->d, d->d, nullptr, st));
    } else if (is_fp8(d)) {
        const int bm = tc_block_m_f8();
        const int max_mt = ceil_div(rows, bm) + G;
        const float* xs = reinterpret_cast<const float*>(static_cast<const uint8_t*>(x) + fp8_scale_offset(x_rows, d->d));
        const float* hs = reinterpret_cast<const float*>(static_cast<const uint8_t*>(hq) + fp8_scale_offset(rows, cw));
        FS_TRY(launch_plan(offsets, G, rows, bm, plan, st));
        if (dp || up) FS_TRY(launch_plan(offsets, G, rows, 256, plan2, st));
        FS_TRY(launch_tc_gemm_f8(EPI_SWIGLU, x, x_rows, xs, w13, packed_scales_fp8(w13, G, 2 * cw, d->d), G, 2 * cw,
                                 d->d, up ? plan2 : plan, up ? max_mt2 : max_mt, h, cw, cw, st, nullptr,
                                 up ? 1 : -1));
        FS_TRY(launch_quant_rows(h, rows, cw, hq, st));
        FS_TRY(launch_tc_gemm_f8(cmb ? EPI_COMBINE : (y_f32 ? EPI_F32 : EPI_BF16), hq, rows, hs, w3,
                                 packed_scales_fp8(w3, G, d->d, cw), G, d->d, cw, dp ? plan2 : plan,
                                 dp ? max_mt2 : max_mt, y, d->d, d->d, st, cmb, dp ? 1 : -1));
    } else if (d->dtype == FS_BF16) {
        const int bm = tc_block_m();
        const int max_mt = ceil_div(rows, bm) + G;
        FS_TRY(launch_plan(offsets, G, rows, bm, plan, st));
        if (dp || up) FS_TRY(launch_plan(offsets, G, rows, 256, plan2, st));
        TcExtra ex;
        ex.aux = gu_save;            // training forward: keep the pre-activations for the backward
        ex.aux_ld = 2LL * cw;
        if (up) ex.variant = 1;
        FS_TRY(launch_tc_gemm(EPI_SWIGLU, x, x_rows, w13, G, 2 * cw, d->d, up ? plan2 : plan, up ? max_mt2 : max_mt,
                              h, cw, cw, gather, rows, true, st, &ex));
        TcExtra ex2;
        ex2.combine = cmb;
        if (dp) ex2.variant = 1;
        FS_TRY(launch_tc_gemm(cmb ? EPI_COMBINE : (y_f32 ? EPI_F32 : EPI_BF16), h, rows, w3, G, d->d, cw,
                              dp ? plan2 : plan, dp ? max_mt2 : max_mt, y, d->d, d->d, nullptr, 0, true, st, &ex2));
    } else {
        const int bm = simt_block_m();
        const int max_mt = ceil_div(rows, bm) + G;
        FS_TRY(launch_plan(offsets, G, rows, bm, plan, st));
        FS_TRY(launch_simt_gemm(EPI_SWIGLU, static_cast<const float*>(x), x_rows, static_cast<const float*>(w13), G,
                                2 * cw, d->d, plan, max_mt, static_cast<float*>(h), cw, cw, gather, rows, st));
        FS_TRY(launch_simt_gemm(EPI_F32, static_cast<const float*>(h), rows, static_cast<const float*>(w3), G, d->d,
                                cw, plan, max_mt, static_cast<float*>(y), d->d, d->d, nullptr, 0, st));
    }
    return FS_OK;
}

static fs_status routed_impl(const fs_layer_desc* d, const void* x_perm, const int32_t* offsets, const void* w13,
                             const void* w3, void* y_perm, void* ws, cudaStream_t st) {
    const Layout l = layout(d, 0);
    const int rows = static_cast<int>(perm_rows(d));
    return swiglu_impl(d, x_perm, rows, nullptr, rows, offsets, d->E, d->c, w13, w3, y_perm, false,
                       at<int>(ws, l.plan_r), at<void>(ws, l.h_r), at<void>(ws, l.hq_r), st, nullptr, nullptr,
                       at<int>(ws, l.plan_r2));
}

static fs_status routed_gather_impl(const fs_layer_desc* d, const void* u, const int32_t* perm_src,
                                    const int32_t* offsets, const void* w13, const void* w3, void* y_perm, void* ws,
                                    cudaStream_t st) {
    const Layout l = layout(d, 0);
    return swiglu_impl(d, u, d->T, perm_src, d->T * d->k, offsets, d->E, d->c, w13, w3, y_perm, false,
                       at<int>(ws, l.plan_r), at<void>(ws, l.h_r), nullptr, st);
}

// FS_FP8: the GEMMs read the quantised u_k in ws (written by the stack's
// Dispatch when u_q_ready, else quantised here from u).
static fs_status shared_impl(const fs_layer_desc* d, const void* u, const void* w13s, const void* w3s, void* s_out,
                             void* ws, cudaStream_t st, bool u_q_ready = false, const CombineEpi* cmb = nullptr) {
    const Layout l = layout(d, 0);
    const void* x = u;
    if (is_fp8(d)) {
        x = at<void>(ws, l.uq);
        if (!u_q_ready) FS_TRY(launch_quant_rows(u, d->T, d->d, at<void>(ws, l.uq), st));
    } else if (is_mx(d)) {
        x = at<void>(ws, l.uq);
        if (!u_q_ready) FS_TRY(launch_quant_rows_mx(u, d->T, d->d, at<void>(ws, l.uq), st));
    }
    return swiglu_impl(d, x, d->T, nullptr, d->T, nullptr, 1, d->n_shared * d->c_shared, w13s, w3s, s_out, true,
                       at<int>(ws, l.plan_s), at<void>(ws, l.h_s), at<void>(ws, l.hq_s), st, nullptr, cmb,
                       at<int>(ws, l.plan_s2));
}

// The shared experts with Combine and the FarSkip update in the epilogue of
// their down projection (tensor-core dtypes, k <= 8): the same results as
// shared_impl followed by combine_impl, without the fp32 S in memory.
static bool fused_combine_ok(const fs_layer_desc* d) {
    return (d->dtype == FS_BF16 || d->dtype == FS_FP8) && d->n_shared > 0 && d->k <= kCombineEpiMaxK;
}

static fs_status shared_combine_impl(const fs_layer_desc* d, const void* u, const void* w13s, const void* w3s,
                                     const void* y_perm, const int32_t* pos, const float* w, const void* o_prev,
                                     int prev_dtype, void* o_partial, void* o_full, int out_dtype, void* u_next,
                                     int wiring, void* ws, cudaStream_t st, bool u_q_ready = false) {
    CombineEpi cmb;
    cmb.y_perm = y_perm;
    cmb.pos = pos;
    cmb.topk_w = w;
    cmb.k = d->k;
    cmb.o_prev = o_prev;
    cmb.prev_bf16 = prev_dtype == FS_BF16;
    cmb.o_partial = o_partial;
    cmb.o_full = o_full;
    cmb.out_bf16 = out_dtype == FS_BF16;
    cmb.u_next = u_next;
    cmb.u_src = wiring == FS_WIRE_PARTIAL ? 0 : (wiring == FS_WIRE_OUTDATED ? 1 : 2);
    return shared_impl(d, u, w13s, w3s, nullptr, ws, st, u_q_ready, &cmb);
}

static fs_status combine_impl(const fs_layer_desc* d, const void* y_perm, const int32_t* pos, const float* w,
                              const void* o_prev, int prev_dtype, const void* s, const float* extra, void* o_partial,
                              void* o_full, int out_dtype, void* u_next, int u_src, void* u_full, cudaStream_t st,
                              int k_override = -1) {
    FS_TRY(launch_combine(y_perm, pos, w, o_prev, prev_dtype == FS_BF16, s, extra, o_partial, o_full,
                          out_dtype == FS_BF16, u_next, u_src, u_full, d->T, d->d, k_override >= 0 ? k_override : d->k,
                          d->dtype != FS_F32, st));
    return FS_OK;
}

// Stand-in attention sub-block: out (fp32) = a W_att^T, a per-token dense GEMM.
static fs_status attn_impl(const fs_layer_desc* d, const void* a, const void* w_att, float* out, void* ws,
                           cudaStream_t st) {
    const Layout l = layout(d, 0);
    int* plan = at<int>(ws, l.plan_a);
    if (d->dtype != FS_F32) {
        const int bm = tc_block_m();
        FS_TRY(launch_plan(nullptr, 1, d->T, bm, plan, st));
        FS_TRY(launch_tc_gemm(EPI_F32, a, d->T, w_att, 1, d->d, d->d, plan, ceil_div(d->T, bm) + 1, out, d->d, d->d,
                              nullptr, 0, false, st));
    } else {
        const int bm = simt_block_m();
        FS_TRY(launch_plan(nullptr, 1, d->T, bm, plan, st));
        FS_TRY(launch_simt_gemm(EPI_F32, static_cast<const float*>(a), d->T, static_cast<const float*>(w_att), 1,
                                d->d, d->d, plan, ceil_div(d->T, bm) + 1, out, d->d, d->d, nullptr, 0, st));
    }
    return FS_OK;
}

}  // namespace fs

using namespace fs;

#define FS_CHECK(expr)              \
    do {                            \
        fs_status s_ = (expr);      \
        if (s_ != FS_OK) return s_; \
    } while (0)

static fs_status need(const void* p) {
    if (!p) return FS_ERR_INVALID_ARG;
    return aligned16(p) ? FS_OK : FS_ERR_UNSUPPORTED;
}

extern "C" {

size_t fs_workspace_bytes(const fs_layer_desc* desc, int L) {
    if (check_desc(desc) != FS_OK || L < 0) return 0;
    const Layout l = layout(desc, L);
    return L >= 1 ? l.end : l.end0;
}

size_t fs_workspace_bytes_attn(const fs_layer_desc* desc, int L) {
    if (check_desc(desc) != FS_OK || L < 1) return 0;
    return layout(desc, L).end_attn;
}

size_t fs_workspace_bytes_overlap(const fs_layer_desc* desc, int L) {
    if (check_desc(desc) != FS_OK || L < 1) return 0;
    return layout_overlap(desc, L).end;
}

static inline bool valid_dtype(int32_t t) { return t == FS_BF16 || t == FS_F32 || t == FS_FP8 || t == FS_MXFP8; }

fs_status fs_pack_w13(int32_t G, int32_t c, int32_t d, int32_t dtype, const void* w1, const void* w2, void* w13,
                      void* stream) {
    if (G < 1 || c < 1 || d < 1 || !valid_dtype(dtype)) return FS_ERR_INVALID_ARG;
    const int q = (dtype == FS_FP8 || dtype == FS_MXFP8) ? 128 : 64;
    if (c % q || d % q) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w1));
    FS_CHECK(need(w2));
    FS_CHECK(need(w13));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == FS_MXFP8)
        FS_TRY(launch_pack_w13_mx(G, c, d, w1, w2, w13, st));
    else if (dtype == FS_FP8)
        FS_TRY(launch_pack_w13_fp8(G, c, d, w1, w2, w13, st));
    else
        FS_TRY(launch_pack_w13(G, c, d, dtype == FS_BF16 ? 2 : 4, w1, w2, w13, st));
    return FS_OK;
}

size_t fs_packed_bytes(int32_t G, int32_t N, int32_t K, int32_t dtype) {
    if (G < 1 || N < 1 || K < 1 || K % 64 || !valid_dtype(dtype)) return 0;
    if (dtype == FS_FP8) return K % 128 ? 0 : packed_bytes_fp8(G, N, K);
    if (dtype == FS_MXFP8) return (K % 128 || N % 128) ? 0 : packed_bytes_mx(G, N, K);
    return packed_bytes(G, N, K, dtype == FS_BF16 ? 2 : 4);
}

fs_status fs_pack_w3(int32_t G, int32_t d, int32_t c, int32_t dtype, const void* w3, void* w3p, void* stream) {
    if (G < 1 || c < 1 || d < 1 || !valid_dtype(dtype)) return FS_ERR_INVALID_ARG;
    const int q = (dtype == FS_FP8 || dtype == FS_MXFP8) ? 128 : 64;
    if (c % q || d % q) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w3));
    FS_CHECK(need(w3p));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == FS_MXFP8)
        FS_TRY(launch_pack_w3_mx(G, d, c, w3, w3p, st));
    else if (dtype == FS_FP8)
        FS_TRY(launch_pack_w3_fp8(G, d, c, w3, w3p, st));
    else
        FS_TRY(launch_pack_w3(G, d, c, dtype == FS_BF16 ? 2 : 4, w3, w3p, st));
    return FS_OK;
}

fs_status fs_pack_w3_shared(int32_t n_shared, int32_t c_shared, int32_t d, int32_t dtype, const void* w3s,
                            void* w3cat, void* stream) {
    if (n_shared < 1 || c_shared < 1 || d < 1 || !valid_dtype(dtype)) return FS_ERR_INVALID_ARG;
    const int q = (dtype == FS_FP8 || dtype == FS_MXFP8) ? 128 : 64;
    if (c_shared % q || d % q) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w3s));
    FS_CHECK(need(w3cat));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == FS_MXFP8)
        FS_TRY(launch_pack_w3_shared_mx(n_shared, c_shared, d, w3s, w3cat, st));
    else if (dtype == FS_FP8)
        FS_TRY(launch_pack_w3_shared_fp8(n_shared, c_shared, d, w3s, w3cat, st));
    else
        FS_TRY(launch_pack_w3_shared(n_shared, c_shared, d, dtype == FS_BF16 ? 2 : 4, w3s, w3cat, st));
    return FS_OK;
}

size_t fs_fp8_rows_bytes(int64_t rows, int32_t cols) {
    if (rows < 1 || cols < 1) return 0;
    return fp8_rows_bytes(rows, cols);
}

fs_status fs_quantize_rows_fp8(int64_t rows, int32_t cols, const void* x, void* q, void* stream) {
    if (rows < 1 || cols < 1) return FS_ERR_INVALID_ARG;
    if (cols % 128 || rows > 0x7fffffffLL) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(x));
    FS_CHECK(need(q));
    FS_TRY(launch_quant_rows(x, rows, cols, q, static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

size_t fs_mx_rows_bytes(int64_t rows, int32_t cols) {
    if (rows < 1 || cols < 1 || cols % 128) return 0;
    return mx_rows_bytes(rows, cols);
}

fs_status fs_quantize_rows_mx(int64_t rows, int32_t cols, const void* x, void* q, void* stream) {
    if (rows < 1 || cols < 1) return FS_ERR_INVALID_ARG;
    if (cols % 128 || rows > 0x7fffffffLL) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(x));
    FS_CHECK(need(q));
    FS_TRY(launch_quant_rows_mx(x, rows, cols, q, static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

int64_t fs_dispatch_rows(const fs_layer_desc* desc) {
    if (check_desc(desc) != FS_OK) return 0;
    return perm_rows(desc);
}

fs_status fs_router_topk(const fs_layer_desc* desc, const void* u, const void* w_r, const float* bias,
                         int32_t* topk_idx, float* topk_w, float* logits, void* ws, size_t ws_bytes, void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(u));
    FS_CHECK(need(w_r));
    FS_CHECK(need(topk_idx));
    FS_CHECK(need(topk_w));
    if (bias && !aligned16(bias)) return FS_ERR_UNSUPPORTED;
    if (logits && !aligned16(logits)) return FS_ERR_UNSUPPORTED;
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    return router_impl(desc, u, w_r, bias, topk_idx, topk_w, logits, ws, static_cast<cudaStream_t>(stream));
}

fs_status fs_dispatch(const fs_layer_desc* desc, const int32_t* topk_idx, const void* u, int32_t* counts,
                      int32_t* offsets, int32_t* pos, int32_t* perm_src, void* x_perm, void* ws, size_t ws_bytes,
                      void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(topk_idx));
    FS_CHECK(need(u));
    FS_CHECK(need(counts));
    FS_CHECK(need(offsets));
    FS_CHECK(need(pos));
    FS_CHECK(need(perm_src));
    if (x_perm && !aligned16(x_perm)) return FS_ERR_UNSUPPORTED;
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    return dispatch_impl(desc, topk_idx, u, counts, offsets, pos, perm_src, x_perm, ws,
                         static_cast<cudaStream_t>(stream));
}

fs_status fs_dispatch_noalloc(const fs_layer_desc* desc, const int32_t* topk_idx, const void* u, int32_t* counts,
                              int32_t* offsets, int32_t* pos, int32_t* perm_src, void* x_perm, void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(topk_idx));
    FS_CHECK(need(u));
    FS_CHECK(need(counts));
    FS_CHECK(need(offsets));
    FS_CHECK(need(pos));
    FS_CHECK(need(perm_src));
    if (x_perm && !aligned16(x_perm)) return FS_ERR_UNSUPPORTED;
    if (dispatch_ws_bytes(desc->T, desc->E) > static_cast<size_t>(kStaticDispatchScratchInts) * sizeof(int32_t)) {
        std::snprintf(g_last_cuda, sizeof g_last_cuda,
                      "fs_dispatch_noalloc: ceil(T/1024) * E = %zu scratch ints exceed the static maximum %d",
                      dispatch_ws_bytes(desc->T, desc->E) / sizeof(int32_t), kStaticDispatchScratchInts);
        return FS_ERR_WORKSPACE;
    }
    FS_TRY(launch_dispatch_noalloc(topk_idx, u, desc->T, desc->d, desc->E, desc->k, elem_bytes(desc), counts, offsets,
                                   pos, perm_src, x_perm, static_cast<cudaStream_t>(stream), qmode(desc),
                                   perm_rows(desc)));
    return FS_OK;
}

fs_status fs_grouped_swiglu(const fs_layer_desc* desc, const void* x_perm, const int32_t* offsets, const void* w13,
                            const void* w3, void* y_perm, void* ws, size_t ws_bytes, void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(x_perm));
    FS_CHECK(need(offsets));
    FS_CHECK(need(w13));
    FS_CHECK(need(w3));
    FS_CHECK(need(y_perm));
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    return routed_impl(desc, x_perm, offsets, w13, w3, y_perm, ws, static_cast<cudaStream_t>(stream));
}

fs_status fs_grouped_swiglu_gather(const fs_layer_desc* desc, const void* u, const int32_t* perm_src,
                                   const int32_t* offsets, const void* w13, const void* w3, void* y_perm, void* ws,
                                   size_t ws_bytes, void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(u));
    FS_CHECK(need(perm_src));
    FS_CHECK(need(offsets));
    FS_CHECK(need(w13));
    FS_CHECK(need(w3));
    FS_CHECK(need(y_perm));
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    if (is_fp8(desc) || is_mx(desc)) return FS_ERR_UNSUPPORTED;
    if (desc->dtype == FS_BF16 && !tc_gather_supported()) return FS_ERR_UNSUPPORTED;
    return routed_gather_impl(desc, u, perm_src, offsets, w13, w3, y_perm, ws, static_cast<cudaStream_t>(stream));
}

fs_status fs_shared_expert(const fs_layer_desc* desc, const void* u, const void* w13_shared, const void* w3_shared,
                           void* s_out, void* ws, size_t ws_bytes, void* stream) {
    FS_CHECK(check_desc(desc));
    if (desc->n_shared < 1) return FS_ERR_INVALID_ARG;
    FS_CHECK(need(u));
    FS_CHECK(need(w13_shared));
    FS_CHECK(need(w3_shared));
    FS_CHECK(need(s_out));
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    return shared_impl(desc, u, w13_shared, w3_shared, s_out, ws, static_cast<cudaStream_t>(stream));
}

fs_status fs_combine(const fs_layer_desc* desc, const void* y_perm, const int32_t* pos, const float* topk_w,
                     const void* o_prev, int32_t prev_dtype, const void* shared_out, const float* extra,
                     void* o_partial, void* o_full, int32_t out_dtype, void* u_next, int32_t wiring, void* u_full,
                     void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(y_perm));
    FS_CHECK(need(pos));
    FS_CHECK(need(topk_w));
    FS_CHECK(need(o_prev));
    FS_CHECK(need(o_full));
    if ((prev_dtype != FS_BF16 && prev_dtype != FS_F32) || (out_dtype != FS_BF16 && out_dtype != FS_F32))
        return FS_ERR_INVALID_ARG;
    if (u_next && (wiring < FS_WIRE_PARTIAL || wiring > FS_WIRE_DISABLED)) return FS_ERR_INVALID_ARG;
    if (shared_out && !aligned16(shared_out)) return FS_ERR_UNSUPPORTED;
    if (o_partial && !aligned16(o_partial)) return FS_ERR_UNSUPPORTED;
    if (u_next && !aligned16(u_next)) return FS_ERR_UNSUPPORTED;
    if (u_full && !aligned16(u_full)) return FS_ERR_UNSUPPORTED;
    if (extra && !aligned16(extra)) return FS_ERR_UNSUPPORTED;
    return combine_impl(desc, y_perm, pos, topk_w, o_prev, prev_dtype, shared_out, extra, o_partial, o_full,
                        out_dtype, u_next, wiring, u_full, static_cast<cudaStream_t>(stream));
}

fs_status fs_shared_expert_combine(const fs_layer_desc* desc, const void* u, const void* w13_shared,
                                   const void* w3_shared, const void* y_perm, const int32_t* pos, const float* topk_w,
                                   const void* o_prev, int32_t prev_dtype, void* o_partial, void* o_full,
                                   int32_t out_dtype, void* u_next, int32_t wiring, void* ws, size_t ws_bytes,
                                   void* stream) {
    FS_CHECK(check_desc(desc));
    if (desc->n_shared < 1) return FS_ERR_INVALID_ARG;
    FS_CHECK(need(u));
    FS_CHECK(need(w13_shared));
    FS_CHECK(need(w3_shared));
    FS_CHECK(need(y_perm));
    FS_CHECK(need(pos));
    FS_CHECK(need(topk_w));
    FS_CHECK(need(o_prev));
    FS_CHECK(need(o_full));
    if ((prev_dtype != FS_BF16 && prev_dtype != FS_F32) || (out_dtype != FS_BF16 && out_dtype != FS_F32))
        return FS_ERR_INVALID_ARG;
    if (u_next && (wiring < FS_WIRE_PARTIAL || wiring > FS_WIRE_DISABLED)) return FS_ERR_INVALID_ARG;
    if (o_partial && !aligned16(o_partial)) return FS_ERR_UNSUPPORTED;
    if (u_next && !aligned16(u_next)) return FS_ERR_UNSUPPORTED;
    if (!fused_combine_ok(desc)) return FS_ERR_UNSUPPORTED;
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    return shared_combine_impl(desc, u, w13_shared, w3_shared, y_perm, pos, topk_w, o_prev, prev_dtype, o_partial,
                               o_full, out_dtype, u_next, wiring, ws, static_cast<cudaStream_t>(stream));
}

fs_status fs_attn_standin(const fs_layer_desc* desc, const void* a, const void* w_att, float* out, void* ws,
                          size_t ws_bytes, void* stream) {
    FS_CHECK(check_desc(desc));
    FS_CHECK(need(a));
    FS_CHECK(need(w_att));
    FS_CHECK(need(out));
    FS_CHECK(check_ws(desc, 0, ws, ws_bytes));
    return attn_impl(desc, a, w_att, out, ws, static_cast<cudaStream_t>(stream));
}

fs_status fs_farskip_stack(const fs_layer_desc* desc, int32_t L, int32_t wiring, const fs_block_weights* blocks,
                           const void* x, void* o_full, void* o_partial, void* ws, size_t ws_bytes, void* stream) {
    FS_CHECK(check_desc(desc));
    if (L < 1 || !blocks) return FS_ERR_INVALID_ARG;
    if (wiring < FS_WIRE_PARTIAL || wiring > FS_WIRE_ATTN_PLAIN) return FS_ERR_INVALID_ARG;
    const bool attn = wiring == FS_WIRE_ATTN_FARSKIP || wiring == FS_WIRE_ATTN_PLAIN;
    FS_CHECK(need(x));
    FS_CHECK(need(o_full));
    if (o_partial && !aligned16(o_partial)) return FS_ERR_UNSUPPORTED;
    for (int b = 0; b < L; ++b) {
        FS_CHECK(need(blocks[b].w_r));
        FS_CHECK(need(blocks[b].w13));
        FS_CHECK(need(blocks[b].w3));
        if (blocks[b].bias && !aligned16(blocks[b].bias)) return FS_ERR_UNSUPPORTED;
        if (desc->n_shared > 0) {
            FS_CHECK(need(blocks[b].w13_shared));
            FS_CHECK(need(blocks[b].w3_shared));
        }
        if (attn) FS_CHECK(need(blocks[b].w_att));
    }
    FS_CHECK(check_ws(desc, L, ws, ws_bytes));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Layout l = layout(desc, L);
    if (attn && ws_bytes < l.end_attn) return FS_ERR_WORKSPACE;
    int32_t* idx = at<int32_t>(ws, l.topk_idx);
    float* w = at<float>(ws, l.topk_w);
    int32_t* counts = at<int32_t>(ws, l.counts);
    int32_t* offsets = at<int32_t>(ws, l.offsets);
    int32_t* pos = at<int32_t>(ws, l.pos);
    int32_t* perm = at<int32_t>(ws, l.perm);
    void* x_perm = at<void>(ws, l.x_perm);
    void* y_perm = at<void>(ws, l.y_perm);
    void* s_out = desc->n_shared > 0 ? at<void>(ws, l.s_out) : nullptr;

    // The stack copies rows in Dispatch: gathering them inside the gate/up GEMM
    // (tile::gather4 moves 512 B per TMA op) is issue-bound on the tensor-core
    // path, and the separate copy runs near HBM peak.
    const void* u = x;        // u_k   (= o_{k-1}* in the page's notation), activation type
    const void* o_prev = x;   // o_{k-1}: the caller's x for k = 1, then the fp32 residual stream
    const void* a_in = x;     // attention input (attention wirings), activation type
    int prev_dtype = act_dtype(desc);
    float* att = at<float>(ws, l.att);
    void* u_q = qmode(desc) != kQuantNone && desc->n_shared > 0 ? at<void>(ws, layout(desc, 0).uq) : nullptr;
    for (int b = 1; b <= L; ++b) {
        const fs_block_weights& bw = blocks[b - 1];
        const bool last = (b == L);
        void* o_k = last ? o_full : at<void>(ws, l.ring[(b - 1) % l.nring]);
        void* os_k = last ? o_partial : nullptr;      // o_k* of an inner block is not read again
        void* u_next = last ? nullptr : at<void>(ws, l.ubuf[(b - 1) % l.nu]);
        void* a_next = last ? nullptr : at<void>(ws, l.abuf[(b - 1) & 1]);
        const int out_dtype = last ? act_dtype(desc) : FS_F32;
        const void* base = o_prev;          // residual the MoE outputs are added to
        int base_dtype = prev_dtype;
        const float* extra = nullptr;
        if (attn) {
            FS_CHECK(attn_impl(desc, a_in, bw.w_att, att, ws, st));
            if (wiring == FS_WIRE_ATTN_PLAIN) {
                // h_k = o_{k-1} + A_k(o_{k-1}) (fp32) and the MoE input bf16(h_k)
                float* h = at<float>(ws, l.hbuf);
                void* m_in = at<void>(ws, l.abuf[b & 1]);
                FS_CHECK(combine_impl(desc, nullptr, nullptr, nullptr, o_prev, prev_dtype, nullptr, att, nullptr, h,
                                      FS_F32, m_in, FS_WIRE_PARTIAL, nullptr, st, 0));
                u = m_in;
                base = h;
                base_dtype = FS_F32;
            } else {
                extra = att;                // o_k = o_{k-1} + A_k(attn-in_k) + S_k + R_k
            }
        }
        FS_CHECK(router_impl(desc, u, bw.w_r, bw.bias, idx, w, nullptr, ws, st));
        FS_CHECK(dispatch_impl(desc, idx, u, counts, offsets, pos, perm, x_perm, ws, st, u_q));
        FS_CHECK(routed_impl(desc, x_perm, offsets, bw.w13, bw.w3, y_perm, ws, st));
        // The shared experts then Combine as two passes: Combine in the shared down
        // projection's epilogue (fs_shared_expert_combine) measured slower at
        // DeepSeek-V3's shapes -- its per-row gathers from eight epilogue warps per
        // SM keep too few loads in flight next to the standalone kernel.
        if (s_out) FS_CHECK(shared_impl(desc, u, bw.w13_shared, bw.w3_shared, s_out, ws, st, u_q != nullptr));
        if (wiring == FS_WIRE_ATTN_FARSKIP) {
            // next attention input bf16(o_k*) = bf16(o_k - R_k), next MoE input bf16(o_k)
            FS_CHECK(combine_impl(desc, y_perm, pos, w, base, base_dtype, s_out, extra, os_k, o_k, out_dtype, a_next,
                                  FS_WIRE_PARTIAL, u_next, st));
            a_in = a_next;
            u = u_next;
        } else if (wiring == FS_WIRE_ATTN_PLAIN) {
            // o_k = h_k + S_k + R_k; next attention input bf16(o_k)
            FS_CHECK(combine_impl(desc, y_perm, pos, w, base, base_dtype, s_out, nullptr, os_k, o_k, out_dtype,
                                  nullptr, FS_WIRE_PARTIAL, a_next, st));
            a_in = a_next;
        } else {
            FS_CHECK(combine_impl(desc, y_perm, pos, w, o_prev, prev_dtype, s_out, nullptr, os_k, o_k, out_dtype,
                                  u_next, wiring, nullptr, st));
            u = u_next;
        }
        o_prev = o_k;
        prev_dtype = out_dtype;
    }
    return FS_OK;
}

fs_status fs_farskip_stack_overlap(const fs_layer_desc* desc, int32_t L, int32_t wiring,
                                   const fs_block_weights* blocks, const void* x, void* o_full, void* o_partial,
                                   void* ws, size_t ws_bytes, void* stream, void* stream2) {
    FS_CHECK(check_desc(desc));
    if (L < 1 || !blocks) return FS_ERR_INVALID_ARG;
    if (wiring != FS_WIRE_PARTIAL && wiring != FS_WIRE_OUTDATED) return FS_ERR_INVALID_ARG;
    if (!stream2 || stream2 == stream) return FS_ERR_INVALID_ARG;
    FS_CHECK(need(x));
    FS_CHECK(need(o_full));
    if (o_partial && !aligned16(o_partial)) return FS_ERR_UNSUPPORTED;
    for (int b = 0; b < L; ++b) {
        FS_CHECK(need(blocks[b].w_r));
        FS_CHECK(need(blocks[b].w13));
        FS_CHECK(need(blocks[b].w3));
        if (blocks[b].bias && !aligned16(blocks[b].bias)) return FS_ERR_UNSUPPORTED;
        if (desc->n_shared > 0) {
            FS_CHECK(need(blocks[b].w13_shared));
            FS_CHECK(need(blocks[b].w3_shared));
        }
    }
    if (!ws) return FS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return FS_ERR_WORKSPACE;
    const OverlapLayout l = layout_overlap(desc, L);
    if (ws_bytes < l.end) return FS_ERR_WORKSPACE;
    cudaEvent_t* ev = nullptr;
    FS_TRY(stack_events(&ev));
    cudaEvent_t evD = ev[0], evU = ev[1], evA = ev[2];
    cudaStream_t sa = static_cast<cudaStream_t>(stream);     // routed experts + combine
    cudaStream_t sb = static_cast<cudaStream_t>(stream2);    // router, dispatch, shared expert, o_k*
    const int act = act_dtype(desc);
    void* y_perm = at<void>(ws, l.y_perm);
    // FP8 / MX: Dispatch also writes the quantised u_k for the shared experts (both on stream2)
    void* u_q = qmode(desc) != kQuantNone && desc->n_shared > 0 ? at<void>(ws, layout(desc, 0).uq) : nullptr;

    // fork: stream2 starts after everything already queued on stream (x ready)
    FS_TRY(cudaEventRecord(evA, sa));
    FS_TRY(cudaStreamWaitEvent(sb, evA, 0));
    const void* u = x;          // u_k, activation type
    const void* o_prev = x;     // o_{k-1}
    int prev_dtype = act;
    for (int b = 1; b <= L; ++b) {
        const fs_block_weights& bw = blocks[b - 1];
        const int sl = (b - 1) & 1;
        const bool last = (b == L);
        int32_t* idx = at<int32_t>(ws, l.idx[sl]);
        float* w = at<float>(ws, l.w[sl]);
        int32_t* counts = at<int32_t>(ws, l.counts[sl]);
        int32_t* offsets = at<int32_t>(ws, l.offsets[sl]);
        int32_t* pos = at<int32_t>(ws, l.pos[sl]);
        int32_t* perm = at<int32_t>(ws, l.perm[sl]);
        void* x_perm = at<void>(ws, l.x_perm[sl]);
        float* s_out = desc->n_shared > 0 ? at<float>(ws, l.s_out[sl]) : nullptr;
        float* ostar = at<float>(ws, l.ostar[sl]);
        void* o_k = last ? o_full : at<void>(ws, l.oring[sl]);
        void* u_next = last ? nullptr : at<void>(ws, l.ubuf[sl]);
        // ---- stream2: everything of block b that does not need the routed experts
        FS_CHECK(router_impl(desc, u, bw.w_r, bw.bias, idx, w, nullptr, ws, sb));
        FS_CHECK(dispatch_impl(desc, idx, u, counts, offsets, pos, perm, x_perm, ws, sb, u_q));
        FS_TRY(cudaEventRecord(evD, sb));
        if (s_out) FS_CHECK(shared_impl(desc, u, bw.w13_shared, bw.w3_shared, s_out, ws, sb, u_q != nullptr));
        if (b > 1) FS_TRY(cudaStreamWaitEvent(sb, evA, 0));       // o_{b-1} from block b-1's combine
        // o_b* = o_{b-1} + S_b (fp32) and the next input (partial: o_b*, outdated: o_{b-1})
        FS_TRY(launch_combine(nullptr, nullptr, nullptr, o_prev, prev_dtype == FS_BF16, s_out, nullptr, nullptr, ostar,
                              0, u_next, wiring, nullptr, desc->T, desc->d, 0, act == FS_BF16, sb));
        FS_TRY(cudaEventRecord(evU, sb));
        // ---- stream: the routed experts, then o_b = o_b* + R_b
        FS_TRY(cudaStreamWaitEvent(sa, evD, 0));
        FS_CHECK(routed_impl(desc, x_perm, offsets, bw.w13, bw.w3, y_perm, ws, sa));
        FS_TRY(cudaStreamWaitEvent(sa, evU, 0));
        FS_CHECK(combine_impl(desc, y_perm, pos, w, ostar, FS_F32, nullptr, nullptr, last ? o_partial : nullptr, o_k,
                              last ? act : FS_F32, nullptr, wiring, nullptr, sa));
        FS_TRY(cudaEventRecord(evA, sa));
        u = u_next;
        o_prev = o_k;
        prev_dtype = FS_F32;
    }
    // join: stream waits for stream2's last work
    FS_TRY(cudaEventRecord(evU, sb));
    FS_TRY(cudaStreamWaitEvent(sa, evU, 0));
    return FS_OK;
}

// ---------------------------------------------------------------- training
// What the backward reads from the training forward, per block (bf16 unless
// noted): the block input u_k, the router logits (fp32, without the bias), the
// routing (top-k indices, gate weights), the Dispatch permutation (offsets,
// pos, perm_src), the routed experts' pre-activations g, a (packed gate/up
// column order) and hidden h, the routed outputs y_perm, and the shared
// experts' pre-activations and hidden.
struct SavedLayout {
    size_t u, logits, idx, w, offsets, pos, perm, xp, gu, h, y, gu_s, h_s, size;
};

static SavedLayout saved_layout(const fs_layer_desc* d) {
    const size_t A = 256;
    const size_t T = d->T, E = d->E, k = d->k, dm = d->d, c = d->c;
    const size_t rows = T * k, cw = static_cast<size_t>(d->n_shared) * d->c_shared;
    SavedLayout l;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at_ = o; o = align_up(o + bytes, A); return at_; };
    l.u = take(T * dm * 2);
    l.logits = take(T * E * 4);
    l.idx = take(rows * 4);
    l.w = take(rows * 4);
    l.offsets = take((E + 1) * 4);
    l.pos = take(rows * 4);
    l.perm = take(rows * 4);
    l.xp = take(rows * dm * 2);
    l.gu = take(rows * 2 * c * 2);
    l.h = take(rows * c * 2);
    l.y = take(rows * dm * 2);
    l.gu_s = take(T * 2 * cw * 2);
    l.h_s = take(T * cw * 2);
    l.size = o;
    return l;
}

// Workspace of the backward: the gradients of the inner residuals o_1..o_{L-1}
// and o_1*..o_{L-1}* (fp32) and the per-block step buffers.
struct BwdLayout {
    size_t go, gos, dy, dw, dS, dgu, dx, dgu_s, dz, plan_r, plan_s, end;
    int Epad;
};

static BwdLayout bwd_layout(const fs_layer_desc* d, int L) {
    const size_t A = 256;
    const size_t T = d->T, E = d->E, k = d->k, dm = d->d, c = d->c;
    const size_t rows = T * k, cw = static_cast<size_t>(d->n_shared) * d->c_shared;
    BwdLayout l;
    l.Epad = static_cast<int>(align_up(E, 64));
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at_ = o; o = align_up(o + bytes, A); return at_; };
    l.go = take(static_cast<size_t>(L) * T * dm * 4);      // gradients of o_1 .. o_{L-1} (slot b)
    l.gos = take(static_cast<size_t>(L) * T * dm * 4);     // and of o_1* .. o_{L-1}*
    l.dy = take(rows * dm * 2);
    l.dw = take(rows * 4);
    l.dS = take(T * dm * 2);
    l.dgu = take(rows * 2 * c * 2);
    l.dx = take(rows * dm * 2);
    l.dgu_s = take(T * 2 * cw * 2);
    l.dz = take(T * l.Epad * 2);
    l.plan_r = take(2 * (E + 1) * sizeof(int));
    l.plan_s = take(4 * sizeof(int));
    l.end = o;
    return l;
}

static fs_status check_train(const fs_layer_desc* desc, int L, int wiring) {
    FS_CHECK(check_desc(desc));
    if (desc->dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
    if (L < 1) return FS_ERR_INVALID_ARG;
    if (wiring < FS_WIRE_PARTIAL || wiring > FS_WIRE_DISABLED) return FS_ERR_INVALID_ARG;
    return FS_OK;
}

size_t fs_train_saved_bytes(const fs_layer_desc* desc, int L) {
    if (check_train(desc, L < 1 ? 1 : L, FS_WIRE_PARTIAL) != FS_OK || L < 1) return 0;
    return static_cast<size_t>(L) * saved_layout(desc).size;
}

size_t fs_workspace_bytes_backward(const fs_layer_desc* desc, int L) {
    if (check_train(desc, L < 1 ? 1 : L, FS_WIRE_PARTIAL) != FS_OK || L < 1) return 0;
    return bwd_layout(desc, L).end;
}

fs_status fs_pack_w13t(int32_t G, int32_t c, int32_t d, const void* w1, const void* w2, void* out, void* stream) {
    if (G < 1 || c < 1 || d < 1) return FS_ERR_INVALID_ARG;
    if (c % 64 || d % 64) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w1));
    FS_CHECK(need(w2));
    FS_CHECK(need(out));
    FS_TRY(launch_pack_t(0, G, d, 2 * c, c, d, 0, 0, w1, w2, out, static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

fs_status fs_pack_w3t(int32_t G, int32_t d, int32_t c, const void* w3, void* out, void* stream) {
    if (G < 1 || c < 1 || d < 1) return FS_ERR_INVALID_ARG;
    if (c % 64 || d % 64) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w3));
    FS_CHECK(need(out));
    FS_TRY(launch_pack_t(1, G, c, d, c, d, 0, 0, w3, nullptr, out, static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

fs_status fs_pack_w3t_shared(int32_t n_shared, int32_t c_shared, int32_t d, const void* w3s, void* out,
                             void* stream) {
    if (n_shared < 1 || c_shared < 1 || d < 1) return FS_ERR_INVALID_ARG;
    if (c_shared % 64 || d % 64) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w3s));
    FS_CHECK(need(out));
    FS_TRY(launch_pack_t(2, 1, n_shared * c_shared, d, 0, d, c_shared, 0, w3s, nullptr, out,
                         static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

fs_status fs_pack_wrt(int32_t E, int32_t d, const void* w_r, void* out, void* stream) {
    if (E < 1 || d < 1) return FS_ERR_INVALID_ARG;
    if (d % 64) return FS_ERR_UNSUPPORTED;
    FS_CHECK(need(w_r));
    FS_CHECK(need(out));
    FS_TRY(launch_pack_t(3, 1, d, static_cast<int>(align_up(E, 64)), 0, d, 0, E, w_r, nullptr, out,
                         static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

fs_status fs_farskip_stack_train(const fs_layer_desc* desc, int32_t L, int32_t wiring, const fs_block_weights* blocks,
                                 const void* x, void* o_full, void* o_partial, void* saved, size_t saved_bytes,
                                 void* ws, size_t ws_bytes, void* stream) {
    FS_CHECK(check_train(desc, L, wiring));
    if (!blocks) return FS_ERR_INVALID_ARG;
    FS_CHECK(need(x));
    FS_CHECK(need(o_full));
    if (o_partial && !aligned16(o_partial)) return FS_ERR_UNSUPPORTED;
    for (int b = 0; b < L; ++b) {
        FS_CHECK(need(blocks[b].w_r));
        FS_CHECK(need(blocks[b].w13));
        FS_CHECK(need(blocks[b].w3));
        if (blocks[b].bias && !aligned16(blocks[b].bias)) return FS_ERR_UNSUPPORTED;
        if (desc->n_shared > 0) {
            FS_CHECK(need(blocks[b].w13_shared));
            FS_CHECK(need(blocks[b].w3_shared));
        }
    }
    FS_CHECK(check_ws(desc, L, ws, ws_bytes));
    if (!saved) return FS_ERR_INVALID_ARG;
    const SavedLayout sl = saved_layout(desc);
    if ((reinterpret_cast<uintptr_t>(saved) & 255u) || saved_bytes < static_cast<size_t>(L) * sl.size)
        return FS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const Layout l = layout(desc, L);
    const Layout l0 = layout(desc, 0);
    const int T = desc->T, rows = desc->T * desc->k, cw = desc->n_shared * desc->c_shared;
    auto sv = [&](int blk, size_t off) { return static_cast<uint8_t*>(saved) + static_cast<size_t>(blk) * sl.size + off; };
    int32_t* counts = at<int32_t>(ws, l.counts);
    void* s_out = cw > 0 ? at<void>(ws, l.s_out) : nullptr;
    FS_TRY(launch_copy(sv(0, sl.u), x, static_cast<size_t>(T) * desc->d * 2, st));
    const void* o_prev = x;
    int prev_dtype = FS_BF16;
    for (int b = 1; b <= L; ++b) {
        const fs_block_weights& bw = blocks[b - 1];
        const int blk = b - 1;
        const bool last = (b == L);
        const void* u = sv(blk, sl.u);
        int32_t* idx = reinterpret_cast<int32_t*>(sv(blk, sl.idx));
        float* w = reinterpret_cast<float*>(sv(blk, sl.w));
        int32_t* offsets = reinterpret_cast<int32_t*>(sv(blk, sl.offsets));
        int32_t* pos = reinterpret_cast<int32_t*>(sv(blk, sl.pos));
        void* y = sv(blk, sl.y);
        FS_CHECK(router_impl(desc, u, bw.w_r, bw.bias, idx, w, reinterpret_cast<float*>(sv(blk, sl.logits)), ws, st));
        void* x_perm = sv(blk, sl.xp);      // kept: the weight-gradient GEMMs read it
        FS_CHECK(dispatch_impl(desc, idx, u, counts, offsets, pos, reinterpret_cast<int32_t*>(sv(blk, sl.perm)),
                               x_perm, ws, st));
        FS_CHECK(swiglu_impl(desc, x_perm, rows, nullptr, rows, offsets, desc->E, desc->c, bw.w13, bw.w3, y, false,
                             at<int>(ws, l0.plan_r), sv(blk, sl.h), nullptr, st, sv(blk, sl.gu)));
        if (s_out)
            FS_CHECK(swiglu_impl(desc, u, T, nullptr, T, nullptr, 1, cw, bw.w13_shared, bw.w3_shared, s_out, true,
                                 at<int>(ws, l0.plan_s), sv(blk, sl.h_s), nullptr, st, sv(blk, sl.gu_s)));
        void* o_k = last ? o_full : at<void>(ws, l.ring[(b - 1) % l.nring]);
        void* os_k = last ? o_partial : at<void>(ws, l.star[(b - 1) % l.nstar]);
        void* u_next = last ? nullptr : sv(b, sl.u);
        const int out_dtype = last ? FS_BF16 : FS_F32;
        FS_CHECK(combine_impl(desc, y, pos, w, o_prev, prev_dtype, s_out, nullptr, os_k, o_k, out_dtype, u_next, wiring,
                              nullptr, st));
        o_prev = o_k;
        prev_dtype = out_dtype;
    }
    return FS_OK;
}

fs_status fs_farskip_stack_backward(const fs_layer_desc* desc, int32_t L, int32_t wiring,
                                    const fs_block_weights* blocks, const fs_block_weights_t* blocks_t,
                                    const void* saved, size_t saved_bytes, const float* d_o, const float* d_os,
                                    float* dx, const fs_block_grads* grads, void* ws, size_t ws_bytes, void* stream) {
    FS_CHECK(check_train(desc, L, wiring));
    if (!blocks || !blocks_t || !grads) return FS_ERR_INVALID_ARG;
    FS_CHECK(need(d_o));
    FS_CHECK(need(dx));
    if (d_os && !aligned16(d_os)) return FS_ERR_UNSUPPORTED;
    const bool sh = desc->n_shared > 0;
    for (int b = 0; b < L; ++b) {
        if (blocks[b].bias && !aligned16(blocks[b].bias)) return FS_ERR_UNSUPPORTED;
        FS_CHECK(need(blocks_t[b].w13t));
        FS_CHECK(need(blocks_t[b].w3t));
        FS_CHECK(need(blocks_t[b].w_rt));
        FS_CHECK(need(grads[b].dw_r));
        FS_CHECK(need(grads[b].dw1));
        FS_CHECK(need(grads[b].dw2));
        FS_CHECK(need(grads[b].dw3));
        if (sh) {
            FS_CHECK(need(blocks_t[b].w13t_shared));
            FS_CHECK(need(blocks_t[b].w3t_shared));
            FS_CHECK(need(grads[b].dw1_shared));
            FS_CHECK(need(grads[b].dw2_shared));
            FS_CHECK(need(grads[b].dw3_shared));
        }
    }
    if (!saved || !ws) return FS_ERR_INVALID_ARG;
    const SavedLayout sl = saved_layout(desc);
    const BwdLayout bl = bwd_layout(desc, L);
    if ((reinterpret_cast<uintptr_t>(saved) & 255u) || saved_bytes < static_cast<size_t>(L) * sl.size)
        return FS_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < bl.end) return FS_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int T = desc->T, E = desc->E, k = desc->k, dm = desc->d, c = desc->c;
    const int rows = T * k, cs = desc->c_shared, cw = desc->n_shared * cs;
    const size_t n = static_cast<size_t>(T) * dm;
    auto sv = [&](int blk, size_t off) {
        return static_cast<const uint8_t*>(saved) + static_cast<size_t>(blk) * sl.size + off;
    };
    float* go = at<float>(ws, bl.go);
    float* gos = at<float>(ws, bl.gos);
    void* dy = at<void>(ws, bl.dy);
    float* dw = at<float>(ws, bl.dw);
    void* dS = at<void>(ws, bl.dS);
    void* dgu = at<void>(ws, bl.dgu);
    void* dxp = at<void>(ws, bl.dx);
    void* dgu_s = at<void>(ws, bl.dgu_s);
    void* dz = at<void>(ws, bl.dz);
    int* plan_r = at<int>(ws, bl.plan_r);
    int* plan_s = at<int>(ws, bl.plan_s);
    const int bm = tc_block_m();
    const int max_mt = ceil_div(rows, bm) + E;
    // gradients of o_b (b = 0..L) and o_b* (b = 1..L): the caller's d_o, d_os for
    // b = L, dx itself for o_0 = x, workspace in between; accumulated into
    auto g_o = [&](int b) -> float* {
        return b == L ? const_cast<float*>(d_o) : (b == 0 ? dx : go + static_cast<size_t>(b) * n);
    };
    auto g_os = [&](int b) -> float* {
        return b == L ? const_cast<float*>(d_os) : gos + static_cast<size_t>(b) * n;
    };
    FS_TRY(launch_zero(dx, n * 4, st));
    if (L > 1) {
        FS_TRY(launch_zero(go + n, static_cast<size_t>(L - 1) * n * 4, st));
        FS_TRY(launch_zero(gos + n, static_cast<size_t>(L - 1) * n * 4, st));
    }
    FS_TRY(launch_plan(nullptr, 1, T, bm, plan_s, st));
    for (int b = L; b >= 1; --b) {
        const int blk = b - 1;
        const fs_block_weights& bw = blocks[blk];
        const fs_block_weights_t& bt = blocks_t[blk];
        const fs_block_grads& gr = grads[blk];
        const void* u = sv(blk, sl.u);
        const int32_t* idx = reinterpret_cast<const int32_t*>(sv(blk, sl.idx));
        const float* w = reinterpret_cast<const float*>(sv(blk, sl.w));
        const int32_t* offsets = reinterpret_cast<const int32_t*>(sv(blk, sl.offsets));
        const int32_t* pos = reinterpret_cast<const int32_t*>(sv(blk, sl.pos));
        // the wiring: block b's do_prev goes to o_{b-1}; its du to where u_b came
        // from (o_{b-1}* partial, o_{b-2} outdated, o_{b-1} disabled, x for b = 1)
        float* target;
        if (b == 1) target = g_o(0);
        else if (wiring == FS_WIRE_PARTIAL) target = g_os(b - 1);
        else if (wiring == FS_WIRE_OUTDATED) target = g_o(b - 2);
        else target = g_o(b - 1);
        // Combine backward: dy_perm, dw, dS = dO + dOs; do_prev accumulated into o_{b-1}'s gradient
        FS_TRY(launch_combine_backward(g_o(b), g_os(b), sv(blk, sl.y), pos, w, T, dm, k, dy, dw, sh ? dS : nullptr,
                                       g_o(b - 1), st));
        // routed experts: dh = dy W3 with the SwiGLU backward in the epilogue, then dx = dgu W13
        FS_TRY(launch_plan(offsets, E, rows, bm, plan_r, st));
        TcExtra exr;
        exr.aux = const_cast<uint8_t*>(sv(blk, sl.gu));
        exr.aux_ld = 2LL * c;
        FS_TRY(launch_tc_gemm(EPI_DSWIGLU, dy, rows, bt.w3t, E, c, dm, plan_r, max_mt, dgu, 2LL * c, c, nullptr, 0, true,
                              st, &exr));
        FS_TRY(launch_tc_gemm(EPI_BF16, dgu, rows, bt.w13t, E, dm, 2 * c, plan_r, max_mt, dxp, dm, dm, nullptr, 0, true,
                              st));
        FS_TRY(launch_gather_sum(dxp, pos, T, dm, k, target, st));     // Dispatch backward
        TcExtra acc;
        acc.accumulate = 1;
        if (sh) {
            TcExtra exs;
            exs.aux = const_cast<uint8_t*>(sv(blk, sl.gu_s));
            exs.aux_ld = 2LL * cw;
            FS_TRY(launch_tc_gemm(EPI_DSWIGLU, dS, T, bt.w3t_shared, 1, cw, dm, plan_s, ceil_div(T, bm) + 1, dgu_s,
                                  2LL * cw, cw, nullptr, 0, true, st, &exs));
            FS_TRY(launch_tc_gemm(EPI_F32, dgu_s, T, bt.w13t_shared, 1, dm, 2 * cw, plan_s, ceil_div(T, bm) + 1, target,
                                  dm, dm, nullptr, 0, true, st, &acc));
        }
        // router: dz through the gate rule, du += dz W_R
        FS_TRY(launch_gate_backward(reinterpret_cast<const float*>(sv(blk, sl.logits)), bw.bias, idx, w, dw, T, E,
                                    bl.Epad, k, desc->gate, dz, st));
        FS_TRY(launch_tc_gemm(EPI_F32, dz, T, bt.w_rt, 1, dm, bl.Epad, plan_s, ceil_div(T, bm) + 1, target, dm, dm,
                              nullptr, 0, true, st, &acc));
        // weight gradients: contractions over each expert's rows (all T rows for
        // the shared experts and the router), the token-row operands read in place
        FS_TRY(launch_wgrad_gemm(dy, dm, sv(blk, sl.h), c, rows, offsets, E, dm, c, gr.dw3, nullptr, 0, 0, st));
        FS_TRY(launch_wgrad_gemm(dgu, 2 * c, sv(blk, sl.xp), dm, rows, offsets, E, 2 * c, dm, gr.dw1, gr.dw2, 1, 0,
                                 st));
        if (sh) {
            FS_TRY(launch_wgrad_gemm(dS, dm, sv(blk, sl.h_s), cw, T, nullptr, 1, dm, cw, gr.dw3_shared, nullptr, 2, cs,
                                     st));
            FS_TRY(launch_wgrad_gemm(dgu_s, 2 * cw, u, dm, T, nullptr, 1, 2 * cw, dm, gr.dw1_shared, gr.dw2_shared, 1,
                                     0, st));
        }
        FS_TRY(launch_wgrad_gemm(dz, bl.Epad, u, dm, T, nullptr, 1, E, dm, gr.dw_r, nullptr, 0, 0, st));
    }
    return FS_OK;
}

fs_status fs_get_error(int32_t* code) {
    int* p = dev_error_ptr();
    if (!p) return cuda_status(cudaGetLastError());
    int v = 0;
    FS_TRY(cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost));
    const int zero = 0;
    FS_TRY(cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice));
    if (code) *code = v;
    return v ? FS_ERR_DEVICE_STATE : FS_OK;
}

fs_status fs_selftest_wait_timeout(int32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 2000000) return FS_ERR_INVALID_ARG;
    FS_TRY(launch_wait_selftest(static_cast<uint64_t>(limit_us) * 1000ull, static_cast<cudaStream_t>(stream)));
    return FS_OK;
}

uint64_t fs_launch_count(void) { return g_launches.load(); }

const char* fs_last_cuda_error(void) { return g_last_cuda; }

const char* fs_status_string(fs_status s) {
    switch (s) {
        case FS_OK: return "FS_OK";
        case FS_ERR_INVALID_ARG: return "FS_ERR_INVALID_ARG";
        case FS_ERR_UNSUPPORTED: return "FS_ERR_UNSUPPORTED";
        case FS_ERR_WORKSPACE: return "FS_ERR_WORKSPACE";
        case FS_ERR_CUDA: return "FS_ERR_CUDA";
        case FS_ERR_DEVICE_STATE: return "FS_ERR_DEVICE_STATE";
        default: return "FS_ERR_UNKNOWN";
    }
}

}  // extern "C"
