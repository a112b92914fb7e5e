// combine.cu -- local Combine fused with the shared-expert add and the
// FarSkip-Collective residual update.
//
// "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
// Models": §2.1 Combine (aggregate and sum the routed expert activations back
// to token order), §3 eq. (8b) (o_k* = o_{k-1} + f_k*(o_{k-1}*), f* = shared
// expert), eq. (8a) and the FarSkip equation (o_k = o_{k-1} + f_k(o_{k-1}*)).
//   R[t]   = sum_{s<k} w[t, s] * y_perm[pos[t k + s]]     (fp32, slot order: no atomics)
//   o*[t]  = o_prev[t] + S[t]
//   o[t]   = o_prev[t] + S[t] + R[t]
//   u'[t]  = the next block's input, rounded to the activation type:
//            o*[t] (partial), o_prev[t] (outdated) or o[t] (disabled)
// An optional fp32 term (the stand-in attention output of the attention
// wirings) is added into o* and o, and o may also be written rounded to the
// activation type (the next MoE input of the attention/MoE wiring).
// The residual stream (o_prev, o*, o) may be fp32 or the activation type; S is
// fp32; the expert rows and u' are in the activation type.  One warp per token
// (or, for few tokens, per run of 256-column steps of a token, so that enough
// warps are in flight), 8 columns per lane step: each lane loads the k expert
// rows of its columns together (k loads in flight), sums in fp32, rounds once
// per output.
#include "common.cuh"
#include "kernels.h"

namespace fs {

constexpr int kCombineWarps = 8;

// 8 consecutive elements at element offset `off` (a multiple of 8)
__device__ __forceinline__ void load8(const void* base, long long off, bool bf16, float (&v)[8]) {
    if (bf16) {
        const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[2 * q] = bf16lo(w[q]);
            v[2 * q + 1] = bf16hi(w[q]);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        const float4 a = p[0], b = p[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ void store8(void* base, long long off, bool bf16, const float (&v)[8]) {
    if (bf16) {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off) =
            make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                       pack_bf16x2(v[6], v[7]));
    } else {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// raw 16-byte vectors of 8 elements of a row (1 for bf16, 2 for fp32)
template <bool BF16>
struct Raw8 {
    uint4 v[BF16 ? 1 : 2];
};

template <bool BF16>
__device__ __forceinline__ void load_raw8(const void* base, long long off, Raw8<BF16>& r) {
    if constexpr (BF16) {
        r.v[0] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + off);
        r.v[0] = p[0];
        r.v[1] = p[1];
    }
}

template <bool BF16>
__device__ __forceinline__ void fma_raw8(float w, const Raw8<BF16>& r, float (&acc)[8]) {
    if constexpr (BF16) {
        const uint32_t q[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = fmaf(w, bf16lo(q[i]), acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, bf16hi(q[i]), acc[2 * i + 1]);
        }
    } else {
        const uint32_t q[8] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w, r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, __uint_as_float(q[i]), acc[i]);
    }
}

template <bool BF16, int KMAX>   // BF16: activation type of y_perm and u_next
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const void* __restrict__ y_perm, const int32_t* __restrict__ pos, const float* __restrict__ topk_w,
               const void* __restrict__ o_prev, bool prev_bf16, const void* __restrict__ shared_out,
               const float* __restrict__ extra, void* __restrict__ o_partial, void* __restrict__ o_full, bool out_bf16,
               void* __restrict__ u_next, int u_src, void* __restrict__ u_full, int T, int d, int k, int nch,
               int cpc) {
    const int lane = threadIdx.x & 31;
    const long long wid = static_cast<long long>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
    const int t = static_cast<int>(wid / nch);
    if (t >= T) return;
    const int c_begin = static_cast<int>(wid - static_cast<long long>(t) * nch) * cpc * 256;   // this warp's columns
    const int c_end = min(d, c_begin + cpc * 256);
    int my_p = -1;
    float my_w = 0.f;
    if (lane < k) {
        my_p = pos[static_cast<long long>(t) * k + lane];
        my_w = topk_w[static_cast<long long>(t) * k + lane];
    }
    int ps[KMAX];
    float ws[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
        ps[s] = __shfl_sync(0xffffffffu, my_p, s);
        ws[s] = __shfl_sync(0xffffffffu, my_w, s);
    }
    const long long row = static_cast<long long>(t) * d;
    for (int c8 = c_begin + lane * 8; c8 < c_end; c8 += 32 * 8) {
        Raw8<BF16> yr[KMAX];
#pragma unroll
        for (int s = 0; s < KMAX; ++s)
            if (s < k && ps[s] >= 0) load_raw8<BF16>(y_perm, static_cast<long long>(ps[s]) * d + c8, yr[s]);
        float base[8], sv[8], acc[8];
        load8(o_prev, row + c8, prev_bf16, base);
        if (shared_out) {
            load8(shared_out, row + c8, false, sv);     // S is fp32
#pragma unroll
            for (int j = 0; j < 8; ++j) base[j] += sv[j];
        }
        if (extra) {                                    // e.g. the attention output (fp32)
            load8(extra, row + c8, false, sv);
#pragma unroll
            for (int j = 0; j < 8; ++j) base[j] += sv[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
        for (int s = 0; s < KMAX; ++s)
            if (s < k && ps[s] >= 0) fma_raw8<BF16>(ws[s], yr[s], acc);
        float full[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) full[j] = base[j] + acc[j];
        if (o_partial) store8(o_partial, row + c8, out_bf16, base);
        store8(o_full, row + c8, out_bf16, full);
        if (u_next) {
            if (u_src == 0) {
                store8(u_next, row + c8, BF16, base);
            } else if (u_src == 1) {
                float op[8];
                load8(o_prev, row + c8, prev_bf16, op);
                store8(u_next, row + c8, BF16, op);
            } else {
                store8(u_next, row + c8, BF16, full);
            }
        }
        if (u_full) store8(u_full, row + c8, BF16, full);
    }
}

cudaError_t launch_combine(const void* y_perm, const int32_t* pos, const float* topk_w, const void* o_prev,
                           int prev_bf16, const void* shared_out, const float* extra, void* o_partial, void* o_full,
                           int out_bf16, void* u_next, int u_src, void* u_full, int T, int d, int k, int is_bf16,
                           cudaStream_t st) {
    // runs of cpc 256-column steps per warp: one run per token when there are
    // many tokens, up to one step per warp for a few (about 16K warps wanted)
    const int steps = (d + 255) / 256;
    const int want = T >= 16384 ? 1 : (16384 + T - 1) / T;
    const int cpc = (steps + want - 1) / want;
    const int nch = (steps + cpc - 1) / cpc;
    const long long warps = static_cast<long long>(T) * nch;
    const int grid = static_cast<int>((warps + kCombineWarps - 1) / kCombineWarps);
    const int threads = kCombineWarps * 32;
#define FS_COMBINE(BF, KM)                                                                                  \
    combine_kernel<BF, KM><<<grid, threads, 0, st>>>(y_perm, pos, topk_w, o_prev, prev_bf16 != 0, shared_out,   \
                                                     extra, o_partial, o_full, out_bf16 != 0, u_next, u_src, u_full, \
                                                     T, d, k, nch, cpc)
    if (is_bf16) {
        if (k <= 8) FS_COMBINE(true, 8); else FS_COMBINE(true, 16);
    } else {
        if (k <= 8) FS_COMBINE(false, 8); else FS_COMBINE(false, 16);
    }
#undef FS_COMBINE
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
