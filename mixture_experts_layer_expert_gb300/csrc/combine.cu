// combine.cu -- local Combine fused with the shared-expert add and the
// FarSkip-Collective residual update.
//
// "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
// Models": §2.1 Combine (aggregate and sum the routed expert activations back
// to token order), §3 eq. (8b) (o_k* = o_{k-1} + f_k*(o_{k-1}*), f* = shared
// expert) and the FarSkip equation (o_k = o_{k-1} + f_k(o_{k-1}*)).
//   R[t]   = sum_{s<k} w[t, s] * y_perm[pos[t k + s]]     (fp32, slot order: no atomics)
//   o*[t]  = o_prev[t] + S[t]
//   o[t]   = o_prev[t] + S[t] + R[t]
// One warp per token, 16-byte vectors: each lane loads the k expert rows of
// its columns together (k loads in flight), sums in fp32, rounds once.
#include "common.cuh"
#include "kernels.h"

namespace fs {

constexpr int kCombineWarps = 8;

template <bool BF16>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const uint4* __restrict__ y_perm, const int32_t* __restrict__ pos, const float* __restrict__ topk_w,
               const uint4* __restrict__ o_prev, const uint4* __restrict__ shared_out, uint4* __restrict__ o_partial,
               uint4* __restrict__ o_full, int T, int row_vecs, int k) {
    constexpr int EPV = BF16 ? 8 : 4;   // elements per 16-byte vector
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_p = -1;
    float my_w = 0.f;
    if (lane < k) {
        my_p = pos[static_cast<long long>(t) * k + lane];
        my_w = topk_w[static_cast<long long>(t) * k + lane];
    }
    int ps[kMaxTopK];
    float ws[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
        ps[s] = __shfl_sync(0xffffffffu, my_p, s);
        ws[s] = __shfl_sync(0xffffffffu, my_w, s);
    }
    const long long row = static_cast<long long>(t) * row_vecs;
    for (int i = lane; i < row_vecs; i += 32) {
        float acc[EPV];
        float base[EPV];
        {
            const uint4 a = o_prev[row + i];
            const uint4 b = shared_out ? shared_out[row + i] : make_uint4(0, 0, 0, 0);
            const uint32_t av[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if constexpr (BF16) {
                    base[2 * q] = bf16lo(av[q]) + bf16lo(bv[q]);
                    base[2 * q + 1] = bf16hi(av[q]) + bf16hi(bv[q]);
                } else {
                    base[q] = __uint_as_float(av[q]) + __uint_as_float(bv[q]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < EPV; ++j) acc[j] = 0.f;
        uint4 yv[kMaxTopK];
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s)
            if (s < k && ps[s] >= 0) yv[s] = y_perm[static_cast<long long>(ps[s]) * row_vecs + i];
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s) {
            if (s < k && ps[s] >= 0) {
                const uint32_t v[4] = {yv[s].x, yv[s].y, yv[s].z, yv[s].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if constexpr (BF16) {
                        acc[2 * q] = fmaf(ws[s], bf16lo(v[q]), acc[2 * q]);
                        acc[2 * q + 1] = fmaf(ws[s], bf16hi(v[q]), acc[2 * q + 1]);
                    } else {
                        acc[q] = fmaf(ws[s], __uint_as_float(v[q]), acc[q]);
                    }
                }
            }
        }
        uint32_t op[4], of[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if constexpr (BF16) {
                op[q] = pack_bf16x2(base[2 * q], base[2 * q + 1]);
                of[q] = pack_bf16x2(base[2 * q] + acc[2 * q], base[2 * q + 1] + acc[2 * q + 1]);
            } else {
                op[q] = __float_as_uint(base[q]);
                of[q] = __float_as_uint(base[q] + acc[q]);
            }
        }
        if (o_partial) o_partial[row + i] = make_uint4(op[0], op[1], op[2], op[3]);
        o_full[row + i] = make_uint4(of[0], of[1], of[2], of[3]);
    }
}

cudaError_t launch_combine(const void* y_perm, const int32_t* pos, const float* topk_w, const void* o_prev,
                           const void* shared_out, void* o_partial, void* o_full, int T, int d, int k,
                           int is_bf16, cudaStream_t st) {
    const int row_vecs = d * (is_bf16 ? 2 : 4) / 16;
    const int grid = (T + kCombineWarps - 1) / kCombineWarps;
    const int threads = kCombineWarps * 32;
    if (is_bf16)
        combine_kernel<true><<<grid, threads, 0, st>>>(
            static_cast<const uint4*>(y_perm), pos, topk_w, static_cast<const uint4*>(o_prev),
            static_cast<const uint4*>(shared_out), static_cast<uint4*>(o_partial), static_cast<uint4*>(o_full), T,
            row_vecs, k);
    else
        combine_kernel<false><<<grid, threads, 0, st>>>(
            static_cast<const uint4*>(y_perm), pos, topk_w, static_cast<const uint4*>(o_prev),
            static_cast<const uint4*>(shared_out), static_cast<uint4*>(o_partial), static_cast<uint4*>(o_full), T,
            row_vecs, k);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
