// router.cu -- top-k selection and gate weights over router logits.
//
// "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
// Models", §2.1: G(A) = s(A W_R^T), a linear classifier followed by a sparse
// selection s().  The logits z = u W_R^T come from the grouped GEMM (tensor
// cores for bf16, fp32 FMA for fp32), for few tokens as partial sums over K
// ranges that this kernel adds in a fixed order (and stores when asked); it
// then adds the bias, selects the
// k largest z (descending, ties to the lower expert index) and computes the
// gate weights of the configured rule.  One warp per token: each lane holds
// E/32 logits in registers, k rounds of a warp-shuffle argmax.
#include "common.cuh"
#include "kernels.h"

namespace fs {

constexpr int kTopkWarps = 8;

template <int EPL>   // experts per lane (E <= 32 * EPL)
__global__ void __launch_bounds__(kTopkWarps * 32)
topk_kernel(const float* __restrict__ logits, int nsplit, const float* __restrict__ bias, int T, int E, int k,
            int gate, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* __restrict__ z_out) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const long long part = static_cast<long long>(T) * E;     // elements between partial sums
    const float* z = logits + static_cast<long long>(t) * E;
    // the K ranges' partials added in order; the lane's EPL logits are independent
    // chains, so each range's EPL loads are in flight together
    float v[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? z[e] : 0.0f;
    }
    for (int s = 1; s < nsplit; ++s) {
        const float* zs = z + s * part;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E) v[j] += zs[e];
        }
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            if (z_out) z_out[static_cast<long long>(t) * E + e] = v[j];
            v[j] += bias ? bias[e] : 0.0f;
        } else {
            v[j] = -INFINITY;
        }
    }
    uint32_t taken = 0;
    float sel_v = 0.f;     // lane s < k keeps slot s
    int sel_i = 0;
    float zmax = 0.f;
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !(taken >> j & 1u) && (v[j] > bv || (v[j] == bv && e < bi))) {
                bv = v[j];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == s) {
            sel_v = bv;
            sel_i = bi;
        }
        if (s == 0) zmax = bv;
    }
    // gate weights (lane s < k holds slot s)
    float w = 0.f;
    if (gate == 0) {               // softmax over all experts
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            if (lane + 32 * j < E) part += expf(v[j] - zmax);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        w = expf(sel_v - zmax) / part;
    } else if (gate == 1) {        // softmax over the k chosen
        float ex = lane < k ? expf(sel_v - zmax) : 0.f;
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        w = ex / sum;
    } else if (gate == 2) {        // sigmoid
        w = 1.0f / (1.0f + expf(-sel_v));
    } else {                       // sigmoid normalised over the k chosen
        float sg = lane < k ? 1.0f / (1.0f + expf(-sel_v)) : 0.f;
        float sum = sg;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        w = sg / sum;
    }
    if (lane < k) {
        topk_idx[static_cast<long long>(t) * k + lane] = sel_i;
        topk_w[static_cast<long long>(t) * k + lane] = w;
    }
}

cudaError_t launch_topk(const float* logits, int nsplit, const float* bias, int T, int E, int k, int gate,
                        int32_t* topk_idx, float* topk_w, float* z_out, cudaStream_t st) {
    const int grid = (T + kTopkWarps - 1) / kTopkWarps;
    const int threads = kTopkWarps * 32;
    if (nsplit < 1) return cudaErrorInvalidValue;
#define FS_TOPK(EPL) \
    topk_kernel<EPL><<<grid, threads, 0, st>>>(logits, nsplit, bias, T, E, k, gate, topk_idx, topk_w, z_out)
    if (E <= 32)
        FS_TOPK(1);
    else if (E <= 128)
        FS_TOPK(4);
    else if (E <= 256)
        FS_TOPK(8);
    else
        FS_TOPK(16);
#undef FS_TOPK
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
