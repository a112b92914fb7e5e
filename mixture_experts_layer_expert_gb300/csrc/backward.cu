// backward.cu -- the memory-bound kernels of the MoE block's backward (training
// form of "FarSkip-Collective", §2.1 MoE and Combine, §3 FarSkip update):
// Combine backward, Dispatch backward (the gather-sum of the permuted input
// gradients), the gate-rule backward of the router and the transposed weight
// packs of the input-gradient GEMMs.  The GEMMs themselves (the weight-gradient
// GEMMs read the token-row activations in place) run in gemm_tc.cu.
#include "common.cuh"
#include "kernels.h"

namespace fs {

constexpr int kBwdWarps = 8;

__device__ __forceinline__ void load8f(const float* p, float* v) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void unpack8(const uint4& q, float* v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = bf16lo(w[i]);
        v[2 * i + 1] = bf16hi(w[i]);
    }
}
__device__ __forceinline__ uint4 pack8(const float* v) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// Combine backward, one warp per token t, with dR = dO and dS = dO + dOs:
//   dy_perm[pos[t, s]] = bf16(w[t, s] dO[t])       (the routed output gradient)
//   dw[t, s]           = <dO[t], y_perm[pos[t, s]]> (fp32; lane partials, then a shuffle tree)
//   dS[t] = bf16(dO + dOs), do_prev[t] += dO + dOs  (when the pointers are set)
template <int KMAX>
__global__ void __launch_bounds__(kBwdWarps * 32)
combine_backward_kernel(const float* __restrict__ dO, const float* __restrict__ dOs, const uint4* __restrict__ y_perm,
                        const int32_t* __restrict__ pos, const float* __restrict__ topk_w, int T, int d, int k,
                        uint4* __restrict__ dy_perm, float* __restrict__ dw, uint4* __restrict__ dS,
                        float* __restrict__ do_prev) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int nv = d / 8;
    int p[KMAX];
    float wv[KMAX], acc[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
        p[s] = s < k ? pos[static_cast<long long>(t) * k + s] : -1;
        wv[s] = s < k ? topk_w[static_cast<long long>(t) * k + s] : 0.0f;
        acc[s] = 0.0f;
    }
    const float* gO = dO + static_cast<long long>(t) * d;
    for (int v = lane; v < nv; v += 32) {
        float g[8];
        load8f(gO + 8 * v, g);
#pragma unroll
        for (int s = 0; s < KMAX; ++s) {
            if (p[s] < 0) continue;
            float y[8], dy[8];
            unpack8(__ldg(y_perm + static_cast<long long>(p[s]) * nv + v), y);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[s] += g[i] * y[i];
                dy[i] = wv[s] * g[i];
            }
            dy_perm[static_cast<long long>(p[s]) * nv + v] = pack8(dy);
        }
        if (dS || do_prev) {
            float sv[8];
            if (dOs) {
                float h[8];
                load8f(dOs + static_cast<long long>(t) * d + 8 * v, h);
#pragma unroll
                for (int i = 0; i < 8; ++i) sv[i] = g[i] + h[i];
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) sv[i] = g[i];
            }
            if (dS) dS[static_cast<long long>(t) * nv + v] = pack8(sv);
            if (do_prev) {
                float4* o = reinterpret_cast<float4*>(do_prev + static_cast<long long>(t) * d + 8 * v);
                const float4 a = o[0], b = o[1];
                o[0] = make_float4(a.x + sv[0], a.y + sv[1], a.z + sv[2], a.w + sv[3]);
                o[1] = make_float4(b.x + sv[4], b.y + sv[5], b.z + sv[6], b.w + sv[7]);
            }
        }
    }
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
        float a = acc[s];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0 && s < k) dw[static_cast<long long>(t) * k + s] = a;
    }
}

// Dispatch backward, one warp per token: du[t] += sum_s dx_perm[pos[t, s]] (fp32, slot order).
__global__ void __launch_bounds__(kBwdWarps * 32)
gather_sum_kernel(const uint4* __restrict__ dx_perm, const int32_t* __restrict__ pos, int T, int d, int k,
                  float* __restrict__ du) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int nv = d / 8;
    const int my_p = lane < k ? pos[static_cast<long long>(t) * k + lane] : -1;
    // steps counted for the whole warp: every lane takes part in the shuffles
    for (int v0 = 0; v0 < nv; v0 += 32) {
        const int v = v0 + lane;
        const bool act = v < nv;
        float sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int s = 0; s < k; ++s) {
            const int p = __shfl_sync(0xffffffffu, my_p, s);
            if (p < 0 || !act) continue;
            float x[8];
            unpack8(__ldg(dx_perm + static_cast<long long>(p) * nv + v), x);
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] += x[i];
        }
        if (!act) continue;
        float4* o = reinterpret_cast<float4*>(du + static_cast<long long>(t) * d + 8 * v);
        const float4 a = o[0], b = o[1];
        o[0] = make_float4(a.x + sum[0], a.y + sum[1], a.z + sum[2], a.w + sum[3]);
        o[1] = make_float4(b.x + sum[4], b.y + sum[5], b.z + sum[6], b.w + sum[7]);
    }
}

// Gate-rule backward, one warp per token: dz = d w / d z applied to dw (z =
// logits + bias; the chosen experts e_s with weights w_s), written as bf16 into
// a dense row of E_pad columns (zeros elsewhere):
//   SOFTMAX         dz_j = -c p_j + [j = e_s] dw_s w_s,  c = sum_s dw_s w_s
//   SOFTMAX_RENORM  dz_{e_r} = w_r (dw_r - c)
//   SIGMOID         dz_{e_s} = dw_s sig (1 - sig)
//   SIGMOID_NORM    dz_{e_r} = (dw_r - c) / sum_s sig_s * sig_r (1 - sig_r)
__global__ void __launch_bounds__(kBwdWarps * 32)
gate_backward_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                     const int32_t* __restrict__ idx, const float* __restrict__ w, const float* __restrict__ dw, int T,
                     int E, int E_pad, int k, int gate, __nv_bfloat16* __restrict__ dz, int* err) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kBwdWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* z = logits + static_cast<long long>(t) * E;
    const int32_t* e = idx + static_cast<long long>(t) * k;
    const float* ws = w + static_cast<long long>(t) * k;
    const float* dws = dw + static_cast<long long>(t) * k;
    float c = 0.0f;
    for (int s = 0; s < k; ++s) c += dws[s] * ws[s];
    __nv_bfloat16* out = dz + static_cast<long long>(t) * E_pad;
    if (gate == 0) {   // softmax over all experts
        const int e0 = e[0];
        if (e0 < 0 || e0 >= E) { set_dev_error(err, DEV_ERR_EXPERT_INDEX); return; }
        const float zmax = z[e0] + (bias ? bias[e0] : 0.0f);
        float den = 0.0f;
        for (int j = lane; j < E; j += 32) den += __expf(z[j] + (bias ? bias[j] : 0.0f) - zmax);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        for (int j = lane; j < E_pad; j += 32) {
            float v = 0.0f;
            if (j < E) {
                v = -c * (__expf(z[j] + (bias ? bias[j] : 0.0f) - zmax) / den);
                for (int s = 0; s < k; ++s)
                    if (e[s] == j) v += dws[s] * ws[s];
            }
            out[j] = __float2bfloat16_rn(v);
        }
        return;
    }
    for (int j = lane; j < E_pad; j += 32) out[j] = __float2bfloat16_rn(0.0f);
    __syncwarp();
    float den = 0.0f;
    if (gate == 3)
        for (int s = 0; s < k; ++s) {
            const int j = e[s];
            if (j >= 0 && j < E) den += 1.0f / (1.0f + __expf(-(z[j] + (bias ? bias[j] : 0.0f))));
        }
    if (lane < k) {
        const int j = e[lane];
        if (j < 0 || j >= E) { set_dev_error(err, DEV_ERR_EXPERT_INDEX); return; }
        float v;
        if (gate == 1) {
            v = ws[lane] * (dws[lane] - c);
        } else {
            const float sg = 1.0f / (1.0f + __expf(-(z[j] + (bias ? bias[j] : 0.0f))));
            v = gate == 2 ? dws[lane] * sg * (1.0f - sg) : (dws[lane] - c) / den * sg * (1.0f - sg);
        }
        out[j] = __float2bfloat16_rn(v);
    }
}

// Transposed weight packs for the input-gradient GEMMs, in the tiled bf16
// layout [G][ceil(N'/256)][K'/64][256][64] of the forward packs; one CTA per
// 32 KB block, thread r = packed row n', 64 consecutive K' elements.
//   mode 0: W13^T  -- n' = i < d, k' = packed gate/up row q < 2c (the page's W1
//                    (up), W2 (gate) [G, c, d])
//   mode 1: W3^T   -- n' = j < c, k' = i < d (W3 [G, d, c])
//   mode 2: W3cat^T -- n' = jj < ns cs, k' = i < d (w3s [ns, d, cs] side by side)
//   mode 3: W_R^T  -- n' = i < d, k' = j < K' (W_R [E, d]; j >= E is zero)
struct TSrc {
    const __nv_bfloat16* a;
    const __nv_bfloat16* b;
    int mode, Np, Kp, c, d, cs, E;
    __device__ __forceinline__ float at(long long g, int n, int k) const {
        switch (mode) {
            case 0: {
                const int blk = k >> 7, within = k & 127;
                const bool gate = within < 64;
                const long long row = g * c + blk * 64 + (gate ? within : within - 64);
                return __bfloat162float((gate ? b : a)[row * d + n]);
            }
            case 1: return __bfloat162float(a[(g * d + k) * c + n]);
            case 2: return __bfloat162float(a[(static_cast<long long>(n / cs) * d + k) * cs + n % cs]);
            default: return k < E ? __bfloat162float(a[static_cast<long long>(k) * d + n]) : 0.0f;
        }
    }
};

__global__ void __launch_bounds__(256) pack_t_kernel(TSrc src, int NB, int KB, uint4* __restrict__ out) {
    const long long blk = blockIdx.x;
    const int kb = static_cast<int>(blk % KB);
    const long long gn = blk / KB;
    const int nb = static_cast<int>(gn % NB);
    const long long g = gn / NB;
    const int n = nb * 256 + threadIdx.x;
    uint4* dst = out + (blk * 256 + threadIdx.x) * 8;
#pragma unroll 1
    for (int q = 0; q < 8; ++q) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = n < src.Np ? src.at(g, n, kb * 64 + q * 8 + i) : 0.0f;
        dst[q] = pack8(v);
    }
}

// Self-test of the pipeline's bounded wait: one thread waits on an mbarrier
// that nothing arrives at, with the given limit, through the helper every
// GEMM wait uses; the wait gives up, records DEV_ERR_TIMEOUT and returns.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, err, limit_ns);
    }
}

__global__ void copy_u4_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

// --------------------------------------------------------------- launchers
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, dev_error_ptr());
    count_launch();
    return cudaGetLastError();
}

__global__ void zero_u4_kernel(uint4* __restrict__ dst, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_zero(void* dst, size_t bytes, cudaStream_t st) {
    const long long n = static_cast<long long>(bytes / 16);
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    if (blocks < 1) blocks = 1;
    zero_u4_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(static_cast<uint4*>(dst), n);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t st) {
    const long long n = static_cast<long long>(bytes / 16);
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    if (blocks < 1) blocks = 1;
    copy_u4_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                                               n);
    count_launch();
    return cudaGetLastError();
}

template <int KMAX>
static void launch_cb(const float* dO, const float* dOs, const void* y_perm, const int32_t* pos, const float* w,
                      int T, int d, int k, void* dy_perm, float* dw, void* dS, float* do_prev, cudaStream_t st) {
    combine_backward_kernel<KMAX><<<(T + kBwdWarps - 1) / kBwdWarps, kBwdWarps * 32, 0, st>>>(
        dO, dOs, static_cast<const uint4*>(y_perm), pos, w, T, d, k, static_cast<uint4*>(dy_perm), dw,
        static_cast<uint4*>(dS), do_prev);
}

cudaError_t launch_combine_backward(const float* dO, const float* dOs, const void* y_perm, const int32_t* pos,
                                    const float* topk_w, int T, int d, int k, void* dy_perm, float* dw, void* dS,
                                    float* do_prev, cudaStream_t st) {
    if (k <= 8) launch_cb<8>(dO, dOs, y_perm, pos, topk_w, T, d, k, dy_perm, dw, dS, do_prev, st);
    else launch_cb<16>(dO, dOs, y_perm, pos, topk_w, T, d, k, dy_perm, dw, dS, do_prev, st);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gather_sum(const void* dx_perm, const int32_t* pos, int T, int d, int k, float* du,
                              cudaStream_t st) {
    gather_sum_kernel<<<(T + kBwdWarps - 1) / kBwdWarps, kBwdWarps * 32, 0, st>>>(static_cast<const uint4*>(dx_perm),
                                                                                   pos, T, d, k, du);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gate_backward(const float* logits, const float* bias, const int32_t* idx, const float* w,
                                 const float* dw, int T, int E, int E_pad, int k, int gate, void* dz,
                                 cudaStream_t st) {
    gate_backward_kernel<<<(T + kBwdWarps - 1) / kBwdWarps, kBwdWarps * 32, 0, st>>>(
        logits, bias, idx, w, dw, T, E, E_pad, k, gate, static_cast<__nv_bfloat16*>(dz), dev_error_ptr());
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pack_t(int mode, int G, int Np, int Kp, int c, int d, int cs, int E, const void* a, const void* b,
                          void* out, cudaStream_t st) {
    TSrc src{static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b), mode, Np, Kp, c, d, cs, E};
    const int NB = (Np + 255) / 256, KB = Kp / 64;
    const long long blocks = static_cast<long long>(G) * NB * KB;
    pack_t_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(src, NB, KB, static_cast<uint4*>(out));
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
