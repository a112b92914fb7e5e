// dispatch.cu -- local Dispatch: stable counting sort of (token, slot) pairs by
// expert and the permuted copy of the token rows.
//
// "FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
// Models", §2.1 Dispatch paragraph: tokens are grouped by the experts the
// router chose for them and the activations are permuted accordingly (on one
// GPU the all-to-all that follows is a local copy).  The order is deterministic
// and stable: expert-major, token order inside an expert.
//
// Four launches, no atomics on global memory, no host synchronisation:
//   1 count   chunk of 1024 tokens per CTA -> per-chunk expert histogram
//   2 scan    one CTA: column scan over chunks, counts, exclusive offsets
//   3 rank    chunk per CTA, one warp per 32 tokens: lane bitmasks per expert
//             give the rank inside the warp, a scan over the CTA's warps the
//             rank inside the chunk -> pos[t k + s], perm_src[p]
//   4 copy    one warp per token: read the row of u once (16-byte vectors),
//             write it to its k permuted rows
#include <mutex>

#include "common.cuh"
#include "fp8.cuh"
#include "kernels.h"

namespace fs {

constexpr int kChunk = 1024;          // tokens per chunk (= threads of count/rank CTAs)
constexpr int kChunkWarps = kChunk / 32;

static inline int n_chunks(int T) { return (T + kChunk - 1) / kChunk; }

size_t dispatch_ws_bytes(int T, int E) { return static_cast<size_t>(n_chunks(T)) * E * sizeof(int32_t); }

__global__ void __launch_bounds__(kChunk)
dispatch_count_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k, int32_t* __restrict__ chunk_hist,
                      int* err) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t = blockIdx.x * kChunk + threadIdx.x;
    if (t < T) {
        for (int s = 0; s < k; ++s) {
            const int e = topk_idx[static_cast<long long>(t) * k + s];
            if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
            else set_dev_error(err, DEV_ERR_EXPERT_INDEX);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_hist[static_cast<long long>(blockIdx.x) * E + e] = hist[e];
}

// One CTA of 1024 threads; thread e owns expert e (E <= 1024).
// pad128: each expert's segment starts at a multiple of 128 rows (the MX
// path): offsets are the exclusive prefix of the counts rounded up to 128.
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks, int E, int32_t* __restrict__ counts,
                     int32_t* __restrict__ offsets, int pad128) {
    __shared__ int warp_sums[32];
    const int e = threadIdx.x;
    int total = 0;
    if (e < E) {
        int b = 0;
        for (; b + 8 <= nchunks; b += 8) {        // 8 independent loads in flight
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = chunk_hist[static_cast<long long>(b + j) * E + e];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                chunk_hist[static_cast<long long>(b + j) * E + e] = total;
                total += c[j];
            }
        }
        for (; b < nchunks; ++b) {
            const int c = chunk_hist[static_cast<long long>(b) * E + e];
            chunk_hist[static_cast<long long>(b) * E + e] = total;
            total += c;
        }
        counts[e] = total;
    }
    // exclusive scan of totals over experts
    const int lane = e & 31, wid = e >> 5;
    const int seg = pad128 ? (total + 127) / 128 * 128 : total;
    int v = seg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int excl = v - seg + (wid > 0 ? warp_sums[wid - 1] : 0);
    if (e < E) {
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + seg;
        for (int b = 0; b < nchunks; ++b) chunk_hist[static_cast<long long>(b) * E + e] += excl;
    }
}

// chunk_base[b][e] = first permuted row of expert e for chunk b.
__global__ void __launch_bounds__(kChunk)
dispatch_rank_kernel(const int32_t* __restrict__ topk_idx, int T, int E, int k,
                     const int32_t* __restrict__ chunk_base, int32_t* __restrict__ pos,
                     int32_t* __restrict__ perm_src) {
    extern __shared__ uint32_t wmask[];     // [kChunkWarps][E]: lane masks, then counts, then prefixes
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) wmask[i] = 0;
    __syncthreads();
    const int t = blockIdx.x * kChunk + threadIdx.x;
    int ex[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
        ex[s] = -1;
        if (s < k && t < T) {
            const int e = topk_idx[static_cast<long long>(t) * k + s];
            if (e >= 0 && e < E) {
                ex[s] = e;
                atomicOr(&wmask[w * E + e], 1u << lane);
            }
        }
    }
    __syncwarp();
    const uint32_t lt = (1u << lane) - 1u;
    int rank[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) rank[s] = ex[s] >= 0 ? __popc(wmask[w * E + ex[s]] & lt) : 0;
    __syncthreads();
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) wmask[i] = __popc(wmask[i]);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        uint32_t run = 0;
        for (int ww = 0; ww < kChunkWarps; ++ww) {
            const uint32_t c = wmask[ww * E + e];
            wmask[ww * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    if (t < T) {
        const int32_t* base = chunk_base + static_cast<long long>(blockIdx.x) * E;
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s) {
            if (s >= k) break;
            int p = -1;
            if (ex[s] >= 0) {
                p = base[ex[s]] + static_cast<int>(wmask[w * E + ex[s]]) + rank[s];
                perm_src[p] = t;
            }
            pos[static_cast<long long>(t) * k + s] = p;
        }
    }
}

constexpr int kCopyWarps = 8;

// One warp per token: x_perm[pos[t, s]] = u[t] for every slot s.
__global__ void __launch_bounds__(kCopyWarps * 32)
dispatch_copy_kernel(const uint4* __restrict__ u, int T, int row_vecs, int k, const int32_t* __restrict__ pos,
                     uint4* __restrict__ x_perm, int nch, int cpc) {
    const int lane = threadIdx.x & 31;
    const long long wid = static_cast<long long>(blockIdx.x) * kCopyWarps + (threadIdx.x >> 5);
    const int t = static_cast<int>(wid / nch);
    if (t >= T) return;
    // this warp's run of cpc 128-vector steps of the row (the whole row when nch = 1)
    const int i_begin = static_cast<int>(wid - static_cast<long long>(t) * nch) * cpc * 128;
    const int i_end = min(row_vecs, i_begin + cpc * 128);
    const int my_p = lane < k ? pos[static_cast<long long>(t) * k + lane] : -1;
    const uint4* src = u + static_cast<long long>(t) * row_vecs;
    for (int i0 = i_begin; i0 < i_end; i0 += 4 * 32) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * 32 + lane;
            if (i < i_end) v[j] = __ldg(src + i);
        }
        for (int s = 0; s < k; ++s) {
            const int p = __shfl_sync(0xffffffffu, my_p, s);
            if (p < 0) continue;
            uint4* dst = x_perm + static_cast<long long>(p) * row_vecs;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * 32 + lane;
                if (i < i_end) dst[i] = v[j];
            }
        }
    }
}

// FP8 expert path: one warp per token quantises u[t] once (one power-of-two
// scale for the row) and writes its E4M3 codes to every slot's row of x_q and,
// when u_q is set, to row t of u_q (the shared experts' operand); each row's
// scale goes with it.
__global__ void __launch_bounds__(kCopyWarps * 32)
dispatch_copy_fp8_kernel(const uint4* __restrict__ u, int T, int d, int k, const int32_t* __restrict__ pos,
                         uint8_t* __restrict__ x_q, float* __restrict__ x_scale, uint8_t* __restrict__ u_q,
                         float* __restrict__ u_scale) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kCopyWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int nv = d / 8;
    const int my_p = lane < k ? pos[static_cast<long long>(t) * k + lane] : -1;
    const uint4* src = u + static_cast<long long>(t) * nv;
    float amax = 0.0f;
    for (int v = lane; v < nv; v += 32) amax = fmaxf(amax, absmax_bf16x8(__ldg(src + v)));
    const RowQuant rq = row_quant(warp_max(amax));
    for (int v0 = 0; v0 < nv; v0 += 4 * 32) {
        uint2 c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int v = v0 + j * 32 + lane;
            if (v < nv) c[j] = quant_bf16x8(__ldg(src + v), rq);
        }
        for (int s = 0; s < k; ++s) {
            const int p = __shfl_sync(0xffffffffu, my_p, s);
            if (p < 0) continue;
            uint2* dst = reinterpret_cast<uint2*>(x_q + static_cast<long long>(p) * d);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = v0 + j * 32 + lane;
                if (v < nv) dst[v] = c[j];
            }
        }
        if (u_q) {
            uint2* dst = reinterpret_cast<uint2*>(u_q + static_cast<long long>(t) * d);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int v = v0 + j * 32 + lane;
                if (v < nv) dst[v] = c[j];
            }
        }
    }
    if (my_p >= 0) x_scale[my_p] = rq.scale;
    if (u_q && lane == 0) u_scale[t] = rq.scale;
}

static cudaError_t set_smem_attr(const void* fn, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

cudaError_t launch_dispatch(const int32_t* topk_idx, const void* u, int T, int d, int E, int k, int elem_bytes,
                            int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src, void* x_perm,
                            int32_t* scratch, cudaStream_t st, int qmode, void* u_q, long long rows_cap) {
    const bool fp8 = qmode == kQuantRow;
    const int nc = n_chunks(T);
    int* err = dev_error_ptr();
    dispatch_count_kernel<<<nc, kChunk, E * sizeof(int32_t), st>>>(topk_idx, T, E, k, scratch, err);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dispatch_scan_kernel<<<1, 1024, 0, st>>>(scratch, nc, E, counts, offsets, qmode == kQuantMx ? 1 : 0);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t rank_smem = static_cast<size_t>(kChunkWarps) * E * sizeof(uint32_t);
    e = set_smem_attr(reinterpret_cast<const void*>(dispatch_rank_kernel), rank_smem);
    if (e != cudaSuccess) return e;
    dispatch_rank_kernel<<<nc, kChunk, rank_smem, st>>>(topk_idx, T, E, k, scratch, pos, perm_src);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!x_perm) return cudaSuccess;     // the caller gathers rows itself (no permuted copy)
    if (qmode == kQuantMx) return launch_dispatch_copy_mx(u, T, d, k, pos, x_perm, rows_cap, u_q, st);
    if (fp8) {
        const long long rows = static_cast<long long>(T) * k;
        uint8_t* xq = static_cast<uint8_t*>(x_perm);
        uint8_t* uq = static_cast<uint8_t*>(u_q);
        dispatch_copy_fp8_kernel<<<(T + kCopyWarps - 1) / kCopyWarps, kCopyWarps * 32, 0, st>>>(
            reinterpret_cast<const uint4*>(u), T, d, k, pos, xq, reinterpret_cast<float*>(xq + fp8_scale_offset(rows, d)),
            uq, uq ? reinterpret_cast<float*>(uq + fp8_scale_offset(T, d)) : nullptr);
        count_launch();
        return cudaGetLastError();
    }
    const int row_vecs = d * elem_bytes / 16;
    // one warp per token, or for few tokens per run of 128-vector steps (about 16K warps wanted)
    const int steps = (row_vecs + 127) / 128;
    const int want = T >= 16384 ? 1 : (16384 + T - 1) / T;
    const int cpc = (steps + want - 1) / want;
    const int nch = (steps + cpc - 1) / cpc;
    const long long warps = static_cast<long long>(T) * nch;
    dispatch_copy_kernel<<<static_cast<int>((warps + kCopyWarps - 1) / kCopyWarps), kCopyWarps * 32, 0, st>>>(
        reinterpret_cast<const uint4*>(u), T, row_vecs, k, pos, reinterpret_cast<uint4*>(x_perm), nch, cpc);
    count_launch();
    return cudaGetLastError();
}

// ------------------------------------------------ dispatch without allocation
// Scratch of fs_dispatch_noalloc: the per-chunk expert histogram lives in this
// file-scope device array instead of a caller-provided workspace.  It is loaded
// with the library on every GPU that loads it and stays until the process exits.
static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticDispatchScratchInts];

static int32_t* g_dispatch_scratch_ptr[64] = {nullptr};
static std::mutex g_dispatch_scratch_mu;

// Device address of g_dispatch_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
static cudaError_t dispatch_scratch_address(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dispatch_scratch_mu);
    if (!g_dispatch_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess) return e;
        g_dispatch_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_dispatch_scratch_ptr[dev];
    return cudaSuccess;
}

cudaError_t launch_dispatch_noalloc(const int32_t* topk_idx, const void* u, int T, int d, int E, int k, int elem_bytes,
                                    int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* perm_src,
                                    void* x_perm, cudaStream_t st, int qmode, long long rows_cap) {
    int32_t* scratch = nullptr;
    cudaError_t e = dispatch_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    return launch_dispatch(topk_idx, u, T, d, E, k, elem_bytes, counts, offsets, pos, perm_src, x_perm, scratch, st,
                           qmode, nullptr, rows_cap);
}

}  // namespace fs
