// pack.cu -- one-time weight repacking into the layouts the GEMMs read.
//
// Gate/up interleave ("FarSkip-Collective", §2.1 MLP equation): for every block
// b of 64 expert columns, rows [128b, 128b+64) of the packed gate/up matrix hold
// W2 (gate) rows [64b, 64b+64) and rows [128b+64, 128b+128) hold W1 (up) rows,
// so one 256-row tile of the gate/up GEMM carries both SwiGLU operands of 128
// expert columns.  Shared experts: their down projections side by side along
// the expert width (the TP-slicing identity of §2.1 read backwards: summing the
// partial MLPs equals one MLP over the concatenated width).
//
// bf16 weights (tensor-core path) are further tiled for HBM streaming: a
// matrix [G, N, K] is stored as [G][ceil(N/256)][K/64][256][64], so every
// 256-row x 64-column TMA box is one contiguous 32 KB block (rows past N are
// zero).  fp32 weights (fp32 FMA path) stay row-major.
#include "common.cuh"
#include "kernels.h"

namespace fs {

static inline long long nblk(int N) { return (N + 255) / 256; }

size_t packed_bytes(int G, int N, int K, int elem_bytes) {
    if (elem_bytes == 2) return static_cast<size_t>(G) * nblk(N) * 256 * K * 2;
    return static_cast<size_t>(G) * N * K * elem_bytes;
}

// source row (element offset of its start) of packed gate/up row n of group g,
// or -1 past the end
__device__ __forceinline__ long long w13_src_row(long long g, int n, int c, int d, bool& from_gate) {
    if (n >= 2 * c) return -1;
    const int blk = n >> 7, within = n & 127;
    from_gate = within < 64;
    const long long r = g * c + blk * 64 + (from_gate ? within : within - 64);
    return r * d;
}

// tiled bf16: one CTA per 32 KB block (g, nb, kb), one thread per row of the block
__global__ void __launch_bounds__(256)
pack_w13_tiled_kernel(const uint4* __restrict__ w1, const uint4* __restrict__ w2, uint4* __restrict__ out, int c,
                      int d, int NB, int KB) {
    const long long blk = blockIdx.x;
    const int kb = static_cast<int>(blk % KB);
    const long long gn = blk / KB;
    const int nb = static_cast<int>(gn % NB);
    const long long g = gn / NB;
    const int r = threadIdx.x;
    bool gate = false;
    const long long src = w13_src_row(g, nb * 256 + r, c, d, gate);
    uint4* dst = out + (blk * 256 + r) * 8;          // 64 bf16 = 8 x 16 B
    if (src < 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* s = (gate ? w2 : w1) + (src + static_cast<long long>(kb) * 64) / 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = s[j];
}

// tiled bf16 of a plain [G, N, K] matrix (the routed down projections)
__global__ void __launch_bounds__(256)
pack_tiled_kernel(const uint4* __restrict__ w, uint4* __restrict__ out, int N, int K, int NB, int KB) {
    const long long blk = blockIdx.x;
    const int kb = static_cast<int>(blk % KB);
    const long long gn = blk / KB;
    const int nb = static_cast<int>(gn % NB);
    const long long g = gn / NB;
    const int r = threadIdx.x;
    const int n = nb * 256 + r;
    uint4* dst = out + (blk * 256 + r) * 8;
    if (n >= N) {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4* s = w + ((g * N + n) * static_cast<long long>(K) + static_cast<long long>(kb) * 64) / 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = s[j];
}

// tiled bf16 of the shared experts' concatenated down projection [d, ns cs]:
// element (i, s cs + j) = w3s[s][i][j]
__global__ void __launch_bounds__(256)
pack_w3_shared_tiled_kernel(const uint4* __restrict__ w3s, uint4* __restrict__ out, int ns, int cs, int d, int NB,
                            int KB) {
    const long long blk = blockIdx.x;
    const int kb = static_cast<int>(blk % KB);
    const int nb = static_cast<int>(blk / KB);
    const int r = threadIdx.x;
    const int i = nb * 256 + r;
    uint4* dst = out + (blk * 256 + r) * 8;
    if (i >= d) {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = make_uint4(0, 0, 0, 0);
        return;
    }
    const int col = kb * 64;
    const int s_idx = col / cs, j0 = col - s_idx * cs;     // cs % 64 == 0: a block never straddles two experts
    const uint4* s = w3s + ((static_cast<long long>(s_idx) * d + i) * cs + j0) / 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = s[j];
}

// ---- fp32 (row-major) layouts
__global__ void pack_w13_kernel(const uint4* __restrict__ w1, const uint4* __restrict__ w2, uint4* __restrict__ w13,
                                int c, int row_vecs, long long total_rows) {
    const long long r = blockIdx.x * static_cast<long long>(blockDim.y) + threadIdx.y;   // row of w13
    if (r >= total_rows) return;
    const long long g = r / (2LL * c);
    const int rr = static_cast<int>(r - g * 2LL * c);
    const int blk = rr >> 7, within = rr & 127;
    const uint4* src = (within < 64) ? w2 + (g * c + blk * 64 + within) * row_vecs
                                     : w1 + (g * c + blk * 64 + within - 64) * row_vecs;
    uint4* dst = w13 + r * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) dst[i] = src[i];
}

__global__ void pack_w3_shared_kernel(const uint4* __restrict__ w3s, uint4* __restrict__ w3cat, int ns, int d,
                                      int cs_vecs) {
    const long long r = blockIdx.x * static_cast<long long>(blockDim.y) + threadIdx.y;   // (i, s) pair
    if (r >= static_cast<long long>(d) * ns) return;
    const int i = static_cast<int>(r / ns), s = static_cast<int>(r % ns);
    const uint4* src = w3s + (static_cast<long long>(s) * d + i) * cs_vecs;
    uint4* dst = w3cat + (static_cast<long long>(i) * ns + s) * cs_vecs;
    for (int j = threadIdx.x; j < cs_vecs; j += blockDim.x) dst[j] = src[j];
}

__global__ void copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_pack_w13(int G, int c, int d, int elem_bytes, const void* w1, const void* w2, void* w13,
                            cudaStream_t st) {
    if (elem_bytes == 2) {
        const int NB = static_cast<int>(nblk(2 * c)), KB = d / 64;
        const long long blocks = static_cast<long long>(G) * NB * KB;
        pack_w13_tiled_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
            static_cast<const uint4*>(w1), static_cast<const uint4*>(w2), static_cast<uint4*>(w13), c, d, NB, KB);
    } else {
        const int row_vecs = d * elem_bytes / 16;
        const long long rows = 2LL * G * c;
        dim3 block(32, 8);
        pack_w13_kernel<<<static_cast<unsigned>((rows + 7) / 8), block, 0, st>>>(
            static_cast<const uint4*>(w1), static_cast<const uint4*>(w2), static_cast<uint4*>(w13), c, row_vecs,
            rows);
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pack_w3(int G, int d, int c, int elem_bytes, const void* w3, void* w3p, cudaStream_t st) {
    if (elem_bytes == 2) {
        const int NB = static_cast<int>(nblk(d)), KB = c / 64;
        const long long blocks = static_cast<long long>(G) * NB * KB;
        pack_tiled_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint4*>(w3),
                                                                          static_cast<uint4*>(w3p), d, c, NB, KB);
    } else {
        const long long n = static_cast<long long>(G) * d * c * elem_bytes / 16;
        copy_kernel<<<1024, 256, 0, st>>>(static_cast<const uint4*>(w3), static_cast<uint4*>(w3p), n);
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pack_w3_shared(int ns, int cs, int d, int elem_bytes, const void* w3s, void* w3cat,
                                  cudaStream_t st) {
    if (elem_bytes == 2) {
        const int NB = static_cast<int>(nblk(d)), KB = ns * cs / 64;
        const long long blocks = static_cast<long long>(NB) * KB;
        pack_w3_shared_tiled_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
            static_cast<const uint4*>(w3s), static_cast<uint4*>(w3cat), ns, cs, d, NB, KB);
    } else {
        const int cs_vecs = cs * elem_bytes / 16;
        const long long rows = static_cast<long long>(d) * ns;
        dim3 block(32, 8);
        pack_w3_shared_kernel<<<static_cast<unsigned>((rows + 7) / 8), block, 0, st>>>(
            static_cast<const uint4*>(w3s), static_cast<uint4*>(w3cat), ns, d, cs_vecs);
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
