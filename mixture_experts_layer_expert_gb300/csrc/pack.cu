// pack.cu -- one-time weight repacking into the layouts the GEMMs read.
//
// w13 [G, 2c, d]: for every block b of 64 expert columns, rows [128b, 128b+64)
// hold W2 (gate) rows [64b, 64b+64) and rows [128b+64, 128b+128) hold W1 (up)
// rows, so one 256-row tile of the gate/up GEMM carries both operands of the
// SwiGLU product for 128 expert columns ("FarSkip-Collective", §2.1 MLP equation).
// w3cat [d, ns cs]: the shared experts' down projections side by side along the
// expert width (the TP-slicing identity of §2.1 read backwards: summing the
// partial MLPs equals one MLP over the concatenated width).
#include "common.cuh"
#include "kernels.h"

namespace fs {

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

cudaError_t launch_pack_w13(int G, int c, int d, int elem_bytes, const void* w1, const void* w2, void* w13,
                            cudaStream_t st) {
    const int row_vecs = d * elem_bytes / 16;
    const long long rows = 2LL * G * c;
    dim3 block(32, 8);
    const long long grid = (rows + 7) / 8;
    pack_w13_kernel<<<static_cast<unsigned>(grid), block, 0, st>>>(
        static_cast<const uint4*>(w1), static_cast<const uint4*>(w2), static_cast<uint4*>(w13), c, row_vecs, rows);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pack_w3_shared(int ns, int cs, int d, int elem_bytes, const void* w3s, void* w3cat,
                                  cudaStream_t st) {
    const int cs_vecs = cs * elem_bytes / 16;
    const long long rows = static_cast<long long>(d) * ns;
    dim3 block(32, 8);
    pack_w3_shared_kernel<<<static_cast<unsigned>((rows + 7) / 8), block, 0, st>>>(
        static_cast<const uint4*>(w3s), static_cast<uint4*>(w3cat), ns, d, cs_vecs);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
