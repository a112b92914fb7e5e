// quant.cu -- FP8 E4M3 quantisation kernels of the FP8 expert path: bf16 rows
// to an FP8 row-scaled matrix (the hidden between the two expert GEMMs, the
// shared experts' token rows), and the one-time packing of bf16 expert weights
// into FP8 codes in the GEMM's tiled layout with one scale per output channel.
//
// Packed FP8 weights [G, N, K]: the codes in [G][ceil(N/256)][K/128][256][128]
// (every 256-row x 128-byte TMA box one contiguous 32 KB block, rows past N
// zero), then from byte G ceil(N/256) 256 K the G N fp32 row scales.
#include "fp8.cuh"
#include "kernels.h"

namespace fs {

// One warp per row (grid-stride): amax over the row, then the codes; the
// second pass re-reads the row, which the first pass left in L1/L2.
__global__ void __launch_bounds__(256)
quant_rows_kernel(const uint4* __restrict__ x, long long rows, int cols, uint8_t* __restrict__ q,
                  float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int nv = cols / 8;
    for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
        const uint4* src = x + r * nv;
        float amax = 0.0f;
        for (int v = lane; v < nv; v += 32) amax = fmaxf(amax, absmax_bf16x8(__ldg(src + v)));
        const RowQuant rq = row_quant(warp_max(amax));
        uint2* dst = reinterpret_cast<uint2*>(q + r * cols);
        if (!rq.wide) {
            for (int v = lane; v < nv; v += 32) dst[v] = quant_bf16x8(__ldg(src + v), rq.mult);
        } else {
            for (int v = lane; v < nv; v += 32) dst[v] = quant_bf16x8_wide(__ldg(src + v), rq.e);
        }
        if (lane == 0) scale[r] = rq.scale;
    }
}

// One warp per packed row (grid-stride over G * NB * 256 rows).
__global__ void __launch_bounds__(256)
pack_fp8_kernel(PackSrc src, int G, int NB, uint8_t* __restrict__ codes, float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int K = src.K, N = src.N, KB = K / 128, nv = K / 8;
    const long long total = static_cast<long long>(G) * NB * 256;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long R = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; R < total; R += nwarps) {
        const long long g = R / (static_cast<long long>(NB) * 256);
        const int nr = static_cast<int>(R - g * NB * 256);       // row inside the group, padded
        const int nb = nr >> 8, rr = nr & 255;
        uint8_t* blk0 = codes + ((g * NB + nb) * KB) * 32768LL + rr * 128;
        if (nr >= N) {
            for (int v = lane; v < nv; v += 32) {
                const int k = 8 * v;
                *reinterpret_cast<uint2*>(blk0 + (k >> 7) * 32768LL + (k & 127)) = make_uint2(0, 0);
            }
            continue;
        }
        float amax = 0.0f;
        for (int v = lane; v < nv; v += 32) amax = fmaxf(amax, absmax_bf16x8(__ldg(src.chunk(g, nr, v))));
        const RowQuant rq = row_quant(warp_max(amax));
        for (int v = lane; v < nv; v += 32) {
            const int k = 8 * v;
            *reinterpret_cast<uint2*>(blk0 + (k >> 7) * 32768LL + (k & 127)) = quant_bf16x8(__ldg(src.chunk(g, nr, v)), rq);
        }
        if (lane == 0) scales[g * N + nr] = rq.scale;
    }
}

static int grid_for(long long warps_needed) {
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = 152LL * 16;
    if (blocks > cap) blocks = cap;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

size_t packed_bytes_fp8(int G, int N, int K) {
    const size_t nb = (static_cast<size_t>(N) + 255) / 256;
    return static_cast<size_t>(G) * nb * 256 * K + static_cast<size_t>(G) * N * sizeof(float);
}

static size_t packed_codes_bytes_fp8(int G, int N, int K) {
    return static_cast<size_t>(G) * ((static_cast<size_t>(N) + 255) / 256) * 256 * K;
}

const float* packed_scales_fp8(const void* packed, int G, int N, int K) {
    return reinterpret_cast<const float*>(static_cast<const uint8_t*>(packed) + packed_codes_bytes_fp8(G, N, K));
}

static cudaError_t launch_pack_fp8(const PackSrc& src, int G, void* out, cudaStream_t st) {
    const int NB = (src.N + 255) / 256;
    uint8_t* codes = static_cast<uint8_t*>(out);
    float* scales = reinterpret_cast<float*>(codes + packed_codes_bytes_fp8(G, src.N, src.K));
    pack_fp8_kernel<<<grid_for(static_cast<long long>(G) * NB * 256), 256, 0, st>>>(src, G, NB, codes, scales);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pack_w13_fp8(int G, int c, int d, const void* w1, const void* w2, void* w13, cudaStream_t st) {
    PackSrc s{static_cast<const uint4*>(w1), static_cast<const uint4*>(w2), 0, 2 * c, d, c, 0};
    return launch_pack_fp8(s, G, w13, st);
}

cudaError_t launch_pack_w3_fp8(int G, int d, int c, const void* w3, void* w3p, cudaStream_t st) {
    PackSrc s{static_cast<const uint4*>(w3), nullptr, 1, d, c, 0, 0};
    return launch_pack_fp8(s, G, w3p, st);
}

cudaError_t launch_pack_w3_shared_fp8(int ns, int cs, int d, const void* w3s, void* w3cat, cudaStream_t st) {
    PackSrc s{static_cast<const uint4*>(w3s), nullptr, 2, d, ns * cs, 0, cs};
    return launch_pack_fp8(s, 1, w3cat, st);
}

cudaError_t launch_quant_rows(const void* x, long long rows, int cols, void* q, cudaStream_t st) {
    uint8_t* codes = static_cast<uint8_t*>(q);
    float* scale = reinterpret_cast<float*>(codes + fp8_scale_offset(rows, cols));
    quant_rows_kernel<<<grid_for(rows), 256, 0, st>>>(static_cast<const uint4*>(x), rows, cols, codes, scale);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
