// mx.cuh -- block-scaled FP8 (MX) operand layouts of the MX expert path.
//
// Every operand row of an expert GEMM is cut, along the contraction, into
// blocks of 32 elements; each block is E4M3 codes times its own power-of-two
// scale 2^e (e the smallest integer with max |x_i| 2^-e <= 448, clamped to the
// UE8M0 range [-127, 127]), stored as the UE8M0 byte e + 127.  The tensor
// cores apply both operands' block scales inside the contraction
// (tcgen05.mma kind::mxf8f6f4.block_scale, scale factors in TMEM).
//
// Scale-factor bytes are kept in the arrangement the scale-factor copy into
// TMEM (tcgen05.cp 32x128b.warpx4) takes: for a group of 128 rows and one
// 128-element stage of the contraction (4 blocks), a 512-byte chunk whose byte
// (m % 32) * 16 + (m / 32) * 4 + b holds row m's scale of block b.
//   MX matrix [rows, cols] (activations): codes [rows128][cols] row-major
//     (rows128 = rows rounded up to 128), then from a 256-byte boundary the
//     chunks [rows128 / 128][cols / 128][512].
//   MX weights [G, N, K]: codes tiled as the FP8 weights
//     [G][ceil(N/256)][K/128][256][128], then the chunks
//     [G][ceil(N/256)][K/128][2][512] (the two 128-row halves of a 256-row tile).
#pragma once

#include "fp8.cuh"

namespace fs {

constexpr int kMxBlock = 32;

__host__ __device__ inline long long mx_rows128(long long rows) { return (rows + 127) / 128 * 128; }
__host__ __device__ inline size_t mx_sf_offset(long long rows, int cols) {
    return (static_cast<size_t>(mx_rows128(rows)) * static_cast<size_t>(cols) + 255) / 256 * 256;
}
__host__ __device__ inline size_t mx_rows_bytes(long long rows, int cols) {
    return mx_sf_offset(rows, cols) + static_cast<size_t>(mx_rows128(rows) / 128) * (cols / 128) * 512;
}
// Byte of row m's scale of block b (32 elements) in an MX matrix's chunks.
__host__ __device__ inline size_t mx_sf_byte(long long m, int b, int cols) {
    return (static_cast<size_t>(m >> 7) * (cols >> 7) + (b >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 +
           (b & 3);
}
// Weights: tile nt of group g, row r of the 256-row tile, block b along K.
__host__ __device__ inline size_t mx_w_sf_byte(long long g, int NB, int nt, int r, int b, int K) {
    return ((static_cast<size_t>(g) * NB + nt) * (K >> 7) + (b >> 2)) * 1024 + (r >> 7) * 512 + (r & 31) * 16 +
           ((r & 127) >> 5) * 4 + (b & 3);
}
inline size_t mx_w_codes_bytes(int G, int N, int K) {
    return static_cast<size_t>(G) * ((static_cast<size_t>(N) + 255) / 256) * 256 * K;
}
inline size_t mx_w_bytes(int G, int N, int K) {
    return mx_w_codes_bytes(G, N, K) + static_cast<size_t>(G) * ((N + 255) / 256) * (K / 128) * 1024;
}

// Quantisation of one block from its largest magnitude: the UE8M0 byte and the
// multiplier 2^-e (fp32 normal unless `wide`, then applied in double).
struct MxQuant {
    RowQuant q;
    uint8_t ue8m0;
};
__device__ __forceinline__ MxQuant mx_quant(float amax) {
    int e = fp8_row_exp(amax);
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    MxQuant m;
    m.q.e = e;
    m.q.wide = (e < -127 || e > 126);
    m.q.mult = m.q.wide ? 0.0f : __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    m.q.scale = 0.0f;   // not used: the scale travels as the UE8M0 byte
    m.ue8m0 = static_cast<uint8_t>(e + 127);
    return m;
}

// Largest magnitude over the 4-lane group holding one 32-element block (lanes
// 4q .. 4q+3 of the warp, 8 elements each).
__device__ __forceinline__ float group4_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
    return v;
}

}  // namespace fs
