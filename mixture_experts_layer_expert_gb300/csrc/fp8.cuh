// fp8.cuh -- FP8 E4M3 row quantisation used by the FP8 expert path: the
// Dispatch copy (token rows), the hidden quantisation between the two expert
// GEMMs, and the weight packing (output-channel rows).
//
// The pages run inference with FP8 quantisation and fused MoE forward kernels
// ("FarSkip-Collective" summary, experimental setup, software configuration:
// inference parameters) without naming a format; here every operand row of an
// expert GEMM, along the contraction, is E4M3 codes times one power-of-two
// scale 2^e, e the smallest integer with max_i |x_i| 2^-e <= 448 (the largest
// finite E4M3 magnitude).  A power of two makes x 2^-e exact, so the only
// rounding is the E4M3 conversion (nearest, ties to even, saturating), and the
// row scale multiplies whole rows of the contraction, so it factors out of the
// GEMM's sum into its epilogue.
#pragma once

#include "common.cuh"

namespace fs {

// Byte layout of an FP8 row-scaled matrix [rows, cols]: the codes row-major,
// then the rows fp32 scales from the next 256-byte boundary.
__host__ __device__ inline size_t fp8_scale_offset(long long rows, int cols) {
    return (static_cast<size_t>(rows) * static_cast<size_t>(cols) + 255) / 256 * 256;
}
__host__ __device__ inline size_t fp8_rows_bytes(long long rows, int cols) {
    return fp8_scale_offset(rows, cols) + static_cast<size_t>(rows) * sizeof(float);
}

// Quantisation parameters of one row from its largest magnitude.
struct RowQuant {
    float scale;   // 2^e: the dequantisation factor stored with the row
    float mult;    // 2^-e when representable as a normal fp32 (wide == false)
    int e;
    bool wide;     // 2^-e outside the fp32 normal range: scale in double
};

__device__ __forceinline__ int fp8_row_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    const uint32_t b = __float_as_uint(amax);
    const int ef = static_cast<int>((b >> 23) & 0xFFu);
    if (ef == 0) {            // subnormal amax: exact search in double
        const double a = amax;
        int s = -160;
        while (a > ldexp(448.0, s)) ++s;
        return s;
    }
    // amax = (1 + m 2^-23) 2^E and 448 2^(E-8) = 1.75 2^E: the answer is E-8
    // when the mantissa is at most 1.75, else E-7
    const int E = ef - 127;
    const uint32_t m = b & 0x7FFFFFu;
    return m <= 0x600000u ? E - 8 : E - 7;
}

__device__ __forceinline__ RowQuant row_quant(float amax) {
    RowQuant q;
    q.e = fp8_row_exp(amax);
    q.wide = (q.e < -127 || q.e > 126);
    q.mult = q.wide ? 0.0f : __uint_as_float(static_cast<uint32_t>(127 - q.e) << 23);
    q.scale = (q.e >= -126 && q.e <= 127) ? __uint_as_float(static_cast<uint32_t>(q.e + 127) << 23)
                                          : static_cast<float>(ldexp(1.0, q.e));
    return q;
}

// x 2^-e for a row whose 2^-e lies outside the fp32 normal range (rows with
// max |x| below about 2^-119 or above 2^134): exact in double.  Kept out of
// line so the per-element fast path stays fp32.
static __device__ __noinline__ float scaled_wide(float x, int e) {
    return static_cast<float>(static_cast<double>(x) * ldexp(1.0, -e));
}

// E4M3 codes of (lo, hi), nearest with ties to even and saturation to +-448;
// lo lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Largest magnitude of the 8 bf16 values in v.
__device__ __forceinline__ float absmax_bf16x8(const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    return m;
}

// 8 bf16 values -> 8 E4M3 codes (element 0 in the lowest byte), scaled by
// the row's multiplier 2^-e (fp32, exact for a power of two).
__device__ __forceinline__ uint2 quant_bf16x8(const uint4& v, float mult) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = cvt_e4m3x2(bf16lo(w[i]) * mult, bf16hi(w[i]) * mult);
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}
static __device__ __noinline__ uint2 quant_bf16x8_wide(const uint4& v, int e) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = cvt_e4m3x2(scaled_wide(bf16lo(w[i]), e), scaled_wide(bf16hi(w[i]), e));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}
__device__ __forceinline__ uint2 quant_bf16x8(const uint4& v, const RowQuant& q) {
    return q.wide ? quant_bf16x8_wide(v, q.e) : quant_bf16x8(v, q.mult);
}

// Where the 8 bf16 source elements [8v, 8v+8) of packed row n of group g live.
// mode 0: gate/up interleave of w1 (up), w2 (gate) [G, c, d] (N = 2c, K = d);
// mode 1: plain [G, N, K];  mode 2: shared down projections w3s [ns, d, cs]
// side by side (N = d, K = ns cs, element (i, s cs + j) = w3s[s][i][j]).
struct PackSrc {
    const uint4* a;
    const uint4* b;
    int mode, N, K, c, cs;
    __device__ __forceinline__ const uint4* chunk(long long g, int n, int v) const {
        if (mode == 0) {
            const int blk = n >> 7, within = n & 127;
            const bool gate = within < 64;
            const long long row = g * c + blk * 64 + (gate ? within : within - 64);
            return (gate ? b : a) + (row * K) / 8 + v;
        }
        if (mode == 1) return a + ((g * N + n) * static_cast<long long>(K)) / 8 + v;
        const int jj = 8 * v, s = jj / cs, j = jj - s * cs;
        return a + ((static_cast<long long>(s) * N + n) * cs + j) / 8;
    }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace fs
