// mx.cu -- quantisation kernels of the block-scaled FP8 (MX) expert path:
// bf16 rows to an MX matrix (the shared experts' token rows), the quantising
// Dispatch copy (each token row quantised once, its codes and block scales
// written to all of its k permuted rows), and the one-time packing of bf16
// expert weights into MX codes and scale chunks (layouts in mx.cuh).
//
// In every kernel a warp walks a row 8 elements (one 16-byte vector) per lane
// and step, so the 4 lanes 4q .. 4q+3 of a step hold one 32-element block:
// its largest magnitude is a 4-lane shuffle maximum, and lane 4q writes the
// block's scale byte.  The steps are counted for the whole warp (a row of
// 16-byte vectors that is not a multiple of 32 leaves lanes idle in its last
// step, they still take part in the shuffles).
#include "kernels.h"
#include "mx.cuh"

namespace fs {

// 8 bf16 values -> 8 E4M3 codes with the block's multiplier.
__device__ __forceinline__ uint2 mx_codes(const uint4& v, const MxQuant& m) {
    return quant_bf16x8(v, m.q);
}

// One warp per row r < rows128 (grid-stride): x [rows, cols] bf16 -> q, an MX
// matrix; rows past `rows` get zero codes and unit scales.
__global__ void __launch_bounds__(256)
quant_rows_mx_kernel(const uint4* __restrict__ x, long long rows, int cols, uint8_t* __restrict__ q) {
    const int lane = threadIdx.x & 31;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int nv = cols / 8;
    uint8_t* sf = q + mx_sf_offset(rows, cols);
    const long long r128 = mx_rows128(rows);
    for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < r128; r += nwarps) {
        uint2* dst = reinterpret_cast<uint2*>(q + r * cols);
        for (int v0 = 0; v0 < nv; v0 += 32) {
            const int v = v0 + lane;
            const bool act = v < nv;
            if (r < rows) {
                const uint4 a = act ? __ldg(x + r * nv + v) : make_uint4(0, 0, 0, 0);
                const MxQuant m = mx_quant(group4_max(absmax_bf16x8(a)));
                if (act) {
                    dst[v] = mx_codes(a, m);
                    if ((lane & 3) == 0) sf[mx_sf_byte(r, v / 4, cols)] = m.ue8m0;
                }
            } else if (act) {
                dst[v] = make_uint2(0, 0);
                if ((lane & 3) == 0) sf[mx_sf_byte(r, v / 4, cols)] = 127;
            }
        }
    }
}

// One warp per token: u[t] quantised in 32-element blocks once; its codes and
// scale bytes go to every slot's row pos[t, s] of x_q (an MX matrix of
// rows_cap rows) and, when u_q is set, to row t of u_q (an MX matrix [T, d]).
__global__ void __launch_bounds__(256)
dispatch_copy_mx_kernel(const uint4* __restrict__ u, int T, int d, int k, const int32_t* __restrict__ pos,
                        uint8_t* __restrict__ x_q, long long rows_cap, uint8_t* __restrict__ u_q) {
    const int lane = threadIdx.x & 31;
    const int t = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    if (t >= T) return;
    const int nv = d / 8;
    const int my_p = lane < k ? pos[static_cast<long long>(t) * k + lane] : -1;
    uint8_t* xsf = x_q + mx_sf_offset(rows_cap, d);
    uint8_t* usf = u_q ? u_q + mx_sf_offset(T, d) : nullptr;
    const uint4* src = u + static_cast<long long>(t) * nv;
    for (int v0 = 0; v0 < nv; v0 += 32) {
        const int v = v0 + lane;
        const bool act = v < nv;
        const uint4 a = act ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        const MxQuant m = mx_quant(group4_max(absmax_bf16x8(a)));
        const uint2 c = mx_codes(a, m);
        const bool lead = (lane & 3) == 0;
        for (int s = 0; s < k; ++s) {
            const int p = __shfl_sync(0xffffffffu, my_p, s);
            if (p < 0 || !act) continue;
            reinterpret_cast<uint2*>(x_q + static_cast<long long>(p) * d)[v] = c;
            if (lead) xsf[mx_sf_byte(p, v / 4, d)] = m.ue8m0;
        }
        if (u_q && act) {
            reinterpret_cast<uint2*>(u_q + static_cast<long long>(t) * d)[v] = c;
            if (lead) usf[mx_sf_byte(t, v / 4, d)] = m.ue8m0;
        }
    }
}

// One warp per packed row (grid-stride over G * NB * 256 rows): codes into the
// tiled layout, scale bytes into the tile's chunks; rows past N: zero codes,
// unit scales.
__global__ void __launch_bounds__(256)
pack_mx_kernel(PackSrc src, int G, int NB, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
    const int lane = threadIdx.x & 31;
    const int K = src.K, N = src.N, KB = K / 128, nv = K / 8;
    const long long total = static_cast<long long>(G) * NB * 256;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long R = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; R < total; R += nwarps) {
        const long long g = R / (static_cast<long long>(NB) * 256);
        const int nr = static_cast<int>(R - g * NB * 256);
        const int nb = nr >> 8, rr = nr & 255;
        uint8_t* blk0 = codes + ((g * NB + nb) * KB) * 32768LL + rr * 128;
        for (int v0 = 0; v0 < nv; v0 += 32) {
            const int v = v0 + lane;
            const bool act = v < nv;
            const int kk = 8 * v;
            uint2 c = make_uint2(0, 0);
            uint8_t byte = 127;
            if (nr < N) {
                const uint4 a = act ? __ldg(src.chunk(g, nr, v)) : make_uint4(0, 0, 0, 0);
                const MxQuant m = mx_quant(group4_max(absmax_bf16x8(a)));
                c = mx_codes(a, m);
                byte = m.ue8m0;
            }
            if (act) {
                *reinterpret_cast<uint2*>(blk0 + (kk >> 7) * 32768LL + (kk & 127)) = c;
                if ((lane & 3) == 0) sf[mx_w_sf_byte(g, NB, nb, rr, v / 4, K)] = byte;
            }
        }
    }
}

static int mx_grid(long long warps_needed) {
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = 152LL * 16;
    if (blocks > cap) blocks = cap;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

size_t packed_bytes_mx(int G, int N, int K) { return mx_w_bytes(G, N, K); }

const uint8_t* packed_sf_mx(const void* packed, int G, int N, int K) {
    return static_cast<const uint8_t*>(packed) + mx_w_codes_bytes(G, N, K);
}

static cudaError_t launch_pack_mx(const PackSrc& src, int G, void* out, cudaStream_t st) {
    const int NB = (src.N + 255) / 256;
    uint8_t* codes = static_cast<uint8_t*>(out);
    uint8_t* sf = codes + mx_w_codes_bytes(G, src.N, src.K);
    pack_mx_kernel<<<mx_grid(static_cast<long long>(G) * NB * 256), 256, 0, st>>>(src, G, NB, codes, sf);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_pack_w13_mx(int G, int c, int d, const void* w1, const void* w2, void* w13, cudaStream_t st) {
    PackSrc s{static_cast<const uint4*>(w1), static_cast<const uint4*>(w2), 0, 2 * c, d, c, 0};
    return launch_pack_mx(s, G, w13, st);
}

cudaError_t launch_pack_w3_mx(int G, int d, int c, const void* w3, void* w3p, cudaStream_t st) {
    PackSrc s{static_cast<const uint4*>(w3), nullptr, 1, d, c, 0, 0};
    return launch_pack_mx(s, G, w3p, st);
}

cudaError_t launch_pack_w3_shared_mx(int ns, int cs, int d, const void* w3s, void* w3cat, cudaStream_t st) {
    PackSrc s{static_cast<const uint4*>(w3s), nullptr, 2, d, ns * cs, 0, cs};
    return launch_pack_mx(s, 1, w3cat, st);
}

cudaError_t launch_quant_rows_mx(const void* x, long long rows, int cols, void* q, cudaStream_t st) {
    quant_rows_mx_kernel<<<mx_grid(mx_rows128(rows)), 256, 0, st>>>(static_cast<const uint4*>(x), rows, cols,
                                                                    static_cast<uint8_t*>(q));
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_dispatch_copy_mx(const void* u, int T, int d, int k, const int32_t* pos, void* x_q,
                                    long long rows_cap, void* u_q, cudaStream_t st) {
    const long long warps = T;
    dispatch_copy_mx_kernel<<<static_cast<int>((warps + 7) / 8), 256, 0, st>>>(
        static_cast<const uint4*>(u), T, d, k, pos, static_cast<uint8_t*>(x_q), rows_cap, static_cast<uint8_t*>(u_q));
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
