// gemm_tc.cu -- persistent grouped GEMM on the 5th-generation tensor cores
// (tcgen05.mma kind::f16 with bf16 operands, or kind::f8f6f4 with FP8 E4M3
// operands; fp32 accumulators in TMEM), operands staged in shared memory by TMA
// with the 128-byte swizzle.  A stage is 128 bytes of K per row either way (64
// bf16 or 128 E4M3 elements); FP8 rows carry power-of-two scales (one per A row,
// one per B row) that the epilogue applies to the fp32 accumulator.
//
// One GEMM shape serves every dense contraction of the MoE layer
// ("FarSkip-Collective: Unhobbling Blocking Communication in Mixture of Experts
// Models", §2.1 MLP and MoE equations):
//   EPI_SWIGLU : H = SiLU(X W2^T) * (X W1^T) from the packed [2c, d] gate/up weight
//   EPI_BF16   : Y = H W3^T                       (down projection, bf16 out)
//   EPI_F32    : Z = U W_R^T                      (router logits, fp32 out)
// Rows are grouped (one group per expert; offsets live on the device and the
// host never reads them).  Each group's rows [row_start[g], row_start[g+1]) are
// multiplied by the group's own B = W[g] ([N, K], K-major).
//
// CTA = 10 warps, one CTA per SM, persistent over a static tile order:
//   warp 0      TMA producer (one lane): A tile 128 x 64 and B tile 256 x 64 per stage
//   warp 1      TMEM owner + MMA issuer (one lane): 4 x (128 x 256 x 16) MMAs per stage
//   warps 2..9  epilogue: two warps per TMEM lane quarter, each taking half of the
//               tile's columns: tcgen05.ld of the accumulator, activation, stores
// TMEM holds two 128 x 256 fp32 accumulators (512 columns) so the epilogue of
// tile i overlaps the MMAs of tile i + 1.  Every wait is bounded in time.
// Tile order inside a group: blocks of M-tiles (the whole group up to 32
// M-tiles, else 16), N-tiles outer inside a block, so the ~152 tiles in flight
// share a few MB of A and B in L2 and each B slab is read from HBM once,
// instead of streaming a tall A operand once per N-tile.
#include <cudaTypedefs.h>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace fs {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;                 // 64 bf16 = 128 B = one swizzle row
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;   // 16 KB
constexpr int B_STAGE = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int NACC = 2;
constexpr int TMEM_COLS = NACC * BN;   // 512
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;   // 320
constexpr int kGroupM = 16;                    // M-tiles per rasterisation block
constexpr int BAR_BYTES = 256;
// bf16 outputs leave through one 2 KB staging piece per epilogue warp (32 rows x
// 32 columns, 64-byte swizzle) and TMA stores, after the barriers and the plan
constexpr int PIECE_OFF = (STAGES * STAGE_BYTES + BAR_BYTES + 2 * (kMaxGroups + 1) * 4 + 1023) / 1024 * 1024;
constexpr int PIECE_BYTES = 2048;
constexpr size_t SMEM_BYTES = 1024 + PIECE_OFF + EPI_WARPS * PIECE_BYTES;

struct Args {
    const int* plan;   // [2 (G + 1)]: m-tile prefix (BM rows), then row_start
    int G;
    int N;             // B rows per group
    int K;
    int n_tiles;       // ceil(N / BN)
    int max_mtiles;    // upper bound of the m-tile count (capacity check)
    void* out;
    long long ldo;     // output row stride in elements
    int out_cols;      // valid output columns (EPI_F32 / EPI_BF16), c for EPI_SWIGLU
    int* err;          // device error word
    const int* gather_rows;  // A row of GEMM row p = gather_rows[p] (tile::gather4), or nullptr
    int gather_limit;        // entries of gather_rows
    int b_blocked;           // B in the tiled weight layout [G][n_tiles][K/BK][256][128 bytes] (3D map)
    const float* a_scale;    // FP8: scale of A row p (a_scale[p])
    const float* b_scale;    // FP8: scale of B row n of group g (b_scale[g N + n])
    void* aux;               // TcExtra::aux (stored pre-activations out / in)
    long long aux_ld;
    int accumulate;          // EPI_F32: out += acc
    int tma_out;             // bf16 out (EPI_SWIGLU h, EPI_BF16) through the output tensor map
    int ksplit = 1;          // EPI_F32: K split into ksplit ranges, each written as its own partial
    long long split_rows = 0;   // rows between the partials of successive K ranges in out
    CombineEpi cmb;          // EPI_COMBINE: Combine operands and outputs
};

struct Tile {
    int g, m, n, a_row, rows_valid, b_row;
};

__device__ __forceinline__ Tile decode_tile(int t, const int* mt_start, const int* row_start, int G,
                                            int n_tiles, int BNrows, int N, int bm = BM) {
    const int q = t / n_tiles;
    int lo = 0, hi = G;            // last g with mt_start[g] <= q
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (mt_start[mid] <= q) lo = mid; else hi = mid;
    }
    Tile r;
    r.g = lo;
    const int mtiles = mt_start[lo + 1] - mt_start[lo];
    const int local = t - mt_start[lo] * n_tiles;
    // groups of up to 2 kGroupM M-tiles form one block, so every B slab of the
    // group is used by all its M-tiles back to back; taller groups use blocks
    // of kGroupM M-tiles
    const int GM = mtiles <= 2 * kGroupM ? mtiles : kGroupM;
    const int blk = local / (GM * n_tiles);                 // block of GM M-tiles
    const int gm = min(GM, mtiles - blk * GM);              // M-tiles in this block
    const int rr = local - blk * GM * n_tiles;
    r.n = rr / gm;
    r.m = blk * GM + (rr - r.n * gm);
    r.a_row = row_start[lo] + r.m * bm;
    const int rem = row_start[lo + 1] - r.a_row;
    r.rows_valid = rem < bm ? rem : bm;
    r.b_row = lo * N + r.n * BNrows;
    return r;
}

// FP8 dequantisation scales of one epilogue thread: its A row's scale, and
// the B scales of the 128 tile columns its warp covers (half `half` of the
// tile), spread over the lanes: lane l holds columns 4l .. 4l + 3 of the half.
// Loaded before the accumulator is ready, so the loads' latency overlaps the
// tile's MMAs instead of stalling each column block of the epilogue.
struct EpiScales {
    float sa = 1.0f;
    float4 sb = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
};

__device__ __forceinline__ EpiScales load_epi_scales(const float* a_scale, const float* b_scale, int N, int g, int n,
                                                     long long orow, bool row_ok, int half, int lane) {
    EpiScales s;
    if (row_ok) s.sa = __ldg(a_scale + orow);
    static_assert(tc::BN == 256, "the epilogue's B scales cover 2 x 128 columns per tile");
    const int col = n * tc::BN + half * (tc::BN / 2) + 4 * lane;
    if (col < N) s.sb = __ldg(reinterpret_cast<const float4*>(b_scale + static_cast<long long>(g) * N + col));
    return s;
}

// v[j] <- (v[j] * sa) * sb[rel + j] for NC (16 or 32) accumulator columns
// starting at column rel (a multiple of 16) of the warp's half; the B scales
// come from the lanes holding them.  Every lane of the warp must call it.
template <int NC>
__device__ __forceinline__ void scale_cols(uint32_t* v, const EpiScales& s, int rel) {
#pragma unroll
    for (int q4 = 0; q4 < NC / 4; ++q4) {
        const int src = (rel >> 2) + q4;
        const float f[4] = {__shfl_sync(0xffffffffu, s.sb.x, src), __shfl_sync(0xffffffffu, s.sb.y, src),
                            __shfl_sync(0xffffffffu, s.sb.z, src), __shfl_sync(0xffffffffu, s.sb.w, src)};
#pragma unroll
        for (int i = 0; i < 4; ++i) v[4 * q4 + i] = __float_as_uint((__uint_as_float(v[4 * q4 + i]) * s.sa) * f[i]);
    }
}

// 16 consecutive residual values (bf16 or fp32) at element offset off.
__device__ __forceinline__ void load16_resid(const void* base, long long off, bool bf16, float (&v)[16]) {
    if (bf16) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            v[2 * q] = bf16lo(w[q]);
            v[2 * q + 1] = bf16hi(w[q]);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 a = __ldg(p + q);
            v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
        }
    }
}

__device__ __forceinline__ void store16_resid(void* base, long long off, bool bf16, const float (&v)[16]) {
    if (bf16) {
        uint4* p = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
        p[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                          pack_bf16x2(v[6], v[7]));
        p[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                          pack_bf16x2(v[14], v[15]));
    } else {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) p[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
}

// EPI_COMBINE for the thread owning token row `orow`, columns [c_lo, c_hi) of
// n-tile n: the accumulator is the shared output S; Combine and the FarSkip
// update follow combine_kernel's arithmetic (see CombineEpi).  Per 16 columns
// the k routed rows' 32-byte pieces are loaded together (k loads in flight).
template <bool F8>
__device__ __forceinline__ void epilogue_combine(uint32_t tbase, bool row_ok, long long orow, int n, int c_lo, int c_hi,
                                                 int half, const EpiScales& sc, const Args& args) {
    const CombineEpi& cb = args.cmb;
    const long long d = args.ldo;
    int ps[kCombineEpiMaxK];
    float wsl[kCombineEpiMaxK];
#pragma unroll
    for (int s = 0; s < kCombineEpiMaxK; ++s) {
        ps[s] = -1;
        wsl[s] = 0.f;
        if (row_ok && s < cb.k) {
            ps[s] = __ldg(cb.pos + orow * cb.k + s);
            wsl[s] = __ldg(cb.topk_w + orow * cb.k + s);
        }
    }
#pragma unroll 1
    for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + c0, v);
        tmem_ld_wait();
        if constexpr (F8) scale_cols<16>(v, sc, c0 - half * (BN / 2));
        if (!row_ok) continue;
        const long long col = static_cast<long long>(n) * BN + c0;
        uint4 yr[kCombineEpiMaxK][2];
#pragma unroll
        for (int s = 0; s < kCombineEpiMaxK; ++s) {
            if (ps[s] >= 0) {
                const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(cb.y_perm) +
                                                                  static_cast<long long>(ps[s]) * d + col);
                yr[s][0] = __ldg(src);
                yr[s][1] = __ldg(src + 1);
            }
        }
        float prev[16], base[16], acc[16], full[16];
        load16_resid(cb.o_prev, orow * d + col, cb.prev_bf16 != 0, prev);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            base[j] = prev[j] + __uint_as_float(v[j]);
            acc[j] = 0.f;
        }
#pragma unroll
        for (int s = 0; s < kCombineEpiMaxK; ++s) {
            if (ps[s] >= 0) {
                const uint32_t q[8] = {yr[s][0].x, yr[s][0].y, yr[s][0].z, yr[s][0].w,
                                       yr[s][1].x, yr[s][1].y, yr[s][1].z, yr[s][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[2 * i] = fmaf(wsl[s], bf16lo(q[i]), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(wsl[s], bf16hi(q[i]), acc[2 * i + 1]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) full[j] = base[j] + acc[j];
        if (cb.o_partial) store16_resid(cb.o_partial, orow * d + col, cb.out_bf16 != 0, base);
        store16_resid(cb.o_full, orow * d + col, cb.out_bf16 != 0, full);
        if (cb.u_next) store16_resid(cb.u_next, orow * d + col, true, cb.u_src == 0 ? base : (cb.u_src == 1 ? prev : full));
    }
}

// Epilogue of one accumulator tile for the thread owning TMEM lane `r` of its
// CTA (row a_row + r of the output), columns of half `half` of the tile.
// With F8 the accumulator is scaled by the A row's and the B rows' scales:
// (acc * a_scale[row]) * b_scale[g N + col].
// One 32-row x 64-byte piece (pk: this lane's row, 16 words: 32 bf16 or 16
// fp32) to global through the warp's staging buffer and a TMA store at (x, y),
// or, with reduce, a TMA add into the fp32 values already there.
__device__ __forceinline__ void store_piece_bf16(const CUtensorMap* tmo, uint8_t* piece, const uint32_t* pk, int lane,
                                                 int x, int y, bool reduce = false) {
    if (lane == 0) bulk_wait_read0();          // the previous piece has left the buffer
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int sw = q ^ ((lane >> 1) & 3);  // 64-byte swizzle of the 16-byte chunks
        *reinterpret_cast<uint4*>(piece + lane * 64 + sw * 16) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (reduce)
            tma_reduce_add_2d(tmo, smem_u32(piece), x, y);
        else
            tma_store_2d(tmo, smem_u32(piece), x, y);
        bulk_commit();
    }
}

template <int EPI, bool F8 = false>
__device__ __forceinline__ void epilogue_tile(uint32_t tbase, int g, int a_row, int rows_valid, int n, int r, int half,
                                              const Args& args, const EpiScales& sc, const CUtensorMap* tmo = nullptr,
                                              uint8_t* piece = nullptr) {
    const Tile tl{g, 0, n, a_row, rows_valid, 0};
    const bool row_ok = r < tl.rows_valid;
    // TMA stores for whole 32-row pieces inside the group; a piece that crosses
    // the group's last row keeps the masked per-thread stores, so the next
    // group's rows are never written here
    const int lane = r & 31, q32 = r & ~31;
    const bool piece_ok = tmo != nullptr && q32 + 32 <= tl.rows_valid;
    const long long orow = static_cast<long long>(tl.a_row + r);
    if constexpr (EPI == EPI_SWIGLU) {
        // packed tile columns: [gate 64 | up 64] x 2 -> 128 expert columns
        const int rem = args.N - tl.n * BN;
        const int npk = (rem >= BN ? BN : rem) / 128;
        __nv_bfloat16* H = reinterpret_cast<__nv_bfloat16*>(args.out);
        for (int g2 = half; g2 < npk; g2 += 2) {
#pragma unroll 1
            for (int j0 = 0; j0 < 64; j0 += 32) {
                uint32_t gv[32], uv[32];
                tmem_ld32(tbase + g2 * 128 + j0, gv);
                tmem_ld32(tbase + g2 * 128 + 64 + j0, uv);
                tmem_ld_wait();
                if constexpr (F8) {          // g2 == half: gate columns j0.., up columns 64 + j0.. of the half
                    scale_cols<32>(gv, sc, j0);
                    scale_cols<32>(uv, sc, 64 + j0);
                }
                if (row_ok) {
                    if (args.aux) {   // training forward: keep g, a (bf16) for the backward
                        uint32_t pg[16], pu[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            pg[q] = pack_bf16x2(__uint_as_float(gv[2 * q]), __uint_as_float(gv[2 * q + 1]));
                            pu[q] = pack_bf16x2(__uint_as_float(uv[2 * q]), __uint_as_float(uv[2 * q + 1]));
                        }
                        __nv_bfloat16* gu = static_cast<__nv_bfloat16*>(args.aux) + orow * args.aux_ld + tl.n * BN +
                                            g2 * 128 + j0;
                        uint4* gd = reinterpret_cast<uint4*>(gu);
                        uint4* ud = reinterpret_cast<uint4*>(gu + 64);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            gd[v] = make_uint4(pg[4 * v], pg[4 * v + 1], pg[4 * v + 2], pg[4 * v + 3]);
                            ud[v] = make_uint4(pu[4 * v], pu[4 * v + 1], pu[4 * v + 2], pu[4 * v + 3]);
                        }
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float h0 = silu_f(__uint_as_float(gv[2 * q])) * __uint_as_float(uv[2 * q]);
                        const float h1 = silu_f(__uint_as_float(gv[2 * q + 1])) * __uint_as_float(uv[2 * q + 1]);
                        pk[q] = pack_bf16x2(h0, h1);
                    }
                    if (piece_ok) {
                        store_piece_bf16(tmo, piece, pk, lane, tl.n * 128 + g2 * 64 + j0, tl.a_row + q32);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(H + orow * args.ldo + tl.n * 128 + g2 * 64 + j0);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
            }
        }
    } else if constexpr (EPI == EPI_BF16) {
        const int rem = args.out_cols - tl.n * BN;
        const int ncols = rem >= BN ? BN : rem;
        __nv_bfloat16* Y = reinterpret_cast<__nv_bfloat16*>(args.out);
        const int cend = min(ncols, (half + 1) * (BN / 2));
#pragma unroll 1
        for (int c0 = half * (BN / 2); c0 < cend; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + c0, v);
            tmem_ld_wait();
            if constexpr (F8) scale_cols<32>(v, sc, c0 - half * (BN / 2));
            if (row_ok) {
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    pk[q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                if (piece_ok) {
                    store_piece_bf16(tmo, piece, pk, lane, tl.n * BN + c0, tl.a_row + q32);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(Y + orow * args.ldo + tl.n * BN + c0);
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                }
            }
        }
    } else if constexpr (EPI == EPI_COMBINE) {
        const int rem = args.out_cols - tl.n * BN;
        const int ncols = rem >= BN ? BN : rem;
        epilogue_combine<F8>(tbase, row_ok, orow, tl.n, half * (BN / 2), min(ncols, (half + 1) * (BN / 2)), half,
                             sc, args);
    } else if constexpr (EPI == EPI_DSWIGLU) {
        // accumulator = dh of hidden columns j = 256 n + c; g_j, a_j sit at packed
        // columns 128 (j / 64) + j % 64 and that + 64 of the aux row, and dg, da
        // go to the same packed columns of out
        const int rem = args.out_cols - tl.n * BN;
        const int ncols = rem >= BN ? BN : rem;
        const __nv_bfloat16* GU = static_cast<const __nv_bfloat16*>(args.aux);
        __nv_bfloat16* D = static_cast<__nv_bfloat16*>(args.out);
        const int cend = min(ncols, (half + 1) * (BN / 2));
#pragma unroll 1
        for (int c0 = half * (BN / 2); c0 < cend; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + c0, v);
            tmem_ld_wait();
            if (row_ok) {
                const int j0 = tl.n * BN + c0;
                const long long pc = 128LL * (j0 >> 6) + (j0 & 63);
                const uint4* gs = reinterpret_cast<const uint4*>(GU + orow * args.aux_ld + pc);
                const uint4* as = reinterpret_cast<const uint4*>(GU + orow * args.aux_ld + pc + 64);
                uint32_t gw[16], aw[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 x = __ldg(gs + q), y = __ldg(as + q);
                    gw[4 * q] = x.x; gw[4 * q + 1] = x.y; gw[4 * q + 2] = x.z; gw[4 * q + 3] = x.w;
                    aw[4 * q] = y.x; aw[4 * q + 1] = y.y; aw[4 * q + 2] = y.z; aw[4 * q + 3] = y.w;
                }
                uint32_t pg[16], pa[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float g0 = bf16lo(gw[q]), g1 = bf16hi(gw[q]);
                    const float a0 = bf16lo(aw[q]), a1 = bf16hi(aw[q]);
                    const float s0 = 1.0f / (1.0f + __expf(-g0)), s1 = 1.0f / (1.0f + __expf(-g1));
                    const float dh0 = __uint_as_float(v[2 * q]), dh1 = __uint_as_float(v[2 * q + 1]);
                    pg[q] = pack_bf16x2(dh0 * a0 * (s0 * (1.0f + g0 * (1.0f - s0))),
                                        dh1 * a1 * (s1 * (1.0f + g1 * (1.0f - s1))));
                    pa[q] = pack_bf16x2(dh0 * (g0 * s0), dh1 * (g1 * s1));
                }
                if (piece_ok) {     // dg and da as two 32 x 32 pieces through TMA stores
                    store_piece_bf16(tmo, piece, pg, lane, static_cast<int>(pc), tl.a_row + q32);
                    store_piece_bf16(tmo, piece, pa, lane, static_cast<int>(pc) + 64, tl.a_row + q32);
                } else {
                    uint4* gd = reinterpret_cast<uint4*>(D + orow * args.ldo + pc);
                    uint4* ad = reinterpret_cast<uint4*>(D + orow * args.ldo + pc + 64);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        gd[w] = make_uint4(pg[4 * w], pg[4 * w + 1], pg[4 * w + 2], pg[4 * w + 3]);
                        ad[w] = make_uint4(pa[4 * w], pa[4 * w + 1], pa[4 * w + 2], pa[4 * w + 3]);
                    }
                }
            }
        }
    } else {  // EPI_F32
        const int rem = args.out_cols - tl.n * BN;
        const int ncols = rem >= BN ? BN : rem;
        float* Z = reinterpret_cast<float*>(args.out);
        const bool vec = (args.ldo & 3) == 0;
        const int cend = min(ncols, (half + 1) * (BN / 2));
#pragma unroll 1
        for (int c0 = half * (BN / 2); c0 < cend; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + c0, v);
            tmem_ld_wait();
            if constexpr (F8) scale_cols<32>(v, sc, c0 - half * (BN / 2));
            if (piece_ok && ncols - c0 >= 32) {       // two 32 x 16 fp32 pieces through TMA stores (adds)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[j] = v[16 * h + j];
                    store_piece_bf16(tmo, piece, pk, lane, tl.n * BN + c0 + 16 * h, tl.a_row + q32, args.accumulate != 0);
                }
            } else if (row_ok) {
                float* dst = Z + orow * args.ldo + tl.n * BN + c0;
                const int nv = ncols - c0 >= 32 ? 32 : ncols - c0;
                if (args.accumulate) {
                    if (vec && nv == 32) {
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            const float4 o = reinterpret_cast<const float4*>(dst)[w];
                            v[4 * w] = __float_as_uint(__uint_as_float(v[4 * w]) + o.x);
                            v[4 * w + 1] = __float_as_uint(__uint_as_float(v[4 * w + 1]) + o.y);
                            v[4 * w + 2] = __float_as_uint(__uint_as_float(v[4 * w + 2]) + o.z);
                            v[4 * w + 3] = __float_as_uint(__uint_as_float(v[4 * w + 3]) + o.w);
                        }
                    } else {
                        for (int j = 0; j < nv; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + dst[j]);
                    }
                }
                if (vec && nv == 32) {
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        reinterpret_cast<uint4*>(dst)[w] = make_uint4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
                } else {
                    for (int j = 0; j < nv; ++j) dst[j] = __uint_as_float(v[j]);
                }
            }
        }
    }
}

template <int EPI, bool F8 = false>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO, const Args args) {
    constexpr int BKE = F8 ? 128 : BK;     // K elements per stage (128 bytes per row)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* full = bars;                 // [STAGES]
    uint64_t* empty = bars + STAGES;       // [STAGES]
    uint64_t* tfull = bars + 2 * STAGES;   // [NACC]
    uint64_t* tempty = tfull + NACC;       // [NACC]
    uint64_t* fin = tempty + NACC;         // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* mt_start = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + BAR_BYTES);
    int* row_start = mt_start + (args.G + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;

    for (int i = threadIdx.x; i < 2 * (G + 1); i += THREADS) mt_start[i] = args.plan[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), EPI_WARPS);
        }
        mbar_init(smem_u32(fin), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int total_mtiles = mt_start[G];
    if (total_mtiles < 0 || total_mtiles > args.max_mtiles) {
        if (threadIdx.x == 0) set_dev_error(args.err, DEV_ERR_OFFSETS);
        total_mtiles = 0;
    }
    const int ksplit = args.ksplit;         // tile t: output tile t / ksplit, K range t % ksplit
    const int total = total_mtiles * args.n_tiles * ksplit;
    const int num_kb = args.K / BKE;

    if (!F8 && warp == 0 && args.gather_rows != nullptr) {
        // ----------------------------------------------- producer, gathered A
        // The whole warp: lane l fetches rows 4l .. 4l+3 of each A tile with one
        // tile::gather4 per k-block (rows of the token matrix named by
        // gather_rows, i.e. the Dispatch permutation), lane 0 arms the stage and
        // loads B.
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
        }
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile tl = decode_tile(t, mt_start, row_start, G, args.n_tiles, BN, args.N);
            int rr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int p = tl.a_row + 4 * lane + j;
                rr[j] = p < args.gather_limit ? __ldg(args.gather_rows + p) : 0;
            }
            for (int kb = 0; kb < num_kb; ++kb) {
                const bool got = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                const uint32_t fb = smem_u32(&full[stage]);
                if (lane == 0) mbar_arrive_expect_tx(fb, STAGE_BYTES);
                uint8_t* sa = smem + stage * STAGE_BYTES;
                tma_gather4(smem_u32(sa) + 512u * lane, &tmA, fb, kb * BK, rr[0], rr[1], rr[2], rr[3]);
                if (lane == 0) {
                    if (args.b_blocked)
                        tma_load_3d(smem_u32(sa + A_STAGE), &tmB, fb, 0, 0, (tl.g * args.n_tiles + tl.n) * num_kb + kb);
                    else
                        tma_load_2d(smem_u32(sa + A_STAGE), &tmB, fb, kb * BK, tl.b_row);
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (lane == 0) {   // drain: the last loads must land before the CTA exits
            const int pending = issued < STAGES ? issued : STAGES;
            for (int j = 1; j <= pending; ++j) {
                int s = stage - j;
                uint32_t ph = phase;
                if (s < 0) { s += STAGES; ph ^= 1u; }
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(smem_u32(&full[s]), ph)) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int tt = t / ksplit, ks = t - tt * ksplit;
                const Tile tl = decode_tile(tt, mt_start, row_start, G, args.n_tiles, BN, args.N);
                const int kb1 = ((ks + 1) * num_kb) / ksplit;
                for (int kb = (ks * num_kb) / ksplit; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    tma_load_2d(smem_u32(sa), &tmA, fb, kb * BKE, tl.a_row);
                    if (args.b_blocked)
                        tma_load_3d(smem_u32(sa + A_STAGE), &tmB, fb, 0, 0, (tl.g * args.n_tiles + tl.n) * num_kb + kb);
                    else
                        tma_load_2d(smem_u32(sa + A_STAGE), &tmB, fb, kb * BKE, tl.b_row);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Drain: the last loads (at most STAGES) must land before the CTA exits.
            const int pending = issued < STAGES ? issued : STAGES;
            for (int j = 1; j <= pending; ++j) {
                int s = stage - j;
                uint32_t ph = phase;
                if (s < 0) { s += STAGES; ph ^= 1u; }
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(smem_u32(&full[s]), ph)) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(smem_u32(&tempty[acc]), (use & 1u) ^ 1u, abort_flag, args.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const int ks = t % ksplit;
                const int kb0 = (ks * num_kb) / ksplit, kb1 = ((ks + 1) * num_kb) / ksplit;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err)) { ok = false; break; }
                    tc_fence_after();
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    const uint64_t adesc = smem_desc_sw128(smem_u32(sa));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(sa + A_STAGE));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // one MMA takes 32 bytes of K (16 bf16 or 32 E4M3): +32 bytes inside the
                        // 128-byte swizzle row = +2 in the >>4 address field
                        if constexpr (F8)
                            tc_mma_f8(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        else
                            tc_mma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc,
                                        (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&tfull[acc]));
            }
            // every MMA issued by this thread completes before TMEM is released
            tc_commit(smem_u32(fin));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(fin), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;          // TMEM lanes [32 quarter, 32 quarter + 32)
        const int half = (warp - 2) >> 2;      // which half of the tile's columns
        const int r = quarter * 32 + lane;     // row of the tile owned by this thread
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int tt = t / ksplit, ks = t - tt * ksplit;
            const Tile tl = decode_tile(tt, mt_start, row_start, G, args.n_tiles, BN, args.N);
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            EpiScales sc;
            if constexpr (F8)
                sc = load_epi_scales(args.a_scale, args.b_scale, args.N, tl.g, tl.n, static_cast<long long>(tl.a_row) + r,
                                     r < tl.rows_valid, half, lane);
            if (!mbar_wait(smem_u32(&tfull[acc]), use & 1u, abort_flag, args.err)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            // K range ks of a split GEMM goes to its own partial, split_rows rows further on
            epilogue_tile<EPI, F8>(tbase, tl.g, tl.a_row + static_cast<int>(ks * args.split_rows), tl.rows_valid, tl.n, r,
                                   half, args, sc,
                                   args.tma_out ? &tmO : nullptr, smem + PIECE_OFF + (warp - 2) * PIECE_BYTES);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        }
        if (args.tma_out && lane == 0) bulk_wait0();     // this warp's TMA stores have completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------- CTA pairs
// The same GEMM on 256 x 256 tiles computed by a pair of CTAs on the two SMs of
// a TPC with the 2-SM MMA (tcgen05.mma.cta_group::2): each CTA stages its own
// 128 rows of A and its half (128 rows) of B per k-block (32 KB, 6 stages), the
// even CTA issues the MMAs, and each CTA's TMEM holds its 128 rows x 256
// columns of the accumulator (two buffers).  Per SM this halves the operand
// bytes per FLOP against the single-CTA 128 x 256 tile.
//   full[s]   (even CTA)  both CTAs' TMA loads complete on it (64 KB expected)
//   empty[s]  (each CTA)  2-SM commit multicast to both CTAs frees stage s
//   tfull[a]  (each CTA)  2-SM commit multicast: accumulator a is ready
//   tempty[a] (even CTA)  16 epilogue warps of the pair release accumulator a
constexpr int P_STAGES = 6;
constexpr int P_A_STAGE = 128 * BK * 2;       // 16 KB: this CTA's 128 rows of A
constexpr int P_B_STAGE = 128 * BK * 2;       // 16 KB: this CTA's half of B
constexpr int P_STAGE_BYTES = P_A_STAGE + P_B_STAGE;
constexpr int P_BM = 256;                     // rows per pair tile
constexpr size_t P_SMEM_BYTES =
    1024 + static_cast<size_t>(P_STAGES) * P_STAGE_BYTES + BAR_BYTES + 2 * (kMaxGroups + 1) * sizeof(int);

template <int EPI, bool F8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const Args args) {
    constexpr int BKE = F8 ? 128 : BK;     // K elements per stage (128 bytes per row)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES);
    uint64_t* full = bars;                   // [P_STAGES]
    uint64_t* empty = bars + P_STAGES;       // [P_STAGES]
    uint64_t* tfull = bars + 2 * P_STAGES;   // [NACC]
    uint64_t* tempty = tfull + NACC;         // [NACC]
    uint64_t* fin = tempty + NACC;           // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* mt_start = reinterpret_cast<int*>(smem + P_STAGES * P_STAGE_BYTES + BAR_BYTES);
    int* row_start = mt_start + (args.G + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    const uint32_t rank = cluster_ctarank();      // 0 = the CTA that issues the MMAs
    const bool leader = rank == 0;

    for (int i = threadIdx.x; i < 2 * (G + 1); i += THREADS) mt_start[i] = args.plan[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 2 * EPI_WARPS);
        }
        mbar_init(smem_u32(fin), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();          // the even CTA's barriers exist before the odd CTA signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int total_mtiles = mt_start[G];
    if (total_mtiles < 0 || total_mtiles > args.max_mtiles) {
        if (threadIdx.x == 0) set_dev_error(args.err, DEV_ERR_OFFSETS);
        total_mtiles = 0;
    }
    const int total = total_mtiles * args.n_tiles;
    const int num_kb = args.K / BKE;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = cid; t < total && ok; t += ncl) {
                const Tile tl = decode_tile(t, mt_start, row_start, G, args.n_tiles, BN, args.N, P_BM);
                const int a_row = tl.a_row + static_cast<int>(rank) * 128;
                const int b_row = tl.b_row + static_cast<int>(rank) * 128;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    const uint32_t fb_local = smem_u32(&full[stage]);
                    if (leader) mbar_arrive_expect_tx(fb_local, 2 * P_STAGE_BYTES);
                    const uint32_t fb = map_to_cta(fb_local, 0);
                    uint8_t* sa = smem + stage * P_STAGE_BYTES;
                    tma_load_2d_pair(smem_u32(sa), &tmA, fb, kb * BKE, a_row);
                    if (args.b_blocked)
                        tma_load_3d_pair(smem_u32(sa + P_A_STAGE), &tmB, fb, 0, static_cast<int>(rank) * 128,
                                         (tl.g * args.n_tiles + tl.n) * num_kb + kb);
                    else
                        tma_load_2d_pair(smem_u32(sa + P_A_STAGE), &tmB, fb, kb * BKE, b_row);
                    ++issued;
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (leader) {   // the loads of both CTAs complete on the even CTA's barriers
                const int pending = issued < P_STAGES ? issued : P_STAGES;
                for (int j = 1; j <= pending; ++j) {
                    int s = stage - j;
                    uint32_t ph = phase;
                    if (s < 0) { s += P_STAGES; ph ^= 1u; }
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(smem_u32(&full[s]), ph)) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            if (leader) {
                constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(P_BM, BN) : idesc_bf16_f32(P_BM, BN);
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                int it = 0;
                for (int t = cid; t < total && ok; t += ncl, ++it) {
                    const int acc = it & 1;
                    const uint32_t use = static_cast<uint32_t>(it >> 1);
                    if (!mbar_wait(smem_u32(&tempty[acc]), (use & 1u) ^ 1u, abort_flag, args.err)) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                    for (int kb = 0; kb < num_kb; ++kb) {
                        if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err)) { ok = false; break; }
                        tc_fence_after();
                        uint8_t* sa = smem + stage * P_STAGE_BYTES;
                        const uint64_t adesc = smem_desc_sw128(smem_u32(sa));
                        const uint64_t bdesc = smem_desc_sw128(smem_u32(sa + P_A_STAGE));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {   // 32 bytes of K per MMA
                            if constexpr (F8)
                                tc_mma_f8_pair(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc,
                                               (kb > 0 || kk > 0) ? 1u : 0u);
                            else
                                tc_mma_bf16_pair(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, idesc,
                                                 (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit_pair_multicast(smem_u32(&empty[stage]), 0x3);
                        if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    tc_commit_pair_multicast(smem_u32(&tfull[acc]), 0x3);
                }
                tc_commit_pair_multicast(smem_u32(fin), 0x3);
            }
            // both CTAs: every MMA writing this CTA's TMEM has completed
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(fin), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;
        int it = 0;
        for (int t = cid; t < total; t += ncl, ++it) {
            const Tile tl = decode_tile(t, mt_start, row_start, G, args.n_tiles, BN, args.N, P_BM);
            const int a_row = tl.a_row + static_cast<int>(rank) * 128;
            // this CTA's rows of the pair tile, clipped to the group (may be none)
            int rows_valid = row_start[tl.g + 1] - a_row;
            rows_valid = rows_valid < 0 ? 0 : (rows_valid > 128 ? 128 : rows_valid);
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            EpiScales sc;
            if constexpr (F8)
                sc = load_epi_scales(args.a_scale, args.b_scale, args.N, tl.g, tl.n, static_cast<long long>(a_row) + r,
                                     r < rows_valid, half, lane);
            if (!mbar_wait(smem_u32(&tfull[acc]), use & 1u, abort_flag, args.err)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            epilogue_tile<EPI, F8>(tbase, tl.g, a_row, rows_valid, tl.n, r, half, args, sc);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(map_to_cta(smem_u32(&tempty[acc]), 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();          // neither CTA releases TMEM or exits while the pair still works
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ----------------------------------------------------------------- plan
// m-tile prefix and row starts of G groups; offsets == nullptr means one group
// of n_rows rows.  Inconsistent offsets record DEV_ERR_OFFSETS and yield an
// empty plan (every GEMM over it then does nothing).
__global__ void plan_kernel(const int* __restrict__ offsets, int G, int n_rows, int bm, int* plan, int* err) {
    __shared__ int warp_sums[32];
    __shared__ int s_bad;
    __shared__ int s_carry;
    if (threadIdx.x == 0) { s_bad = 0; s_carry = 0; }
    __syncthreads();
    int* mt = plan;
    int* rs = plan + (G + 1);
    for (int base = 0; base < G; base += blockDim.x) {
        const int g = base + threadIdx.x;
        int cnt = 0;
        if (g < G) {
            const int a = offsets ? offsets[g] : 0;
            const int b = offsets ? offsets[g + 1] : n_rows;
            if (a < 0 || b < a || b > n_rows) s_bad = 1;
            rs[g] = a;
            if (g == G - 1) rs[G] = b;
            cnt = b > a ? (b - a + bm - 1) / bm : 0;
        }
        // block-wide exclusive scan of cnt
        int v = cnt;
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) warp_sums[wid] = v;
        __syncthreads();
        if (wid == 0) {
            int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int n = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += n;
            }
            warp_sums[lane] = w;   // inclusive
        }
        __syncthreads();
        const int excl = v - cnt + (wid > 0 ? warp_sums[wid - 1] : 0) + s_carry;
        if (g < G) mt[g] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) s_carry = excl + cnt;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        mt[G] = s_carry;
        if (s_bad) {
            for (int g = 0; g <= G; ++g) mt[g] = 0;
            set_dev_error(err, DEV_ERR_OFFSETS);
        }
    }
}

// ------------------------------------------------------- weight gradients
// out_g = A_g^T B_g (launch_wgrad_gemm): A [P, lda] and B [P, ldb] bf16 with one
// row per token (as the forward and the input-gradient GEMMs leave them), the
// contraction over group g's rows [offs[g], offs[g+1]).  The operands are read
// where they lie: TMA boxes of 64 rows x 64 columns (128-byte swizzle) are
// MN-major tiles, so no transposed copy is made.  The warp roles, pipeline and
// bounded waits are those of grouped_gemm_kernel; tiles (g, m, n) of 128 x 256
// (m inner, so consecutive tiles share the B rows in L2), K blocks of 64 rows
// from the group's first row.  In a group's last block the rows past its end
// belong to the next group (or are the zero fill past P): the MMA warp zeroes
// A's rows up to the next multiple of 16 (B there is finite data or zero fill,
// so those products vanish) and skips the 16-row steps past it.  A group with
// no rows issues no MMAs and its epilogue writes zeros.
struct WArgs {
    const int* offs;   // [G + 1] row offsets (device), or nullptr: one group [0, P)
    long long P;
    int G, M, N, m_tiles, n_tiles;
    int remap, split;
    int* err;
};

constexpr int W_BOX = 64 * 128;        // one 64-row x 64-column bf16 box, 8 KB

// The output is written by TMA stores from a 2 KB staging buffer per epilogue
// warp (32 rows x 16 fp32 columns, 64-byte swizzle): one store instruction per
// piece instead of 32 rows' worth of 16-byte stores per instruction.
constexpr int W_STAGE_OFF = (STAGES * STAGE_BYTES + BAR_BYTES + 2 * (kMaxGroups + 1) * 4 + 1023) / 1024 * 1024;
constexpr int W_PIECE = 32 * 16 * 4;
constexpr size_t W_SMEM_BYTES = 1024 + W_STAGE_OFF + EPI_WARPS * W_PIECE;

// Destination (map, x, y) of the 32 x 16 piece at output row row0, column col of group g:
//   remap 0: out [G M, N];  remap 1: packed gate/up rows -> W2 (gate, map 2) or W1 (up, map 1)
//   row 64 (q / 128) + q % 64 of [G M/2, N];  remap 2: column jj -> [jj / split][row][jj % split]
__device__ __forceinline__ const CUtensorMap* wgrad_piece(const WArgs& a, const CUtensorMap* o1, const CUtensorMap* o2,
                                                          int g, int row0, int col, int& x, int& y) {
    if (a.remap == 1) {
        x = col;
        y = g * (a.M / 2) + 64 * (row0 >> 7) + (row0 & 63);
        return (row0 & 127) < 64 ? o2 : o1;
    }
    if (a.remap == 2) {
        x = col % a.split;
        y = (col / a.split) * a.M + row0;
        return o1;
    }
    x = col;
    y = g * a.M + row0;
    return o1;
}

__global__ void __launch_bounds__(THREADS, 1)
wgrad_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2, const WArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + NACC;
    uint64_t* fin = tempty + NACC;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* offs = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + BAR_BYTES);    // [G + 1]
    int* bad = offs + kMaxGroups + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    if (threadIdx.x == 0) {
        *bad = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), EPI_WARPS);
        }
        mbar_init(smem_u32(fin), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    for (int i = threadIdx.x; i <= G; i += THREADS) {
        int v;
        bool ok;
        if (args.offs) {
            v = args.offs[i];
            ok = v >= 0 && v <= args.P && (i == 0 || v >= args.offs[i - 1]);
        } else {
            v = i == 0 ? 0 : static_cast<int>(args.P);
            ok = true;
        }
        offs[i] = v;
        if (!ok) *bad = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0 && *bad) {      // corrupt offsets: record it, every group empty
        set_dev_error(args.err, DEV_ERR_OFFSETS);
        for (int i = 0; i <= G; ++i) offs[i] = 0;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int per_g = args.m_tiles * args.n_tiles;
    const int total = G * per_g;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int g = t / per_g, rr = t - g * per_g;
                const int m = rr % args.m_tiles, n = rr / args.m_tiles;
                for (int r = offs[g]; r < offs[g + 1]; r += 64) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
#pragma unroll
                    for (int j = 0; j < BM / 64; ++j) tma_load_2d(sa + j * W_BOX, &tmA, fb, m * BM + 64 * j, r);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sa + A_STAGE + j * W_BOX, &tmB, fb, n * BN + 64 * j, r);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            const int pending = issued < STAGES ? issued : STAGES;
            for (int j = 1; j <= pending; ++j) {
                int s = stage - j;
                uint32_t ph = phase;
                if (s < 0) { s += STAGES; ph ^= 1u; }
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(smem_u32(&full[s]), ph)) {
                    if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // the whole warp walks the schedule: lane 0 waits and issues, all lanes
        // zero the rows past a group's end in its last K block
        constexpr uint32_t idesc = idesc_bf16_f32_mn(BM, BN);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int it = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
            const int g = t / per_g;
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (lane == 0) ok = mbar_wait(smem_u32(&tempty[acc]), (use & 1u) ^ 1u, abort_flag, args.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            const int r0 = offs[g], r1 = offs[g + 1];
            for (int r = r0; r < r1; r += 64) {
                if (lane == 0) ok = mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                uint8_t* sa = smem + stage * STAGE_BYTES;
                const int nrow = min(64, r1 - r);
                const int nk = (nrow + 15) >> 4;            // 16-row MMA steps that hold rows of the group
                const int zrows = 16 * nk - nrow;
                if (zrows > 0) {
                    // every lane sees the stage complete (the wait returns at once) before writing into it
                    if (mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err)) {
                        for (int i = lane; i < (BM / 64) * zrows * 8; i += 32) {
                            const int box = i / (zrows * 8), rem = i - box * zrows * 8;
                            *reinterpret_cast<uint4*>(sa + box * W_BOX + (nrow + (rem >> 3)) * 128 + (rem & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t adesc = smem_desc_sw128_mn(smem_u32(sa), W_BOX);
                    const uint64_t bdesc = smem_desc_sw128_mn(smem_u32(sa + A_STAGE), W_BOX);
                    for (int kk = 0; kk < nk; ++kk)       // 16 rows = 2048 B = 128 descriptor units
                        tc_mma_bf16(d_tmem, adesc + 128ull * kk, bdesc + 128ull * kk, idesc,
                                    (r > r0 || kk > 0) ? 1u : 0u);
                    tc_commit(smem_u32(&empty[stage]));
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(smem_u32(&tfull[acc]));
            __syncwarp();
        }
        if (lane == 0) {
            tc_commit(smem_u32(fin));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(fin), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
            }
        }
        __syncwarp();
    } else {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        uint8_t* piece = smem + W_STAGE_OFF + (warp - 2) * W_PIECE;
        const uint32_t piece_s = smem_u32(piece);
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int g = t / per_g, rr = t - g * per_g;
            const int m = rr % args.m_tiles, n = rr / args.m_tiles;
            const bool any = offs[g + 1] > offs[g];
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait(smem_u32(&tfull[acc]), use & 1u, abort_flag, args.err)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            const int row0 = m * BM + quarter * 32;       // this warp's 32 rows
            const int rem = args.N - n * BN;
            const int ncols = rem >= BN ? BN : rem;
            const int cend = min(ncols, (half + 1) * (BN / 2));
            if (row0 < args.M) {
#pragma unroll 1
                for (int c0 = half * (BN / 2); c0 < cend; c0 += 32) {
                    uint32_t v[32];
                    if (any) {
                        tmem_ld32(tbase + c0, v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0u;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = n * BN + c0 + 16 * h;
                        if (col >= args.N) break;
                        if (lane == 0) bulk_wait_read0();      // the previous piece has left the buffer
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int sw = q ^ ((lane >> 1) & 3);     // 64-byte swizzle of the 16-byte chunks
                            *reinterpret_cast<uint4*>(piece + lane * 64 + sw * 16) =
                                make_uint4(v[16 * h + 4 * q], v[16 * h + 4 * q + 1], v[16 * h + 4 * q + 2],
                                           v[16 * h + 4 * q + 3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            int x, y;
                            const CUtensorMap* map = wgrad_piece(args, &tmO1, &tmO2, g, row0, col, x, y);
                            tma_store_2d(map, piece_s, x, y);
                            bulk_commit();
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        }
        if (lane == 0) bulk_wait0();      // every store of this warp has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace tc

// ------------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static cudaError_t get_encode() {
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// 2D tensor map over a [rows, cols] row-major matrix of bf16 (f8 = false) or
// 8-bit codes (f8 = true) with a box of box_rows x 128 bytes and the 128-byte
// swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows, bool f8) {
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    const int es = f8 ? 1 : 2;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * es};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3D tensor map over the tiled weight layout [nblocks][256][128 bytes] (each
// block a contiguous 32 KB tile of 256 rows) with a box of box_rows x 128 bytes.
cudaError_t make_map_blocked(CUtensorMap* m, const void* base, long long nblocks, int box_rows, bool f8) {
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    const int es = f8 ? 1 : 2;
    cuuint64_t gdim[3] = {static_cast<cuuint64_t>(128 / es), 256, static_cast<cuuint64_t>(nblocks)};
    cuuint64_t gstride[2] = {128, 256 * 128};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2D bf16 output map [rows, cols] (row stride ldo elements) for 32 x 32 pieces
// stored with the 64-byte swizzle.
cudaError_t make_out_map_bf16(CUtensorMap* m, void* base, long long rows, long long cols, long long ldo) {
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ldo) * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2D fp32 output map [rows, cols] (row stride ldo elements) for 32 x 16 pieces.
static cudaError_t make_out_map_f32(CUtensorMap* m, void* base, long long rows, long long cols, long long ldo) {
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ldo) * 4};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, gdim, gstride, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The output map of a launch, when its epilogue stores pieces by TMA: bf16 h
// and y, dg/da of the SwiGLU backward, and fp32 outputs (written, or added by
// TMA reductions when accumulating).
static cudaError_t output_map(int epi, bool pair, void* out, long long out_rows, int out_cols,
                              long long ldo, CUtensorMap* m, int* use) {
    *use = 0;
    if (pair || out_rows < 1 || (reinterpret_cast<uintptr_t>(out) & 15u)) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (epi == EPI_SWIGLU || epi == EPI_BF16) {
        if (out_cols % 32 || ldo % 8) return cudaSuccess;
        e = make_out_map_bf16(m, out, out_rows, out_cols, ldo);
    } else if (epi == EPI_F32) {          // accumulate: the pieces are added by TMA reductions
        if (out_cols % 32 || ldo % 4) return cudaSuccess;
        e = make_out_map_f32(m, out, out_rows, out_cols, ldo);
    } else if (epi == EPI_DSWIGLU) {      // dg, da in the packed gate/up columns: 2 out_cols wide
        if (out_cols % 32 || ldo % 8) return cudaSuccess;
        e = make_out_map_bf16(m, out, out_rows, 2LL * out_cols, ldo);
    } else {
        return cudaSuccess;
    }
    if (e == cudaSuccess) *use = 1;
    return e;
}

static int g_num_sms[kMaxDevices];

cudaError_t num_sms(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_num_sms[dev]) {
        e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    *out = g_num_sms[dev];
    return cudaSuccess;
}

cudaError_t smem_attr_once(const void* fn, size_t bytes, bool (&set)[kMaxDevices]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (set[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) set[dev] = true;
    return e;
}

cudaError_t launch_plan(const int* offsets, int G, int n_rows, int bm, int* plan, cudaStream_t st) {
    tc::plan_kernel<<<1, 1024, 0, st>>>(offsets, G, n_rows, bm, plan, dev_error_ptr());
    count_launch();
    return cudaGetLastError();
}

// Kernel variant: the single-CTA kernel, or the CTA-pair kernel when the
// environment sets FS_TC_VARIANT=pair; FS_TC_VARIANT=pair_down (pair_up) keeps
// the single-CTA kernel except for the forward down (gate/up) projections.
static int variant_mode() {
    static int mode = -1;
    if (mode < 0) {
        const char* e = getenv("FS_TC_VARIANT");
        mode = 0;
        if (e && std::strcmp(e, "pair") == 0) mode = 1;
        if (e && std::strcmp(e, "pair_down") == 0) mode = 2;
        if (e && std::strcmp(e, "pair_up") == 0) mode = 3;
    }
    return mode;
}
static bool use_pair() { return variant_mode() == 1; }
bool tc_down_pair() { return variant_mode() == 2; }
bool tc_up_pair() { return variant_mode() == 3; }

template <int EPI>
static cudaError_t launch_tc_impl(const void* A, long long a_rows, const void* B, int G, int N, int K,
                                  const int* plan, int max_mtiles, void* out, long long ldo, int out_cols,
                                  const int* gather_rows, int gather_limit, bool b_blocked, cudaStream_t st,
                                  const TcExtra* ex) {
    const bool pair = (ex && ex->variant >= 0) ? ex->variant == 1 : use_pair();
    if (pair && gather_rows) return cudaErrorNotSupported;
    static bool set_single[kMaxDevices], set_pair[kMaxDevices];
    cudaError_t e = pair ? smem_attr_once(reinterpret_cast<const void*>(tc::pair_gemm_kernel<EPI>), tc::P_SMEM_BYTES,
                                          set_pair)
                         : smem_attr_once(reinterpret_cast<const void*>(tc::grouped_gemm_kernel<EPI>), tc::SMEM_BYTES,
                                          set_single);
    if (e != cudaSuccess) return e;
    CUtensorMap ta, tb;
    e = make_map(&ta, A, a_rows, K, gather_rows ? 1 : 128);
    if (e != cudaSuccess) return e;
    const int n_tiles = (N + tc::BN - 1) / tc::BN;
    if (b_blocked)
        e = make_map_blocked(&tb, B, static_cast<long long>(G) * n_tiles * (K / tc::BK), pair ? 128 : tc::BN);
    else
        e = make_map(&tb, B, static_cast<long long>(G) * N, K, pair ? 128 : tc::BN);
    if (e != cudaSuccess) return e;
    tc::Args args;
    args.plan = plan;
    args.G = G;
    args.N = N;
    args.K = K;
    args.n_tiles = (N + tc::BN - 1) / tc::BN;
    args.max_mtiles = max_mtiles;
    args.out = out;
    args.ldo = ldo;
    args.out_cols = out_cols;
    args.err = dev_error_ptr();
    args.gather_rows = gather_rows;
    args.gather_limit = gather_limit;
    args.b_blocked = b_blocked ? 1 : 0;
    args.a_scale = nullptr;
    args.b_scale = nullptr;
    args.aux = ex ? ex->aux : nullptr;
    args.aux_ld = ex ? ex->aux_ld : 0;
    args.accumulate = ex ? ex->accumulate : 0;
    int ksplit = ex ? ex->ksplit : 1;
    if (ksplit < 1 || ksplit > K / tc::BK) return cudaErrorInvalidValue;
    if (ksplit > 1 && (EPI != EPI_F32 || G != 1 || args.accumulate || gather_rows)) return cudaErrorInvalidValue;
    if (pair) ksplit = 1;
    args.ksplit = ksplit;
    args.split_rows = a_rows;
    if (EPI == EPI_COMBINE) {
        if (!ex || !ex->combine || G != 1 || gather_rows || ex->combine->k < 1 || ex->combine->k > kCombineEpiMaxK)
            return cudaErrorInvalidValue;
        args.cmb = *ex->combine;
    }
    CUtensorMap to = ta;
    e = output_map(EPI, pair, out, (gather_rows ? gather_limit : a_rows) * ksplit, out_cols, ldo, &to,
                   &args.tma_out);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = num_sms(&sms);
    if (e != cudaSuccess) return e;
    const long long max_tiles = static_cast<long long>(max_mtiles) * args.n_tiles * ksplit;
    if (pair) {
        long long clusters = sms / 2;
        if (max_tiles < clusters) clusters = max_tiles;
        if (clusters < 1) clusters = 1;
        tc::pair_gemm_kernel<EPI><<<static_cast<int>(2 * clusters), tc::THREADS, tc::P_SMEM_BYTES, st>>>(ta, tb, args);
    } else {
        int grid = static_cast<int>(max_tiles < sms ? max_tiles : sms);
        if (grid < 1) grid = 1;
        tc::grouped_gemm_kernel<EPI><<<grid, tc::THREADS, tc::SMEM_BYTES, st>>>(ta, tb, to, args);
    }
    count_launch();
    return cudaGetLastError();
}

template <int EPI>
static cudaError_t launch_tc_f8_impl(const void* A, long long a_rows, const float* a_scale, const void* B,
                                     const float* b_scale, int G, int N, int K, const int* plan, int max_mtiles,
                                     void* out, long long ldo, int out_cols, cudaStream_t st,
                                     const CombineEpi* cmb = nullptr, int variant = -1) {
    const bool pair = variant >= 0 ? variant == 1 : use_pair();
    static bool set_single[kMaxDevices], set_pair[kMaxDevices];
    cudaError_t e = pair ? smem_attr_once(reinterpret_cast<const void*>(tc::pair_gemm_kernel<EPI, true>),
                                          tc::P_SMEM_BYTES, set_pair)
                         : smem_attr_once(reinterpret_cast<const void*>(tc::grouped_gemm_kernel<EPI, true>),
                                          tc::SMEM_BYTES, set_single);
    if (e != cudaSuccess) return e;
    if (K % 128 || N % 128) return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    e = make_map(&ta, A, a_rows, K, 128, true);
    if (e != cudaSuccess) return e;
    const int n_tiles = (N + tc::BN - 1) / tc::BN;
    e = make_map_blocked(&tb, B, static_cast<long long>(G) * n_tiles * (K / 128), pair ? 128 : tc::BN, true);
    if (e != cudaSuccess) return e;
    tc::Args args;
    args.plan = plan;
    args.G = G;
    args.N = N;
    args.K = K;
    args.n_tiles = n_tiles;
    args.max_mtiles = max_mtiles;
    args.out = out;
    args.ldo = ldo;
    args.out_cols = out_cols;
    args.err = dev_error_ptr();
    args.gather_rows = nullptr;
    args.gather_limit = 0;
    args.b_blocked = 1;
    args.a_scale = a_scale;
    args.b_scale = b_scale;
    args.aux = nullptr;
    args.aux_ld = 0;
    args.accumulate = 0;
    if (EPI == EPI_COMBINE) {
        if (!cmb || G != 1 || cmb->k < 1 || cmb->k > kCombineEpiMaxK) return cudaErrorInvalidValue;
        args.cmb = *cmb;
    }
    CUtensorMap to = ta;
    e = output_map(EPI, pair, out, a_rows, out_cols, ldo, &to, &args.tma_out);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = num_sms(&sms);
    if (e != cudaSuccess) return e;
    const long long max_tiles = static_cast<long long>(max_mtiles) * n_tiles;
    if (pair) {
        long long clusters = sms / 2;
        if (max_tiles < clusters) clusters = max_tiles;
        if (clusters < 1) clusters = 1;
        tc::pair_gemm_kernel<EPI, true><<<static_cast<int>(2 * clusters), tc::THREADS, tc::P_SMEM_BYTES, st>>>(ta, tb,
                                                                                                           args);
    } else {
        int grid = static_cast<int>(max_tiles < sms ? max_tiles : sms);
        if (grid < 1) grid = 1;
        tc::grouped_gemm_kernel<EPI, true><<<grid, tc::THREADS, tc::SMEM_BYTES, st>>>(ta, tb, to, args);
    }
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_tc_gemm_f8(int epi, const void* A, long long a_rows, const float* a_scale, const void* B,
                              const float* b_scale, int G, int N, int K, const int* plan, int max_mtiles, void* out,
                              long long ldo, int out_cols, cudaStream_t st, const CombineEpi* combine, int variant) {
    switch (epi) {
        case EPI_COMBINE:
            return launch_tc_f8_impl<EPI_COMBINE>(A, a_rows, a_scale, B, b_scale, G, N, K, plan, max_mtiles, out, ldo,
                                                  out_cols, st, combine, variant);
        case EPI_SWIGLU:
            return launch_tc_f8_impl<EPI_SWIGLU>(A, a_rows, a_scale, B, b_scale, G, N, K, plan, max_mtiles, out, ldo,
                                                 out_cols, st, nullptr, variant);
        case EPI_BF16:
            return launch_tc_f8_impl<EPI_BF16>(A, a_rows, a_scale, B, b_scale, G, N, K, plan, max_mtiles, out, ldo,
                                               out_cols, st, nullptr, variant);
        case EPI_F32:
            return launch_tc_f8_impl<EPI_F32>(A, a_rows, a_scale, B, b_scale, G, N, K, plan, max_mtiles, out, ldo,
                                              out_cols, st, nullptr, variant);
        default:
            return cudaErrorInvalidValue;
    }
}

bool tc_gather_supported() { return !use_pair(); }

cudaError_t launch_tc_gemm(int epi, const void* A, long long a_rows, const void* B, int G, int N, int K,
                           const int* plan, int max_mtiles, void* out, long long ldo, int out_cols,
                           const int* gather_rows, int gather_limit, bool b_blocked, cudaStream_t st,
                           const TcExtra* ex) {
    switch (epi) {
        case EPI_SWIGLU:
            return launch_tc_impl<EPI_SWIGLU>(A, a_rows, B, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                              gather_rows, gather_limit, b_blocked, st, ex);
        case EPI_BF16:
            return launch_tc_impl<EPI_BF16>(A, a_rows, B, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                            gather_rows, gather_limit, b_blocked, st, ex);
        case EPI_F32:
            return launch_tc_impl<EPI_F32>(A, a_rows, B, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                           gather_rows, gather_limit, b_blocked, st, ex);
        case EPI_COMBINE:
            return launch_tc_impl<EPI_COMBINE>(A, a_rows, B, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                               gather_rows, gather_limit, b_blocked, st, ex);
        case EPI_DSWIGLU:
            if (!ex || !ex->aux) return cudaErrorInvalidValue;
            return launch_tc_impl<EPI_DSWIGLU>(A, a_rows, B, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                               gather_rows, gather_limit, b_blocked, st, ex);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_wgrad_gemm(const void* A, int lda, const void* B, int ldb, long long P, const int* offs, int G,
                              int M, int N, float* out, float* out2, int remap, int split, cudaStream_t st) {
    if (G < 1 || G > kMaxGroups || M < 1 || N < 1 || N % 32 || P < 1 || P > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (M > lda || N > ldb || lda % 8 || ldb % 8 || (!offs && G != 1)) return cudaErrorInvalidValue;
    if (G > 1 && M % 32) return cudaErrorInvalidValue;      // a 32-row piece never spans two groups
    if (remap == 1 && (M % 128 || !out2)) return cudaErrorInvalidValue;
    if (remap == 2 && (G != 1 || M % 32 || split < 32 || split % 32 || N % split)) return cudaErrorInvalidValue;
    static bool set_w[kMaxDevices];
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(tc::wgrad_gemm_kernel), tc::W_SMEM_BYTES, set_w);
    if (e != cudaSuccess) return e;
    // the operands as they lie: [P rows, lda] and [P rows, ldb], boxes of 64 rows x 64 columns
    CUtensorMap ta, tb;
    e = make_map(&ta, A, P, lda, 64);
    if (e == cudaSuccess) e = make_map(&tb, B, P, ldb, 64);
    if (e != cudaSuccess) return e;
    // fp32 outputs, written as 32-row x 16-column pieces with the 64-byte swizzle
    auto out_map = [&](CUtensorMap* mp, float* base, long long rows, long long cols) -> cudaError_t {
        cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
        cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 4};
        cuuint32_t box[2] = {16, 32};
        cuuint32_t estr[2] = {1, 1};
        return g_encode(mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, gdim, gstride, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
                   ? cudaSuccess
                   : cudaErrorInvalidValue;
    };
    CUtensorMap to1, to2;
    if (remap == 1) {
        e = out_map(&to1, out, static_cast<long long>(G) * (M / 2), N);
        if (e == cudaSuccess) e = out_map(&to2, out2, static_cast<long long>(G) * (M / 2), N);
    } else if (remap == 2) {
        e = out_map(&to1, out, static_cast<long long>(N / split) * M, split);
        to2 = to1;
    } else {
        e = out_map(&to1, out, static_cast<long long>(G) * M, N);
        to2 = to1;
    }
    if (e != cudaSuccess) return e;
    tc::WArgs args;
    args.offs = offs;
    args.P = P;
    args.G = G;
    args.M = M;
    args.N = N;
    args.m_tiles = (M + tc::BM - 1) / tc::BM;
    args.n_tiles = (N + tc::BN - 1) / tc::BN;
    args.remap = remap;
    args.split = split;
    args.err = dev_error_ptr();
    int sms = 0;
    e = num_sms(&sms);
    if (e != cudaSuccess) return e;
    const long long total = static_cast<long long>(G) * args.m_tiles * args.n_tiles;
    int grid = static_cast<int>(total < sms ? total : sms);
    if (grid < 1) grid = 1;
    tc::wgrad_gemm_kernel<<<grid, tc::THREADS, tc::W_SMEM_BYTES, st>>>(ta, tb, to1, to2, args);
    count_launch();
    return cudaGetLastError();
}

int tc_block_m() { return use_pair() ? tc::P_BM : tc::BM; }

int tc_router_ksplit(long long T, int E, int d) {
    if (use_pair() || T < 1) return 1;
    const long long tiles = ((T + tc::BM - 1) / tc::BM) * ((E + tc::BN - 1) / tc::BN);
    long long s = 148 / tiles;                  // about one CTA per SM of a 148-152 SM part
    const long long by_k = (d / tc::BK) / 2;    // at least two k-blocks per range
    if (s > 16) s = 16;
    if (s > by_k) s = by_k;
    return s < 1 ? 1 : static_cast<int>(s);
}
int tc_block_m_f8() { return use_pair() ? tc::P_BM : tc::BM; }

}  // namespace fs
