// gemm_mx.cu -- persistent grouped GEMM on block-scaled FP8 operands (the MX
// expert path): tcgen05.mma kind::mxf8f6f4.block_scale with E4M3 codes in
// shared memory (TMA, 128-byte swizzle) and one UE8M0 scale per row per 32
// elements of K for each operand, the scales copied into TMEM with tcgen05.cp
// (layouts in mx.cuh).  fp32 accumulate in TMEM.
//
// The grouped structure, warp roles, tile order and bounded waits are those of
// gemm_tc.cu (one CTA per SM, 10 warps: TMA producer, MMA issuer, 8 epilogue
// warps), with two differences forced by the scales:
//  * TMEM holds one 128 x 256 fp32 accumulator (256 columns) plus a ring of
//    scale-factor slots; two accumulators would fill all 512 columns.  So the
//    epilogue warps first copy their whole share of the accumulator into
//    registers (128 columns each), release TMEM, and only then compute and
//    store: the next tile's MMAs wait for that copy only.
//  * every group's rows start at a multiple of 128 (the MX Dispatch pads each
//    expert's segment), so an A tile's scales are one 512-byte chunk per stage.
// One stage = 128 K elements: A 128 x 128 B + B 256 x 128 B of codes, 512 B of
// A scales, 1 KB of B scales; per stage 4 MMAs of 128 x 256 x 32, MMA kk using
// byte kk of each scale word (the 4 blocks of 32 of the stage).
//
// Epilogues: EPI_SWIGLU writes the hidden h = SiLU(g) u rounded to bf16 and
// quantised in blocks of 32 straight into an MX matrix (codes and scales: the
// down projection's A operand); EPI_BF16 writes y (bf16); EPI_F32 writes fp32.
#include <cudaTypedefs.h>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "mx.cuh"

namespace fs {
namespace mx {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;                       // K elements (bytes) per stage
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK;              // 16 KB
constexpr int B_STAGE = BN * BK;              // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int SFA_BYTES = 512;
constexpr int SFB_BYTES = 1024;
constexpr int SF_STAGE = SFA_BYTES + SFB_BYTES;
constexpr int SF_OFF = STAGES * STAGE_BYTES;                  // scale chunks after the code stages
constexpr int BAR_OFF = SF_OFF + STAGES * SF_STAGE;
constexpr int BAR_BYTES = 256;
constexpr int PLAN_OFF = BAR_OFF + BAR_BYTES;
constexpr int PIECE_OFF = (PLAN_OFF + 2 * (kMaxGroups + 1) * 4 + 1023) / 1024 * 1024;
constexpr int PIECE_BYTES = 2048;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr size_t SMEM_BYTES = 1024 + PIECE_OFF + EPI_WARPS * PIECE_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int SF_SLOTS = 8;                   // scale-factor slots in TMEM (a ring, two per smem stage)
constexpr int SF_COL0 = BN;                   // slot j: A scales at SF_COL0 + 12 j (4 columns), B at + 4 (8)
constexpr int kGroupM = 16;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(SF_COL0 + 12 * SF_SLOTS <= TMEM_COLS, "TMEM columns");

struct Args {
    const int* plan;          // [2 (G + 1)]: m-tile prefix, row starts (multiples of 128)
    int G, N, K, n_tiles, max_mtiles;
    const uint8_t* a_sf;      // A scale chunks [rows128 / 128][K / 128][512]
    const uint8_t* b_sf;      // B scale chunks [G][n_tiles][K / 128][1024]
    void* out;
    long long ldo;            // output row stride (elements)
    int out_cols;
    uint8_t* h_sf;            // EPI_SWIGLU: scale chunks of the MX hidden out (codes at out, row stride ldo bytes)
    int tma_out;
    int* err;
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// TMEM <- shared memory scale chunk: 32 rows of 16 bytes, each row i copied to
// lane i of every lane quarter, 4 columns (tcgen05.cp 32x128b.warpx4).  The
// source descriptor: start >> 4, no swizzle, 8-row core groups 128 B apart.
__device__ __forceinline__ void sf_copy(uint32_t taddr, uint32_t saddr) {
    uint64_t desc = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    desc |= static_cast<uint64_t>(128u >> 4) << 16;
    desc |= static_cast<uint64_t>(128u >> 4) << 32;
    desc |= 1ull << 46;
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// D (fp32, TMEM) (+)= (A * sA) (B * sB)^T, E4M3 codes with UE8M0 block scales.
__device__ __forceinline__ void mma_mx(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Instruction descriptor, kind::mxf8f6f4: B scale byte (bits 4-5), A and B
// E4M3 (format 0 in bits 7-9, 10-12), K-major, N >> 3 (17-22), UE8M0 scales
// (bit 23), M >> 4 (24-28), A scale byte (29-30).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, int sf_id) {
    return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

struct Tile {
    int g, m, n, a_row, rows_valid;
};

__device__ __forceinline__ Tile decode(int t, const int* mt_start, const int* row_start, int G, int n_tiles) {
    const int q = t / n_tiles;
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (mt_start[mid] <= q) lo = mid; else hi = mid;
    }
    Tile r;
    r.g = lo;
    const int mtiles = mt_start[lo + 1] - mt_start[lo];
    const int local = t - mt_start[lo] * n_tiles;
    const int GM = mtiles <= 2 * kGroupM ? mtiles : kGroupM;
    const int blk = local / (GM * n_tiles);
    const int gm = min(GM, mtiles - blk * GM);
    const int rr = local - blk * GM * n_tiles;
    r.n = rr / gm;
    r.m = blk * GM + (rr - r.n * gm);
    r.a_row = row_start[lo] + r.m * BM;
    const int rem = row_start[lo + 1] - r.a_row;
    r.rows_valid = rem < BM ? rem : BM;
    return r;
}

// One 32 x 32 bf16 piece through the warp's staging buffer and a TMA store.
__device__ __forceinline__ void store_piece(const CUtensorMap* tmo, uint8_t* piece, const uint32_t* pk, int lane, int x,
                                            int y) {
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int sw = q ^ ((lane >> 1) & 3);
        *reinterpret_cast<uint4*>(piece + lane * 64 + sw * 16) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmo, smem_u32(piece), x, y);
        bulk_commit();
    }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmO, const Args args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* full = bars;                 // [STAGES]
    uint64_t* empty = bars + STAGES;       // [STAGES]
    uint64_t* tfull = bars + 2 * STAGES;   // [1]
    uint64_t* tempty = tfull + 1;          // [1]
    uint64_t* fin = tempty + 1;            // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* mt_start = reinterpret_cast<int*>(smem + PLAN_OFF);
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
        mbar_init(smem_u32(tfull), 1);
        mbar_init(smem_u32(tempty), EPI_WARPS);
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
    const int total = total_mtiles * args.n_tiles;
    const int num_kb = args.K / BK;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = decode(t, mt_start, row_start, G, args.n_tiles);
                const uint8_t* sfa = args.a_sf + static_cast<size_t>(tl.a_row / BM) * num_kb * SFA_BYTES;
                const uint8_t* sfb = args.b_sf + (static_cast<size_t>(tl.g) * args.n_tiles + tl.n) * num_kb * SFB_BYTES;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES + SF_STAGE);
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    uint8_t* sf = smem + SF_OFF + stage * SF_STAGE;
                    tma_load_2d(smem_u32(sa), &tmA, fb, kb * BK, tl.a_row);
                    tma_load_3d(smem_u32(sa + A_STAGE), &tmB, fb, 0, 0, (tl.g * args.n_tiles + tl.n) * num_kb + kb);
                    bulk_load(smem_u32(sf), sfa + static_cast<size_t>(kb) * SFA_BYTES, SFA_BYTES, fb);
                    bulk_load(smem_u32(sf + SFA_BYTES), sfb + static_cast<size_t>(kb) * SFB_BYTES, SFB_BYTES, fb);
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
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            uint32_t slot = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                // the epilogue has copied the previous tile out of TMEM
                if (!mbar_wait(smem_u32(tempty), (static_cast<uint32_t>(it) & 1u) ^ 1u, abort_flag, args.err)) break;
                tc_fence_after();
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err)) { ok = false; break; }
                    tc_fence_after();
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    const uint32_t sf = smem_u32(smem + SF_OFF + stage * SF_STAGE);
                    const uint32_t tsa = tmem_base + SF_COL0 + 12u * slot;
                    const uint32_t tsb = tsa + 4u;
                    sf_copy(tsa, sf);                       // A: 128 rows x 4 blocks
                    sf_copy(tsb, sf + SFA_BYTES);           // B rows 0..127
                    sf_copy(tsb + 4u, sf + SFA_BYTES + 512u);   // B rows 128..255
                    const uint64_t adesc = smem_desc_sw128(smem_u32(sa));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(sa + A_STAGE));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mx(tmem_base, adesc + 2ull * kk, bdesc + 2ull * kk, idesc_mx(BM, BN, kk), tsa, tsb,
                               (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(smem_u32(&empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    slot = (slot + 1u) % SF_SLOTS;
                }
                if (!ok) break;
                tc_commit(smem_u32(tfull));
            }
            tc_commit(smem_u32(fin));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(fin), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) { set_dev_error(args.err, DEV_ERR_TIMEOUT); break; }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;          // which 128 columns of the tile
        const int r = quarter * 32 + lane;
        uint8_t* piece = smem + PIECE_OFF + (warp - 2) * PIECE_BYTES;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const Tile tl = decode(t, mt_start, row_start, G, args.n_tiles);
            if (!mbar_wait(smem_u32(tfull), static_cast<uint32_t>(it) & 1u, abort_flag, args.err)) break;
            tc_fence_after();
            // this warp's 32 rows x 128 columns, copied out of TMEM at once
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * 128);
            uint32_t v[128];
            tmem_ld32(tb, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tb + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld32(tb + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
            tmem_ld32(tb + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(tempty));
            const bool row_ok = r < tl.rows_valid;
            const long long orow = static_cast<long long>(tl.a_row) + r;
            const int lanew = r & 31, q32 = r & ~31;
            const bool piece_ok = args.tma_out && q32 + 32 <= tl.rows_valid;
            if constexpr (EPI == EPI_SWIGLU) {
                // packed columns of this half: gate 64 | up 64 -> hidden columns
                // 128 n + 64 half + [0, 64), two blocks of 32
                const int hc0 = tl.n * 128 + half * 64;
                if (row_ok && hc0 < args.out_cols) {
                    uint8_t* H = static_cast<uint8_t*>(args.out) + orow * args.ldo;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        float h[32];
                        float amax = 0.0f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float g = __uint_as_float(v[32 * b + j]), u = __uint_as_float(v[64 + 32 * b + j]);
                            // the stored hidden: bf16 rounding of SiLU(g) u
                            h[j] = __bfloat162float(__float2bfloat16_rn(silu_f(g) * u));
                            amax = fmaxf(amax, fabsf(h[j]));
                        }
                        const MxQuant m = mx_quant(amax);
                        uint32_t c[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float a0, a1, a2, a3;
                            if (!m.q.wide) {
                                a0 = h[4 * j] * m.q.mult; a1 = h[4 * j + 1] * m.q.mult;
                                a2 = h[4 * j + 2] * m.q.mult; a3 = h[4 * j + 3] * m.q.mult;
                            } else {
                                a0 = scaled_wide(h[4 * j], m.q.e); a1 = scaled_wide(h[4 * j + 1], m.q.e);
                                a2 = scaled_wide(h[4 * j + 2], m.q.e); a3 = scaled_wide(h[4 * j + 3], m.q.e);
                            }
                            c[j] = cvt_e4m3x2(a0, a1) | (cvt_e4m3x2(a2, a3) << 16);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(H + hc0 + 32 * b);
                        dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
                        dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
                        args.h_sf[mx_sf_byte(orow, (hc0 + 32 * b) / 32, args.out_cols)] = m.ue8m0;
                    }
                }
            } else if constexpr (EPI == EPI_BF16) {
                const int c_base = tl.n * BN + half * 128;
                __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(args.out);
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    if (c_base + c0 >= args.out_cols) break;
                    uint32_t pk[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        pk[q] = pack_bf16x2(__uint_as_float(v[c0 + 2 * q]), __uint_as_float(v[c0 + 2 * q + 1]));
                    if (piece_ok) {
                        store_piece(&tmO, piece, pk, lanew, c_base + c0, tl.a_row + q32);
                    } else if (row_ok) {
                        uint4* dst = reinterpret_cast<uint4*>(Y + orow * args.ldo + c_base + c0);
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                    }
                }
            } else {   // EPI_F32
                const int c_base = tl.n * BN + half * 128;
                float* Z = static_cast<float*>(args.out);
                if (row_ok) {
#pragma unroll
                    for (int c0 = 0; c0 < 128; c0 += 4) {
                        if (c_base + c0 >= args.out_cols) break;
                        *reinterpret_cast<uint4*>(Z + orow * args.ldo + c_base + c0) =
                            make_uint4(v[c0], v[c0 + 1], v[c0 + 2], v[c0 + 3]);
                    }
                }
            }
        }
        if (args.tma_out && lane == 0) bulk_wait0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace mx

// ------------------------------------------------------------------- host
template <int EPI>
static cudaError_t launch_mx_impl(const void* A, long long a_rows, const uint8_t* a_sf, const void* B,
                                  const uint8_t* b_sf, int G, int N, int K, const int* plan, int max_mtiles, void* out,
                                  long long ldo, int out_cols, uint8_t* h_sf, cudaStream_t st) {
    static bool set_mx[kMaxDevices];
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(mx::mx_gemm_kernel<EPI>), mx::SMEM_BYTES, set_mx);
    if (e != cudaSuccess) return e;
    if (K % 128 || N % 128 || a_rows % 128 || G < 1 || G > kMaxGroups) return cudaErrorInvalidValue;
    CUtensorMap ta, tb, to;
    e = make_map(&ta, A, a_rows, K, 128, true);
    if (e != cudaSuccess) return e;
    const int n_tiles = (N + mx::BN - 1) / mx::BN;
    e = make_map_blocked(&tb, B, static_cast<long long>(G) * n_tiles * (K / 128), mx::BN, true);
    if (e != cudaSuccess) return e;
    mx::Args args;
    args.plan = plan;
    args.G = G;
    args.N = N;
    args.K = K;
    args.n_tiles = n_tiles;
    args.max_mtiles = max_mtiles;
    args.a_sf = a_sf;
    args.b_sf = b_sf;
    args.out = out;
    args.ldo = ldo;
    args.out_cols = out_cols;
    args.h_sf = h_sf;
    args.err = dev_error_ptr();
    args.tma_out = 0;
    to = ta;
    if (EPI == EPI_BF16 && out_cols % 32 == 0 && ldo % 8 == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
        e = make_out_map_bf16(&to, out, a_rows, out_cols, ldo);
        if (e != cudaSuccess) return e;
        args.tma_out = 1;
    }
    if (EPI == EPI_SWIGLU && (!h_sf || ldo < out_cols)) return cudaErrorInvalidValue;
    int sms = 0;
    e = num_sms(&sms);
    if (e != cudaSuccess) return e;
    const long long max_tiles = static_cast<long long>(max_mtiles) * n_tiles;
    int grid = static_cast<int>(max_tiles < sms ? max_tiles : sms);
    if (grid < 1) grid = 1;
    mx::mx_gemm_kernel<EPI><<<grid, mx::THREADS, mx::SMEM_BYTES, st>>>(ta, tb, to, args);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_mx_gemm(int epi, const void* A, long long a_rows, const uint8_t* a_sf, const void* B,
                           const uint8_t* b_sf, int G, int N, int K, const int* plan, int max_mtiles, void* out,
                           long long ldo, int out_cols, uint8_t* h_sf, cudaStream_t st) {
    switch (epi) {
        case EPI_SWIGLU:
            return launch_mx_impl<EPI_SWIGLU>(A, a_rows, a_sf, B, b_sf, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                              h_sf, st);
        case EPI_BF16:
            return launch_mx_impl<EPI_BF16>(A, a_rows, a_sf, B, b_sf, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                            h_sf, st);
        case EPI_F32:
            return launch_mx_impl<EPI_F32>(A, a_rows, a_sf, B, b_sf, G, N, K, plan, max_mtiles, out, ldo, out_cols,
                                           h_sf, st);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace fs
