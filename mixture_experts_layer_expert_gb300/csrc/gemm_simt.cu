// gemm_simt.cu -- grouped GEMM in fp32 FMA for the fp32 workload.
//
// The fp32 configuration must match an fp64 definition to 1e-5 relative, which
// rules out TF32 tensor cores; its shapes are small (launch-bound), so a
// shared-memory-tiled SIMT kernel is the right tool.  Same grouping, plan and
// epilogues as the tensor-core kernel ("FarSkip-Collective", §2.1 MLP and MoE
// equations):
//   EPI_SWIGLU : H = SiLU(X W2^T) * (X W1^T)  (tile = 64 rows x [64 gate | 64 up])
//   EPI_F32    : Y = A B^T                      (tile = 64 x 64)
#include "common.cuh"
#include "kernels.h"

namespace fs {
namespace simt {

constexpr int BM = 64;
constexpr int BK = 16;
constexpr int THREADS = 256;

struct Args {
    const int* plan;
    int G, N, K, n_tiles, max_mtiles;
    float* out;
    long long ldo;
    int out_cols;
    int* err;
    const int* gather_rows;   // A row of GEMM row p = gather_rows[p], or nullptr
    int gather_limit;
    long long a_rows;         // rows of A (bound of a gathered row)
};

template <int EPI>
__global__ void __launch_bounds__(THREADS)
simt_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B, const Args args) {
    constexpr int BNT = (EPI == EPI_SWIGLU) ? 128 : 64;   // B rows per tile
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BNT + 4];

    const int* mt_start = args.plan;
    const int* row_start = args.plan + args.G + 1;
    int total_m = mt_start[args.G];
    if (total_m < 0 || total_m > args.max_mtiles) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_dev_error(args.err, DEV_ERR_OFFSETS);
        return;
    }
    const int t = blockIdx.x;
    if (t >= total_m * args.n_tiles) return;
    const int q = t / args.n_tiles;
    int lo = 0, hi = args.G;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (mt_start[mid] <= q) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int mtiles = mt_start[g + 1] - mt_start[g];
    const int local = t - mt_start[g] * args.n_tiles;
    const int n = local / mtiles;
    const int m = local - n * mtiles;
    const int a_row = row_start[g] + m * BM;
    const int row_end = row_start[g + 1];
    const long long b_row0 = static_cast<long long>(g) * args.N + static_cast<long long>(n) * BNT;
    const int b_rows_valid = args.N - n * BNT;

    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4] = {};
    float acc2[4][4] = {};   // up half (EPI_SWIGLU)

    for (int k0 = 0; k0 < args.K; k0 += BK) {
        {   // A: 64 rows x 16 -> one float4 per thread
            const int r = tid >> 2, kq = (tid & 3) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (a_row + r < row_end) {
                long long src = a_row + r;
                if (args.gather_rows) {
                    src = a_row + r < args.gather_limit ? args.gather_rows[a_row + r] : 0;
                    if (src < 0 || src >= args.a_rows) {      // corrupt permutation: record, read nothing
                        set_dev_error(args.err, DEV_ERR_OFFSETS);
                        src = -1;
                    }
                }
                if (src >= 0) v = *reinterpret_cast<const float4*>(A + src * args.K + k0 + kq);
            }
            As[kq + 0][r] = v.x; As[kq + 1][r] = v.y; As[kq + 2][r] = v.z; As[kq + 3][r] = v.w;
        }
        for (int i = tid; i < BNT * 4; i += THREADS) {   // B: BNT rows x 16
            const int r = i >> 2, kq = (i & 3) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < b_rows_valid)
                v = *reinterpret_cast<const float4*>(B + (b_row0 + r) * args.K + k0 + kq);
            Bs[kq + 0][r] = v.x; Bs[kq + 1][r] = v.y; Bs[kq + 2][r] = v.z; Bs[kq + 3][r] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4], b2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
            if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
                for (int j = 0; j < 4; ++j) b2[j] = Bs[kk][64 + tx * 4 + j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if constexpr (EPI == EPI_SWIGLU) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = a_row + ty * 4 + i;
        if (row >= row_end) continue;
        float* orow = args.out + static_cast<long long>(row) * args.ldo;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (EPI == EPI_SWIGLU) {
                // packed rows [n*128, n*128+64) gate, [n*128+64, n*128+128) up -> columns n*64 + j
                const int col = n * 64 + tx * 4 + j;
                const float gte = acc[i][j];
                orow[col] = (gte / (1.0f + expf(-gte))) * acc2[i][j];
            } else {
                const int col = n * 64 + tx * 4 + j;
                if (col < args.out_cols) orow[col] = acc[i][j];
            }
        }
    }
}

}  // namespace simt

int simt_block_m() { return simt::BM; }

cudaError_t launch_simt_gemm(int epi, const float* A, long long a_rows, const float* B, int G, int N, int K,
                             const int* plan, int max_mtiles, float* out, long long ldo, int out_cols,
                             const int* gather_rows, int gather_limit, cudaStream_t st) {
    simt::Args args;
    args.plan = plan;
    args.G = G;
    args.N = N;
    args.K = K;
    args.n_tiles = (epi == EPI_SWIGLU) ? N / 128 : (N + 63) / 64;
    args.max_mtiles = max_mtiles;
    args.out = out;
    args.ldo = ldo;
    args.out_cols = out_cols;
    args.err = dev_error_ptr();
    args.gather_rows = gather_rows;
    args.gather_limit = gather_limit;
    args.a_rows = a_rows;
    long long grid = static_cast<long long>(max_mtiles) * args.n_tiles;
    if (grid < 1) grid = 1;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (epi == EPI_SWIGLU)
        simt::simt_gemm_kernel<EPI_SWIGLU><<<static_cast<unsigned>(grid), simt::THREADS, 0, st>>>(A, B, args);
    else
        simt::simt_gemm_kernel<EPI_F32><<<static_cast<unsigned>(grid), simt::THREADS, 0, st>>>(A, B, args);
    count_launch();
    return cudaGetLastError();
}

}  // namespace fs
