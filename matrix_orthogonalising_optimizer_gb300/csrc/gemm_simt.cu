// fp32 FFMA batched GEMM with the fused Muon epilogue.
//
// Serves the fp32 validation mode (every product in true fp32, no tensor
// cores) and, in bf16 mode, the m x m Newton-Schulz products of small Gram
// buckets (m <= 256), where bf16 operands lose too much accuracy and the
// m^3 work is a small share of the step.
//
// One 64 x 64 output tile per block, 256 threads, each owning a 4 x 4
// sub-tile; K is consumed in slabs of 16 staged through shared memory.
// Symmetric products visit only the lower-triangle tiles and mirror.
#include "epilogue.cuh"

namespace dmuon {
namespace {

constexpr int BK = 16;

__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(const __grid_constant__ LaunchList L) {
    __shared__ float As[BK][kSimtBM + 4];
    __shared__ float Bs[BK][kSimtBN + 4];

    const int t = blockIdx.x;
    int gi = 0;
    while (gi + 1 < L.n && L.begin[gi + 1] <= t) ++gi;
    const GemmGroup& g = L.groups[L.idx[gi]];
    const int local = t - L.begin[gi];
    const int mat = local / g.tiles_per_mat;
    int idx = local % g.tiles_per_mat;
    int tm, tn;
    if (g.sym) {
        tm = 0;
        while (idx > tm) {  // row tile i holds i + 1 tiles
            idx -= tm + 1;
            ++tm;
        }
        tn = idx;
    } else {
        tm = idx / g.tiles_n;
        tn = idx % g.tiles_n;
    }

    const int tid = threadIdx.x;
    const int ty = tid / 16, tx = tid % 16;
    const int row0 = tm * kSimtBM, col0 = tn * kSimtBN;
    const char* A = static_cast<const char*>(g.a) + mat * g.a_bs * elem_size(g.a_type);
    const char* B = static_cast<const char*>(g.b) + mat * g.b_bs * elem_size(g.b_type);

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < g.K; k0 += BK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int q = tid + e * kSimtThreads;
            {  // A tile: 64 rows x 16 k, consecutive threads walk k
                const int i = q / BK, kk = q % BK;
                const int r = row0 + i, k = k0 + kk;
                As[kk][i] = (r < g.M && k < g.K)
                                ? load_elem(A, static_cast<int64_t>(r) * g.lda + k, g.a_type) : 0.0f;
            }
            if (!g.b_mn_major) {  // B stored N x K
                const int j = q / BK, kk = q % BK;
                const int c = col0 + j, k = k0 + kk;
                Bs[kk][j] = (c < g.N && k < g.K)
                                ? load_elem(B, static_cast<int64_t>(c) * g.ldb + k, g.b_type) : 0.0f;
            } else {              // B stored K x N
                const int kk = q / kSimtBN, j = q % kSimtBN;
                const int c = col0 + j, k = k0 + kk;
                Bs[kk][j] = (c < g.N && k < g.K)
                                ? load_elem(B, static_cast<int64_t>(k) * g.ldb + c, g.b_type) : 0.0f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

    const EpiCtx ctx = make_epi_ctx(g, L, mat);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + ty * 4 + i;
        if (r >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = col0 + tx * 4 + j;
            if (c < g.N) epi_element(g, ctx, L, r, c, acc[i][j]);
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const LaunchList& l, cudaStream_t s) {
    if (l.total_tiles <= 0) return cudaSuccess;
    gemm_simt_kernel<<<l.total_tiles, kSimtThreads, 0, s>>>(l);
    return cudaGetLastError();
}

}  // namespace dmuon
