// fp32 FFMA batched GEMM with the fused Muon epilogue.
//
// Serves the fp32 validation mode (every product in true fp32, no tensor
// cores) and, in bf16 mode, the m x m Newton-Schulz products of small Gram
// buckets (m <= 256), where bf16 operands lose too much accuracy and the
// m^3 work is a small share of the step.
//
// One 64 x 64 output tile per block, 256 threads, each owning a 4 x 4
// sub-tile; K is consumed in slabs of 32 staged through shared memory, the
// next slab's global loads in flight during the current slab's FFMAs, with
// float4 shared-memory reads.
// Symmetric products visit only the lower-triangle tiles and mirror.
#include "epilogue.cuh"

namespace dmuon {
namespace {

constexpr int BK = 32;
constexpr int LDS = kSimtBM + 4;  // padded row: 272 bytes keeps float4 reads aligned

// Operand tile loads for one K slab: A as As[k][i] (64 rows x BK), B as
// Bs[k][j].  Each thread holds 8 elements of each between slabs, so the next
// slab's global loads overlap this slab's FFMAs.
struct SlabRegs {
    float a[8], b[8];
};

__device__ __forceinline__ void load_slab(const GemmGroup& g, const char* A, const char* B, int row0, int col0,
                                          int k0, int tid, SlabRegs& sr) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int q = tid + e * kSimtThreads;
        {  // A: consecutive threads walk k (32 consecutive k per row)
            const int i = q / BK, kk = q % BK;
            const int r = row0 + i, k = k0 + kk;
            sr.a[e] = (r < g.M && k < g.K) ? load_elem(A, static_cast<int64_t>(r) * g.lda + k, g.a_type) : 0.0f;
        }
        if (!g.b_mn_major) {  // B stored N x K
            const int j = q / BK, kk = q % BK;
            const int c = col0 + j, k = k0 + kk;
            sr.b[e] = (c < g.N && k < g.K) ? load_elem(B, static_cast<int64_t>(c) * g.ldb + k, g.b_type) : 0.0f;
        } else {              // B stored K x N
            const int kk = q / kSimtBN, j = q % kSimtBN;
            const int c = col0 + j, k = k0 + kk;
            sr.b[e] = (c < g.N && k < g.K) ? load_elem(B, static_cast<int64_t>(k) * g.ldb + c, g.b_type) : 0.0f;
        }
    }
}

__device__ __forceinline__ void store_slab(const GemmGroup& g, int tid, const SlabRegs& sr, float (*As)[LDS],
                                           float (*Bs)[LDS]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int q = tid + e * kSimtThreads;
        As[q % BK][q / BK] = sr.a[e];
        if (!g.b_mn_major) Bs[q % BK][q / BK] = sr.b[e];
        else Bs[q / kSimtBN][q % kSimtBN] = sr.b[e];
    }
}

__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(const __grid_constant__ LaunchList L) {
    __shared__ __align__(16) float As[BK][LDS];
    __shared__ __align__(16) float Bs[BK][LDS];

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

    SlabRegs sr;
    load_slab(g, A, B, row0, col0, 0, tid, sr);
    for (int k0 = 0; k0 < g.K; k0 += BK) {
        store_slab(g, tid, sr, As, Bs);
        __syncthreads();
        if (k0 + BK < g.K) load_slab(g, A, B, row0, col0, k0 + BK, tid, sr);  // in flight during the FFMAs
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }

    const EpiRegs e = load_epi(g, L, mat);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + ty * 4 + i;
        if (r >= e.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = col0 + tx * 4 + j;
            if (c < e.N) epi_element_regs(e, r, c, acc[i][j]);
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
