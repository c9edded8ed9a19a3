// Momentum + pack + sum-of-squares kernel, and the per-matrix norm finalise.
//
// DMuon's Newton-Schulz runs on "momentum-aggregated gradients" (gist.science
// technical summary, section 1).  Per element, in fp32:
//   M' = beta*M + grad          (stored back in the momentum's dtype)
//   u  = grad + beta*M'         (Nesterov; u = M' when disabled)
// u is written, in the operand dtype, into the bucket's packed [batch, m, n]
// buffer -- transposed for tall matrices so every packed matrix has m <= n --
// and sum(u^2) is reduced per 64 x 64 tile.  The finalise kernel sums a
// matrix's tile partials in a fixed order (so the result does not depend on
// which other matrices share the launch) and writes inv = 1/(||u||_F + eps).
//
// HBM-bound: 128-bit loads and stores along rows, the transpose staged
// through shared memory so both sides stay coalesced.
#include <cuda_bf16.h>

#include "internal.h"

namespace dmuon {
namespace {

constexpr int T = kMomTile;

__device__ __forceinline__ void load8(const void* base, int64_t i, int32_t type, float (&v)[8]) {
    if (type == ELEM_BF16) {
        const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + i);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(h[k]);
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
        const float4 a = p[0], b = p[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ void store8(void* base, int64_t i, int32_t type, const float (&v)[8]) {
    if (type == ELEM_BF16) {
        uint4 q;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + i) = q;
    } else {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + i);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

__device__ __forceinline__ float ld1(const void* p, int64_t i, int32_t t) {
    return t == ELEM_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                          : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st1(void* p, int64_t i, int32_t t, float v) {
    if (t == ELEM_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else static_cast<float*>(p)[i] = v;
}

__global__ void __launch_bounds__(kMomThreads) momentum_pack_kernel(const __grid_constant__ MomentumArgs a) {
    __shared__ float tile[T][T + 1];
    __shared__ float red[kMomThreads / 32];
    const int tid = threadIdx.x;

    for (int64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
        int lo = 0, hi = a.nslots - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.infos[mid].tile_begin <= t) lo = mid;
            else hi = mid - 1;
        }
        const MatInfo& mi = a.infos[lo];
        const int local = static_cast<int>(t - mi.tile_begin);
        const int r0 = (local / mi.tiles_c) * T, c0 = (local % mi.tiles_c) * T;
        const void* grad = a.grads[mi.gidx];
        void* mom = a.moms[mi.gidx];
        const int rows = mi.rows, cols = mi.cols;
        const int dt = mi.dtype;
        // 128-bit access along rows needs every row start on 16 bytes
        const bool rows_vec = (static_cast<int64_t>(cols) * (dt == ELEM_BF16 ? 2 : 4)) % 16 == 0;
        float ss = 0.0f;

#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int rr = tid / 8 + 32 * p, cc = (tid % 8) * 8;
            const int r = r0 + rr, c = c0 + cc;
            float u[8];
            if (r < rows && rows_vec && c + 8 <= cols) {
                const int64_t i = static_cast<int64_t>(r) * cols + c;
                float g[8], m[8];
                load8(grad, i, dt, g);
                load8(mom, i, dt, m);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    m[k] = fmaf(a.beta, m[k], g[k]);
                    u[k] = a.nesterov ? fmaf(a.beta, m[k], g[k]) : m[k];
                    ss = fmaf(u[k], u[k], ss);
                }
                store8(mom, i, dt, m);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    u[k] = 0.0f;
                    if (r < rows && c + k < cols) {
                        const int64_t i = static_cast<int64_t>(r) * cols + c + k;
                        const float g = ld1(grad, i, dt);
                        const float m = fmaf(a.beta, ld1(mom, i, dt), g);
                        st1(mom, i, dt, m);
                        u[k] = a.nesterov ? fmaf(a.beta, m, g) : m;
                        ss = fmaf(u[k], u[k], ss);
                    }
                }
            }
            if (!mi.transposed) {
                if (r < rows) {
                    if (c + 8 <= cols) {
                        store8(mi.x, static_cast<int64_t>(r) * mi.ldx + c, mi.x_type, u);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (c + k < cols) st1(mi.x, static_cast<int64_t>(r) * mi.ldx + c + k, mi.x_type, u[k]);
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) tile[rr][cc + k] = u[k];
            }
        }

        if (mi.transposed) {
            __syncthreads();
            // packed row = original column; 16 consecutive original rows per thread
            const int xr = tid / 4, rr0 = (tid % 4) * 16;
            const int c = c0 + xr;
            if (c < cols) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = tile[rr0 + e][xr];
                const int r = r0 + rr0;
                const int64_t base = static_cast<int64_t>(c) * mi.ldx + r;
                if (r + 16 <= rows) {
                    float v0[8], v1[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        v0[e] = v[e];
                        v1[e] = v[8 + e];
                    }
                    store8(mi.x, base, mi.x_type, v0);
                    store8(mi.x, base + 8, mi.x_type, v1);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (r + e < rows) st1(mi.x, base + e, mi.x_type, v[e]);
                }
            }
        }

        // deterministic block reduction of sum(u^2)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        if (tid == 0) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < kMomThreads / 32; ++w) s += red[w];
            mi.partials[local] = s;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) norm_finalize_kernel(const __grid_constant__ MomentumArgs a) {
    __shared__ double red[8];
    const MatInfo& mi = a.infos[blockIdx.x];
    double s = 0.0;
    for (int i = threadIdx.x; i < mi.ntiles; i += 256) s += static_cast<double>(mi.partials[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += red[w];
        const double inv = 1.0 / (sqrt(tot) + static_cast<double>(a.eps));
        SlotScalars sc;
        sc.inv = static_cast<float>(inv);
        sc.inv2 = static_cast<float>(inv * inv);
        a.scalars[blockIdx.x] = sc;
    }
}

}  // namespace

cudaError_t launch_momentum_pack(const MomentumArgs& a, cudaStream_t s) {
    if (a.total_tiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // persistent blocks: exactly as many as fit at once (a grid of 8 per SM,
    // 6 resident, ran its last 2 per SM as a second wave after the others)
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, momentum_pack_kernel, kMomThreads, 0) != cudaSuccess ||
            n < 1)
            n = 1;
        per_sm = n;
    }
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * per_sm;
    const int grid = static_cast<int>(a.total_tiles < cap ? a.total_tiles : cap);
    momentum_pack_kernel<<<grid, kMomThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const MomentumArgs& a, cudaStream_t s) {
    if (a.nslots <= 0) return cudaSuccess;
    norm_finalize_kernel<<<a.nslots, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dmuon
