// Momentum + pack + sum-of-squares kernel, and the per-matrix norm finalise.
//
// DMuon's Newton-Schulz runs on "momentum-aggregated gradients" (gist.science
// technical summary, section 1).  Per element, in fp32:
//   M' = beta*M + grad          (stored back in the momentum's dtype)
//   u  = grad + beta*M'         (Nesterov; u = M' when disabled)
// u is written, in the operand dtype, into the bucket's packed [batch, m, n]
// buffer -- transposed for tall matrices so every packed matrix has m <= n --
// and sum(u^2) is reduced per warp of each 64 x 64 tile.  The finalise kernel
// sums a matrix's partials in a fixed order (so the result does not depend on
// which other matrices share the launch) and writes inv = 1/(||u||_F + eps).
//
// HBM-bound.  Persistent blocks walk the tiles of every matrix of the wave,
// keeping the current matrix's record and pointers in registers (a lookup
// per tile would put a chain of dependent loads before every tile's data).
// Each thread issues its 128-bit grad and momentum loads for both of its rows
// before using any; stores are 128-bit along rows, the transpose for tall
// matrices staged through a double-buffered shared tile so both sides stay
// coalesced with one barrier per transposed tile and none otherwise.
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

__device__ __forceinline__ void unpack8(const uint4& q, float (&v)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(h[k]);
        v[2 * k] = f.x;
        v[2 * k + 1] = f.y;
    }
}

// Registers are capped so five blocks fit on an SM with both rows' loads in
// flight per thread.
constexpr int kMomMinBlocks = 5;

__global__ void __launch_bounds__(kMomThreads, kMomMinBlocks) momentum_pack_kernel(
    const __grid_constant__ MomentumArgs a) {
    // two transpose tiles: a block writes one while others may still read the
    // other, so one barrier per transposed tile is enough
    __shared__ float tile[2][T][T + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // the record of the matrix holding this block's current tile, and its
    // grad and momentum pointers, kept while the block's tiles stay inside it
    int slot = -1;
    int64_t begin = 0, end = 0;
    const void* grad = nullptr;
    void* mom = nullptr;
    int buf = 0;
    for (int64_t t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
        if (t >= end) {
            // tiles are numbered matrix after matrix: search forward, trying
            // the next matrix first
            int lo = slot + 1, hi = a.nslots - 1;
            if (lo < hi && a.infos[lo + 1].tile_begin > t) hi = lo;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.infos[mid].tile_begin <= t) lo = mid;
                else hi = mid - 1;
            }
            slot = lo;
            const MatInfo& nm = a.infos[slot];
            begin = nm.tile_begin;
            end = begin + nm.ntiles;
            grad = a.grads[nm.gidx];
            mom = a.moms[nm.gidx];
        }
        const MatInfo& mi = a.infos[slot];
        const int local = static_cast<int>(t - begin);
        const int r0 = (local / mi.tiles_c) * T, c0 = (local % mi.tiles_c) * T;
        const int rows = mi.rows, cols = mi.cols;
        const int dt = mi.dtype;
        // 128-bit access along rows needs every row start on 16 bytes
        const bool rows_vec = (static_cast<int64_t>(cols) * (dt == ELEM_BF16 ? 2 : 4)) % 16 == 0;
        float ss = 0.0f;

        // bf16 storage: both rows' grad and momentum loads go out before any use
        const bool bf_vec = dt == ELEM_BF16 && rows_vec;
        uint4 rg[2], rm[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int r = r0 + tid / 8 + 32 * p, c = c0 + (tid % 8) * 8;
            if (bf_vec && r < rows && c + 8 <= cols) {
                const int64_t i = static_cast<int64_t>(r) * cols + c;
                rg[p] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(grad) + i);
                rm[p] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(mom) + i);
            }
        }

#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int rr = tid / 8 + 32 * p, cc = (tid % 8) * 8;
            const int r = r0 + rr, c = c0 + cc;
            float u[8];
            if (r < rows && rows_vec && c + 8 <= cols) {
                const int64_t i = static_cast<int64_t>(r) * cols + c;
                float g[8], m[8];
                if (bf_vec) {
                    unpack8(rg[p], g);
                    unpack8(rm[p], m);
                } else {
                    load8(grad, i, dt, g);
                    load8(mom, i, dt, m);
                }
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
                for (int k = 0; k < 8; ++k) tile[buf][rr][cc + k] = u[k];
            }
        }

        if (mi.transposed) {  // the same for the whole block
            __syncthreads();
            // packed row = original column; 16 consecutive original rows per thread
            const int xr = tid / 4, rr0 = (tid % 4) * 16;
            const int c = c0 + xr;
            if (c < cols) {
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = tile[buf][rr0 + e][xr];
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
            buf ^= 1;
        }

        // sum(u^2) of this warp's part of the tile; the finalise adds the
        // partials in a fixed order
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
        if (lane == 0) mi.partials[static_cast<int64_t>(local) * kMomPartials + warp] = ss;
    }
}

constexpr int kFinThreads = 256;

__global__ void __launch_bounds__(kFinThreads) norm_finalize_kernel(const __grid_constant__ MomentumArgs a) {
    __shared__ double red[kFinThreads / 32];
    const MatInfo& mi = a.infos[blockIdx.x];
    double s = 0.0;
    // A tile's partials are two 16-byte loads (the buffer starts on 256 bytes
    // and a tile's partials take 32).  They are added in fp32 in warp order,
    // then the tile sums in double: fp64 is slow on this part, so one
    // conversion and one add per tile.
    static_assert(kMomPartials == 8, "a tile's partials are read as two float4");
    const float4* p4 = reinterpret_cast<const float4*>(mi.partials);
    for (int i = threadIdx.x; i < mi.ntiles; i += kFinThreads) {
        const float4 x = p4[2 * i], y = p4[2 * i + 1];
        s += static_cast<double>(x.x + x.y + x.z + x.w + y.x + y.y + y.z + y.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
#pragma unroll
        for (int w = 0; w < kFinThreads / 32; ++w) tot += red[w];
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
    static PerDevice per_sm_per_device;
    int per_sm = 1;
    per_sm_per_device.get(dev, &per_sm, [](int* out) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, momentum_pack_kernel, kMomThreads, 0) != cudaSuccess ||
            n < 1)
            n = 1;
        *out = n;
        return cudaSuccess;
    });
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * per_sm;
    const int grid = static_cast<int>(a.total_tiles < cap ? a.total_tiles : cap);
    momentum_pack_kernel<<<grid, kMomThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const MomentumArgs& a, cudaStream_t s) {
    if (a.nslots <= 0) return cudaSuccess;
    norm_finalize_kernel<<<a.nslots, kFinThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dmuon
