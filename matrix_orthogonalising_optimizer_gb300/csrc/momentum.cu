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
// HBM-bound.  Matrices whose u has the gradient's own layout (bf16, not
// transposed, rows starting on 16 bytes) go through a flat pass: persistent
// blocks stream chunks of kMomChunk elements of G and M into a six-stage
// shared-memory ring with bulk asynchronous copies (cp.async.bulk, completion
// counted on the stage's mbarrier) while the block's threads update the
// current chunk from shared memory and store M' and u with 16-byte accesses;
// a chunk leaves one sum-of-squares partial per warp, the tile pass's layout.
// The other matrices go through the tile pass below, which jumps over the
// flat matrices' index ranges.
//
// Tile pass.  Persistent blocks walk the tiles of every matrix of the wave,
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

__device__ __forceinline__ void prefetch_l2(uint64_t addr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
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
        if (t >= end || t < begin) {
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
            if (nm.flat) {
                // streamed by the flat pass: continue at this block's first
                // index at or past the matrix's end
                t += (end - t + gridDim.x - 1) / gridDim.x * gridDim.x - gridDim.x;
                continue;
            }
            grad = a.grads[nm.gidx];
            mom = a.moms[nm.gidx];
        }
        const MatInfo& mi = a.infos[slot];
        const int local = static_cast<int>(t - begin);
        const int r0 = (local / mi.tiles_c) * T, c0 = (local % mi.tiles_c) * T;
        const int rows = mi.rows, cols = mi.cols;
        const int dt = mi.dtype;
        // L2 prefetch of this block's next tile in the same matrix (grad and
        // momentum rows): its loads then wait on L2, not HBM.  Thread tid
        // takes row tid / 4 of that tile; bit 1 picks the array, bit 0 the
        // first or the last 128-byte line of the row's segment (the last one
        // only where it is another line).
        if (t + gridDim.x < end) {
            const int l2 = static_cast<int>(t + gridDim.x - begin);
            const int pr = (l2 / mi.tiles_c) * T + tid / 4, pc = (l2 % mi.tiles_c) * T;
            if (pr < rows) {
                const int es = dt == ELEM_BF16 ? 2 : 4;
                const int64_t e0 = static_cast<int64_t>(pr) * cols + pc;
                const int64_t e1 = static_cast<int64_t>(pr) * cols + min(pc + T, cols) - 1;
                const char* arr = static_cast<const char*>((tid & 2) ? static_cast<const void*>(mom) : grad);
                const uint64_t first = reinterpret_cast<uint64_t>(arr + e0 * es);
                const uint64_t last = reinterpret_cast<uint64_t>(arr + e1 * es);
                if (!(tid & 1)) prefetch_l2(first);
                else if ((last >> 7) != (first >> 7)) prefetch_l2(last);
            }
        }
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
            // packed row = original column: a quad of threads per packed row,
            // thread q taking original rows 8q .. 8q + 7 and 32 + 8q .. 32 + 8q + 7,
            // so each store instruction covers whole sectors (rows 0 .. 31 of
            // the segment, then 32 .. 63) and the shared-memory reads hit 32
            // different banks
            const int xr = tid / 4, q = tid % 4;
            const int c = c0 + xr;
            if (c < cols) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int rr0 = 8 * q + 32 * h;
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = tile[buf][rr0 + e][xr];
                    const int r = r0 + rr0;
                    const int64_t base = static_cast<int64_t>(c) * mi.ldx + r;
                    if (r + 8 <= rows) {
                        store8(mi.x, base, mi.x_type, v);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (r + e < rows) st1(mi.x, base + e, mi.x_type, v[e]);
                    }
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

// ---------------------------------------------------------------- flat pass

constexpr int kFlatThreads = 256;
constexpr int kFlatStages = 6;
constexpr int kFlatPiece = kMomChunk * 2;  // 8 KB: one bf16 array's share of a chunk
constexpr int kFlatBlocksPerSm = 2;
constexpr uint64_t kWaitNs = 2000000000ull;  // bounded waits: about 2 s
static_assert(kMomChunk == 2 * 8 * kFlatThreads, "a thread updates two 8-element vectors of a chunk");

struct __align__(128) FlatSmem {
    uint8_t piece[kFlatStages][2][kFlatPiece];  // grad, momentum
    uint64_t full[kFlatStages];                 // both pieces landed (count 1 + bytes)
    uint64_t empty[kFlatStages];                // every warp has read the stage
};

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of the given parity; false (and DEV_TIMEOUT in
// the status word) after about 2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitNs) {
            atomicExch(status, DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Position (in the flat list) of the flat slot holding chunk c of the wave's
// flat index, at or after position `from`, whose matrix starts at or before
// c: that one if the next matrix starts past c, else a binary search.
__device__ __forceinline__ int find_flat(const MomentumArgs& a, int64_t c, int from) {
    int lo = from, hi = a.nflat - 1;
    if (lo < hi && a.infos[a.flat_slots[lo + 1]].flat_begin > c) return lo;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.infos[a.flat_slots[mid]].flat_begin <= c) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// One thread's view of the flat matrix it is working in: the record is
// re-read only when the chunk leaves the matrix.
struct FlatCursor {
    int pos = -1;  // position in the flat list (-1: none yet)
    int64_t begin = 0, end = 0, elems = 0;
    const __nv_bfloat16* grad = nullptr;
    __nv_bfloat16* mom = nullptr;
    __nv_bfloat16* x = nullptr;
    float* partials = nullptr;

    __device__ __forceinline__ void seek(const MomentumArgs& a, int64_t c) {
        if (c >= begin && c < end) return;
        // chunks come in increasing order: past this matrix, the next one on
        pos = find_flat(a, c, c >= end ? pos + 1 : 0);
        const MatInfo& mi = a.infos[a.flat_slots[pos]];
        begin = mi.flat_begin;
        end = begin + mi.ntiles;
        elems = static_cast<int64_t>(mi.rows) * mi.cols;
        grad = static_cast<const __nv_bfloat16*>(a.grads[mi.gidx]);
        mom = static_cast<__nv_bfloat16*>(a.moms[mi.gidx]);
        x = static_cast<__nv_bfloat16*>(mi.x);
        partials = mi.partials;
    }
};

// Thread 0: stream chunk c (if it is below c_end) into `stage`.  A chunk's
// bytes are a multiple of 16 (the matrix's element count is a multiple of 8).
__device__ __forceinline__ void flat_issue(const MomentumArgs& a, FlatSmem& S, FlatCursor& cur, int stage,
                                           int64_t c, int64_t c_end) {
    uint32_t bytes = 0;
    int64_t e0 = 0;
    if (c < c_end) {
        cur.seek(a, c);
        e0 = (c - cur.begin) * kMomChunk;
        bytes = static_cast<uint32_t>(min(static_cast<int64_t>(kMomChunk), cur.elems - e0) * 2);
    }
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(&S.full[stage])),
                 "r"(2 * bytes)
                 : "memory");
    if (bytes == 0) return;
    const void* src[2] = {cur.grad + e0, cur.mom + e0};
#pragma unroll
    for (int k = 0; k < 2; ++k)
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         saddr(S.piece[stage][k])),
                     "l"(reinterpret_cast<uint64_t>(src[k])), "r"(bytes), "r"(saddr(&S.full[stage]))
                     : "memory");
}

__global__ void __launch_bounds__(kFlatThreads, kFlatBlocksPerSm) momentum_flat_kernel(
    const __grid_constant__ MomentumArgs a) {
    extern __shared__ uint8_t smem_raw[];
    FlatSmem& S = *reinterpret_cast<FlatSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < kFlatStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&S.full[s])), "r"(1) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&S.empty[s])),
                         "r"(kFlatThreads / 32)
                         : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // a contiguous range of chunks per block: consecutive chunks mostly lie in
    // one matrix, so its record is looked up once
    const int64_t c_begin = a.flat_chunks * blockIdx.x / gridDim.x;
    const int64_t c_end = a.flat_chunks * (blockIdx.x + 1) / gridDim.x;
    FlatCursor issue_cur, cur;
    if (tid == 0)
        for (int s = 0; s < kFlatStages; ++s) flat_issue(a, S, issue_cur, s, c_begin + s, c_end);
    bool ok = true;
    int64_t it = 0;
    for (int64_t c = c_begin; c < c_end; ++c, ++it) {
        const int stage = static_cast<int>(it % kFlatStages);
        const uint32_t phase = static_cast<uint32_t>(it / kFlatStages) & 1u;
        if (!mbar_wait(&S.full[stage], phase, a.status)) {
            ok = false;
            break;
        }
        cur.seek(a, c);
        const int64_t local = c - cur.begin, e0 = local * kMomChunk;
        const int64_t nb = min(static_cast<int64_t>(kMomChunk), cur.elems - e0);
        float ss = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = tid * 8 + h * (kMomChunk / 2);
            if (e < nb) {
                float g[8], m[8], u[8];
                unpack8(*reinterpret_cast<const uint4*>(S.piece[stage][0] + 2 * e), g);
                unpack8(*reinterpret_cast<const uint4*>(S.piece[stage][1] + 2 * e), m);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    m[k] = fmaf(a.beta, m[k], g[k]);
                    u[k] = a.nesterov ? fmaf(a.beta, m[k], g[k]) : m[k];
                    ss = fmaf(u[k], u[k], ss);
                }
                store8(cur.mom, e0 + e, ELEM_BF16, m);
                store8(cur.x, e0 + e, ELEM_BF16, u);
            }
        }
        // the warp's partial of this chunk (elements 256 w .. and 2048 + 256 w ..)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
        if (lane == 0) cur.partials[local * kMomPartials + warp] = ss;
        __syncwarp();
        if (lane == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&S.empty[stage])) : "memory");
        if (tid == 0) {
            // every warp has read the stage: refill it
            if (!mbar_wait(&S.empty[stage], phase, a.status)) {
                ok = false;
                break;
            }
            flat_issue(a, S, issue_cur, stage, c + kFlatStages, c_end);
        }
    }
    if (tid == 0 && !ok) {
        // let copies already issued land before the block exits
        for (int s = 0; s < kFlatStages; ++s) {
            const int64_t k = it + ((s - static_cast<int>(it % kFlatStages)) + kFlatStages) % kFlatStages;
            mbar_wait(&S.full[s], static_cast<uint32_t>(k / kFlatStages) & 1u, a.status);
        }
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

cudaError_t launch_momentum_flat(const MomentumArgs& a, cudaStream_t s) {
    if (a.flat_chunks <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = sizeof(FlatSmem) + 128;
    static PerDevice attr_per_device;
    int unused = 0;
    cudaError_t e = attr_per_device.get(dev, &unused, [&](int* out) {
        *out = 1;
        return cudaFuncSetAttribute(momentum_flat_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem));
    });
    if (e != cudaSuccess) return e;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * kFlatBlocksPerSm;
    const int grid = static_cast<int>(a.flat_chunks < cap ? a.flat_chunks : cap);
    momentum_flat_kernel<<<grid, kFlatThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const MomentumArgs& a, cudaStream_t s) {
    if (a.nslots <= 0) return cudaSuccess;
    norm_finalize_kernel<<<a.nslots, kFinThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dmuon
