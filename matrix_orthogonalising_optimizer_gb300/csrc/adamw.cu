// Multi-tensor AdamW step: the element-wise optimizer the DMuon pages measure
// the Muon step against ("+2 % step time over AdamW", DMuon technical summary
// on gist.science, section 4), run on the same tensors so the two optimizer
// steps can be timed side by side on one GPU.
//
// Per element, in fp32 from the stored values (decoupled weight decay with
// bias correction, the published AdamW):
//   m  = beta1*m + (1-beta1)*g
//   v  = beta2*v + (1-beta2)*g^2
//   W  = (1 - lr*wd)*W - (lr / (1-beta1^t)) * m / (sqrt(v) / sqrt(1-beta2^t) + eps)
// W, m and v are stored back in the tensor's dtype (round to nearest even).
//
// HBM-bound: 14 bytes per bf16 element (read W, g, m, v; write W, m, v), 28
// per fp32 element.  Each tensor is cut into chunks of 32 KB of input (8 KB of
// each of W, g, m, v: 4096 bf16 or 2048 fp32 elements).  Persistent blocks
// (two per SM) walk the chunks of every tensor of a launch through a
// three-stage shared-memory ring: one thread streams a chunk's four 8 KB
// pieces in with bulk asynchronous copies (cp.async.bulk, completion counted
// on the stage's mbarrier) two chunks ahead, while the 256 threads update the
// current chunk from shared memory and store W, m, v straight to HBM with
// 16-byte accesses.  That keeps 6 chunks (192 KB) of loads in flight per SM
// with few registers.  A tensor's last n mod 8 elements (not a multiple of 16
// bytes) are updated from global memory by the block holding its last chunk.
// The tensor table travels as the kernel parameter (up to kAdamPerLaunch
// tensors per launch), so the call needs no device allocation.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <string>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {
void set_last_error(const std::string& msg);
}

namespace {

constexpr int kAdamPerLaunch = 256;
constexpr int kAdamThreads = 256;
constexpr int kAdamStages = 3;
constexpr int kPieceBytes = 8192;               // one array's share of a chunk
constexpr int kBlocksPerSm = 2;
constexpr uint64_t kWaitNs = 2000000000ull;     // bounded waits: about 2 s

struct AdamTensor {
    void* w;
    const void* g;
    void* m;
    void* v;
    int64_t n;            // elements
    int64_t bulk;         // n rounded down to a multiple of 8: moved by bulk copies
    int64_t chunk_begin;  // first chunk of this tensor in the launch
    int32_t dtype;
    int32_t chunk_elems;  // kPieceBytes / element size
};

struct AdamArgs {
    AdamTensor t[kAdamPerLaunch];
    int32_t count;
    int32_t pad;
    int64_t total_chunks;
    float decay;       // 1 - lr*wd
    float beta1, beta2, omb1, omb2;
    float step_size;   // lr / (1 - beta1^t)
    float inv_bc2_sqrt;  // 1 / sqrt(1 - beta2^t)
    float eps;
};

struct __align__(128) AdamSmem {
    uint8_t piece[kAdamStages][4][kPieceBytes];
    uint64_t full[kAdamStages];
    uint64_t empty[kAdamStages];
};

// set by a wait that gave up; read and cleared by dmuon_adamw_status
__device__ int32_t g_adamw_status = 0;

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

// Bounded wait for the phase of the given parity; false (and the status
// flag) after about 2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitNs) {
            atomicExch(&g_adamw_status, 1);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(saddr(bar))
                 : "memory");
}

__device__ __forceinline__ int find_tensor(const AdamArgs& a, int64_t c) {
    int lo = 0, hi = a.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.t[mid].chunk_begin <= c) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float ld1(const void* p, int64_t i, int32_t dt) {
    return dt == dmuon::ELEM_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                                  : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st1(void* p, int64_t i, int32_t dt, float x) {
    if (dt == dmuon::ELEM_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
    else static_cast<float*>(p)[i] = x;
}

// The update's square root and reciprocal use the approximate PTX forms
// (relative error about 2^-23 each): the update then errs by a few fp32 ulps
// of itself, below the rounding of every stored bf16 value, and the kernel
// stays a memory-bound stream instead of an instruction-bound one.
__device__ __forceinline__ float sqrt_approx(float x) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void adam_elem(const AdamArgs& a, float& w, float g, float& m, float& v) {
    m = fmaf(a.beta1, m, a.omb1 * g);
    v = fmaf(a.beta2, v, a.omb2 * g * g);
    const float denom = fmaf(sqrt_approx(v), a.inv_bc2_sqrt, a.eps);
    w = fmaf(-a.step_size, m * rcp_approx(denom), a.decay * w);
}

// 16 bytes at byte offset `off` of a piece: 8 bf16 or 4 fp32 values
template <int N>
__device__ __forceinline__ void unpack(const uint4& q, float (&x)[N]) {
    if constexpr (N == 8) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(h[k]);
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    } else {
        x[0] = __uint_as_float(q.x);
        x[1] = __uint_as_float(q.y);
        x[2] = __uint_as_float(q.z);
        x[3] = __uint_as_float(q.w);
    }
}

template <int N>
__device__ __forceinline__ uint4 pack(const float (&x)[N]) {
    uint4 q;
    if constexpr (N == 8) {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
    } else {
        q = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
    return q;
}

// One 16-byte vector (N elements) of a chunk held in shared memory.
template <int N>
__device__ __forceinline__ void update_vec(const AdamArgs& a, const AdamTensor& T, uint8_t (*piece)[kPieceBytes],
                                           int off, int64_t e0) {
    float w[N], g[N], m[N], v[N];
    unpack<N>(*reinterpret_cast<const uint4*>(piece[0] + off), w);
    unpack<N>(*reinterpret_cast<const uint4*>(piece[1] + off), g);
    unpack<N>(*reinterpret_cast<const uint4*>(piece[2] + off), m);
    unpack<N>(*reinterpret_cast<const uint4*>(piece[3] + off), v);
#pragma unroll
    for (int k = 0; k < N; ++k) adam_elem(a, w[k], g[k], m[k], v[k]);
    const int64_t byte = e0 * (N == 8 ? 2 : 4);
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(T.w) + byte) = pack<N>(w);
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(T.m) + byte) = pack<N>(m);
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(T.v) + byte) = pack<N>(v);
}

// Thread 0: stream chunk `c` (if it exists) into `stage`.
__device__ __forceinline__ void issue_chunk(const AdamArgs& a, AdamSmem& S, int stage, int64_t c) {
    uint32_t bytes = 0;
    const AdamTensor* T = nullptr;
    int64_t e0 = 0;
    if (c < a.total_chunks) {
        T = &a.t[find_tensor(a, c)];
        e0 = (c - T->chunk_begin) * T->chunk_elems;
        const int64_t e1 = min(e0 + T->chunk_elems, T->bulk);
        const int es = T->dtype == dmuon::ELEM_BF16 ? 2 : 4;
        bytes = e1 > e0 ? static_cast<uint32_t>((e1 - e0) * es) : 0u;
    }
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(&S.full[stage])),
                 "r"(4 * bytes)
                 : "memory");
    if (bytes == 0) return;
    const int es = T->dtype == dmuon::ELEM_BF16 ? 2 : 4;
    const void* src[4] = {T->w, T->g, T->m, T->v};
#pragma unroll
    for (int k = 0; k < 4; ++k)
        bulk_load(S.piece[stage][k], static_cast<const uint8_t*>(src[k]) + e0 * es, bytes, &S.full[stage]);
}

__global__ void __launch_bounds__(kAdamThreads, kBlocksPerSm) adamw_kernel(const __grid_constant__ AdamArgs a) {
    extern __shared__ uint8_t smem_raw[];
    AdamSmem& S = *reinterpret_cast<AdamSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kAdamStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&S.full[s])), "r"(1) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&S.empty[s])),
                         "r"(kAdamThreads / 32)
                         : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t first = blockIdx.x, stride = gridDim.x;
    if (tid == 0)
        for (int s = 0; s < kAdamStages; ++s) issue_chunk(a, S, s, first + s * stride);
    bool ok = true;
    int64_t it = 0;
    for (int64_t c = first; c < a.total_chunks && ok; c += stride, ++it) {
        const int stage = static_cast<int>(it % kAdamStages);
        const uint32_t phase = static_cast<uint32_t>(it / kAdamStages) & 1u;
        if (!mbar_wait(&S.full[stage], phase)) {
            ok = false;
            break;
        }
        const AdamTensor& T = a.t[find_tensor(a, c)];
        const int64_t e0 = (c - T.chunk_begin) * T.chunk_elems;
        const int64_t nb = min(static_cast<int64_t>(T.chunk_elems), max(T.bulk - e0, int64_t(0)));  // staged
        if (T.dtype == dmuon::ELEM_BF16) {
            for (int e = tid * 8; e < nb; e += kAdamThreads * 8) update_vec<8>(a, T, S.piece[stage], e * 2, e0 + e);
        } else {
            for (int e = tid * 4; e < nb; e += kAdamThreads * 4) update_vec<4>(a, T, S.piece[stage], e * 4, e0 + e);
        }
        // the tensor's tail beyond its last whole 16 bytes, straight from HBM
        if (e0 + T.chunk_elems >= T.n) {
            const int64_t i = T.bulk + tid;
            if (i < T.n) {
                float w = ld1(T.w, i, T.dtype), m = ld1(T.m, i, T.dtype), v = ld1(T.v, i, T.dtype);
                adam_elem(a, w, ld1(T.g, i, T.dtype), m, v);
                st1(T.w, i, T.dtype, w);
                st1(T.m, i, T.dtype, m);
                st1(T.v, i, T.dtype, v);
            }
        }
        __syncwarp();
        if (lane == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&S.empty[stage])) : "memory");
        if (tid == 0) {
            // every warp has read the stage: refill it
            if (!mbar_wait(&S.empty[stage], phase)) {
                ok = false;
                break;
            }
            issue_chunk(a, S, stage, c + kAdamStages * stride);
        }
    }
    if (tid == 0 && !ok) {
        // let copies already issued land before the block exits
        for (int s = 0; s < kAdamStages; ++s) {
            const int64_t k = it + ((s - static_cast<int>(it % kAdamStages)) + kAdamStages) % kAdamStages;
            mbar_wait(&S.full[s], static_cast<uint32_t>(k / kAdamStages) & 1u);
        }
    }
}

int fail(int code, const std::string& msg) {
    dmuon::set_last_error(msg);
    return code;
}

}  // namespace

extern "C" int dmuon_adamw_step(void* const* params, const void* const* grads, void* const* exp_avgs,
                                void* const* exp_avg_sqs, const int64_t* numels, const int32_t* dtypes, int64_t count,
                                float lr, float beta1, float beta2, float eps, float wd, int64_t step, void* stream) {
    if (count < 0 || (count > 0 && (!params || !grads || !exp_avgs || !exp_avg_sqs || !numels || !dtypes)))
        return fail(DMUON_ERR_INVALID_ARG, "dmuon_adamw_step: bad count or NULL array");
    if (step < 1 || !(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) || !(eps > 0.0f) ||
        !std::isfinite(lr) || !std::isfinite(wd))
        return fail(DMUON_ERR_INVALID_ARG, "dmuon_adamw_step: step must be >= 1, betas in [0, 1), eps > 0");
    for (int64_t i = 0; i < count; ++i) {
        if (numels[i] < 0) return fail(DMUON_ERR_INVALID_ARG, "dmuon_adamw_step: negative numel");
        if (dtypes[i] != DMUON_BF16 && dtypes[i] != DMUON_FP32)
            return fail(DMUON_ERR_UNSUPPORTED_DTYPE, "dmuon_adamw_step: dtype must be DMUON_BF16 or DMUON_FP32");
        if (numels[i] == 0) continue;
        const void* ptrs[4] = {params[i], grads[i], exp_avgs[i], exp_avg_sqs[i]};
        for (const void* p : ptrs)
            if (!p || (reinterpret_cast<uintptr_t>(p) & 15) != 0)
                return fail(DMUON_ERR_ALIGN, "dmuon_adamw_step: tensor " + std::to_string(i) +
                                                 " is NULL or not 16-byte aligned");
    }
    if (std::all_of(numels, numels + count, [](int64_t n) { return n == 0; })) return DMUON_OK;  // no work
    // bias corrections in double, as the formula states them
    const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(step));
    const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(step));
    AdamArgs a;
    a.decay = static_cast<float>(1.0 - static_cast<double>(lr) * wd);
    a.beta1 = beta1;
    a.beta2 = beta2;
    a.omb1 = static_cast<float>(1.0 - beta1);
    a.omb2 = static_cast<float>(1.0 - beta2);
    a.step_size = static_cast<float>(lr / bc1);
    a.inv_bc2_sqrt = static_cast<float>(1.0 / std::sqrt(bc2));
    a.eps = eps;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return fail(DMUON_ERR_CUDA, "dmuon_adamw_step: no CUDA device");
    const size_t smem = sizeof(AdamSmem) + 128;
    // the shared-memory attribute, once per device with that device current
    static dmuon::PerDevice configured;
    int unused = 0;
    const cudaError_t ce = configured.get(dev, &unused, [&](int*) {
        return cudaFuncSetAttribute(adamw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    });
    if (ce != cudaSuccess) return fail(DMUON_ERR_CUDA, std::string("dmuon_adamw_step: ") + cudaGetErrorString(ce));
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t i = 0;
    while (i < count) {
        a.count = 0;
        a.total_chunks = 0;
        for (; i < count && a.count < kAdamPerLaunch; ++i) {
            if (numels[i] == 0) continue;
            AdamTensor& t = a.t[a.count++];
            t.w = params[i];
            t.g = grads[i];
            t.m = exp_avgs[i];
            t.v = exp_avg_sqs[i];
            t.n = numels[i];
            t.bulk = numels[i] & ~int64_t(7);
            t.dtype = dtypes[i];
            t.chunk_elems = kPieceBytes / (dtypes[i] == DMUON_BF16 ? 2 : 4);
            t.chunk_begin = a.total_chunks;
            a.total_chunks += (numels[i] + t.chunk_elems - 1) / t.chunk_elems;
        }
        if (a.count == 0) continue;
        const int64_t cap = static_cast<int64_t>(sms) * kBlocksPerSm;
        const int grid = static_cast<int>(std::min<int64_t>(a.total_chunks, cap));
        adamw_kernel<<<grid, kAdamThreads, smem, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return fail(DMUON_ERR_CUDA, std::string("dmuon_adamw_step: launch failed: ") + cudaGetErrorString(e));
    }
    return DMUON_OK;
}

extern "C" int dmuon_adamw_status(void) {
    int32_t v = 0;
    const int32_t zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_adamw_status, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_adamw_status, &zero, sizeof(zero)) != cudaSuccess)
        return fail(DMUON_ERR_CUDA, "dmuon_adamw_status: cannot read the status flag");
    return v ? DMUON_ERR_DEVICE_TIMEOUT : DMUON_OK;
}
