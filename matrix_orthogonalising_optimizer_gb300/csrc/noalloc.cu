// Muon step for one small matrix that allocates no device memory.
//
// dmuon_step needs a caller-provided workspace.  Some callers cannot provide
// one: their device memory is entirely reserved by another allocator (a
// framework's caching pool that owns the GPU), or they run under a fixed
// memory budget and may not grow device allocations once training started.
// This entry point keeps its scratch in a file-scope __device__ array instead,
// so it needs neither cudaMalloc nor a workspace; the caller still passes the
// parameter, gradient and momentum.
//
// The scratch is one static array of kScratchFloats floats (1.3125 MiB), held
// by every GPU that loads the library until the process exits.  It bounds the
// matrices this entry point accepts: min(rows, cols) <= 128 and
// rows * cols <= 2^18.  All calls on a device share the array, and a call
// leaves its contents behind; every element a call reads it has written first
// in the same call, so nothing needs clearing, but two calls that overlap on
// the GPU (different streams, no ordering between them) race on the array.
//
// The arithmetic is the fp32 validation mode of dmuon_step on a Gram bucket:
// Nesterov momentum, Frobenius normalisation, Gram-space Newton-Schulz with
// the quintic (3.4445, -4.7750, 2.0315), eps = 1e-7, the aspect scale and
// decoupled weight decay, all products in fp32 FFMA, in a single thread block
// (no inter-block synchronisation).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {
void set_last_error(const std::string& msg);
}

namespace {

constexpr int kMaxM = 128;
constexpr int64_t kMaxElems = 1 << 18;
constexpr int64_t kMM = static_cast<int64_t>(kMaxM) * kMaxM;
constexpr int64_t kScratchFloats = kMaxElems + 5 * kMM;  // X, then R, P, Q0, Q1, RP
constexpr int kThreads = 512;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

struct SmallArgs {
    void* w;
    const void* grad;
    void* mom;
    float* scratch;
    int rows, cols, m, n, transposed, dtype, steps;
    float beta, decay, lrs, a, b, c, eps;
};

__device__ __forceinline__ float ld(const void* p, int64_t i, int t) {
    return t == dmuon::ELEM_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                                 : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st(void* p, int64_t i, int t, float v) {
    if (t == dmuon::ELEM_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else static_cast<float*>(p)[i] = v;
}

// Symmetric product out = f(A B) over the lower triangle, mirrored:
// out = alpha * (c_acc * (A B) + c_diag * I + c_aux * aux).  A, B, aux are
// m x m row-major with leading dimension m.
__device__ void sym_product(float* out, float* out2, const float* A, const float* B, const float* aux, int m,
                            float alpha, float c_acc, float c_diag, float c_aux) {
    for (int e = threadIdx.x; e < m * m; e += blockDim.x) {
        const int i = e / m, j = e % m;
        if (j > i) continue;
        float acc = 0.0f;
        for (int l = 0; l < m; ++l) acc = fmaf(A[i * m + l], B[l * m + j], acc);
        float t = c_acc * acc;
        if (i == j) t += c_diag;
        if (aux) t = fmaf(c_aux, aux[i * m + j], t);
        const float v = alpha * t;
        out[i * m + j] = v;
        out[j * m + i] = v;
        if (out2) {
            out2[i * m + j] = v;
            out2[j * m + i] = v;
        }
    }
}

__global__ void __launch_bounds__(kThreads) muon_small_kernel(const __grid_constant__ SmallArgs s) {
    __shared__ double red[kThreads / 32];
    __shared__ float inv_sh;
    const int m = s.m, n = s.n;
    float* X = s.scratch;
    float* R = X + kMaxElems;
    float* P = R + kMM;
    float* Q[2] = {P + kMM, P + 2 * kMM};
    float* RP = P + 3 * kMM;

    // momentum, Nesterov direction u packed as X (m x n), sum of squares
    const int64_t total = static_cast<int64_t>(s.rows) * s.cols;
    double ss = 0.0;
    for (int64_t idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int r = static_cast<int>(idx / s.cols), c = static_cast<int>(idx % s.cols);
        const float g = ld(s.grad, idx, s.dtype);
        const float mo = fmaf(s.beta, ld(s.mom, idx, s.dtype), g);
        st(s.mom, idx, s.dtype, mo);
        const float u = fmaf(s.beta, mo, g);
        ss += static_cast<double>(u) * u;
        if (!s.transposed) X[static_cast<int64_t>(r) * n + c] = u;
        else X[static_cast<int64_t>(c) * n + r] = u;
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
        inv_sh = static_cast<float>(1.0 / (sqrt(tot) + static_cast<double>(s.eps)));
    }
    __syncthreads();
    const float inv = inv_sh;

    // R0 = inv^2 X X^T
    for (int e = threadIdx.x; e < m * m; e += blockDim.x) {
        const int i = e / m, j = e % m;
        if (j > i) continue;
        float acc = 0.0f;
        for (int k = 0; k < n; ++k) acc = fmaf(X[static_cast<int64_t>(i) * n + k], X[static_cast<int64_t>(j) * n + k], acc);
        const float v = (inv * inv) * acc;
        R[i * m + j] = v;
        R[j * m + i] = v;
    }
    __syncthreads();

    for (int k = 0; k < s.steps; ++k) {
        // P = aI + bR + cR^2 (and Q_0 = P)
        sym_product(P, k == 0 ? Q[0] : nullptr, R, R, R, m, 1.0f, s.c, s.a, s.b);
        __syncthreads();
        if (k >= 1) sym_product(Q[k % 2], nullptr, P, Q[(k - 1) % 2], nullptr, m, 1.0f, 1.0f, 0.0f, 0.0f);
        if (k < s.steps - 1) sym_product(RP, nullptr, R, P, nullptr, m, 1.0f, 1.0f, 0.0f, 0.0f);
        __syncthreads();
        if (k < s.steps - 1) {
            sym_product(R, nullptr, P, RP, nullptr, m, 1.0f, 1.0f, 0.0f, 0.0f);
            __syncthreads();
        }
    }

    // W = decay W - lr s (inv Q X) in W's own orientation
    const float* Qf = Q[(s.steps - 1) % 2];
    for (int64_t e = threadIdx.x; e < static_cast<int64_t>(m) * n; e += blockDim.x) {
        const int i = static_cast<int>(e / n), j = static_cast<int>(e % n);
        float acc = 0.0f;
        for (int l = 0; l < m; ++l) acc = fmaf(Qf[i * m + l], X[static_cast<int64_t>(l) * n + j], acc);
        const float v = inv * acc;
        const int64_t wi = s.transposed ? static_cast<int64_t>(j) * s.cols + i : static_cast<int64_t>(i) * s.cols + j;
        st(s.w, wi, s.dtype, fmaf(-s.lrs, v, s.decay * ld(s.w, wi, s.dtype)));
    }
}

// The device address of the scratch is looked up once per CUDA context and
// cached with the context's unique id: after the context is destroyed (for
// example by cudaDeviceReset) and a new one is created, the module is loaded
// again and the array may sit elsewhere, so a new id triggers a new lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_mu;
struct ScratchEntry {
    unsigned long long ctx_id;
    float* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

// Unique id of the calling thread's current context (0 if none is current).
bool current_context_id(unsigned long long* id) {
    if (!g_ctx_current || !g_ctx_id) {
        void* f0 = nullptr;
        void* f1 = nullptr;
        cudaDriverEntryPointQueryResult q0, q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 4000, cudaEnableDefault, &q0) != cudaSuccess ||
            q0 != cudaDriverEntryPointSuccess || !f0 ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || !f1)
            return false;
        g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f0);
        g_ctx_id = reinterpret_cast<CtxGetIdFn>(f1);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
    *id = 0;
    if (!ctx) return true;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int dmuon_step_noalloc(void* param, const void* grad, void* momentum, int64_t rows, int64_t cols,
                                  int32_t dtype, float lr, float beta, float wd, int32_t ns_steps, void* stream) {
    using dmuon::set_last_error;
    if (!param || !grad || !momentum) {
        set_last_error("dmuon_step_noalloc: NULL tensor pointer");
        return DMUON_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(param) | reinterpret_cast<uintptr_t>(grad) |
         reinterpret_cast<uintptr_t>(momentum)) & 15) {
        set_last_error("dmuon_step_noalloc: tensors must start on 16-byte boundaries");
        return DMUON_ERR_ALIGN;
    }
    if (dtype != DMUON_BF16 && dtype != DMUON_FP32) {
        set_last_error("dmuon_step_noalloc: unknown dtype");
        return DMUON_ERR_UNSUPPORTED_DTYPE;
    }
    // each side is bounded before the product, so rows * cols cannot overflow
    if (rows < 1 || cols < 1 || rows > kMaxElems || cols > kMaxElems || (rows < cols ? rows : cols) > kMaxM ||
        rows * cols > kMaxElems) {
        set_last_error("dmuon_step_noalloc: " + std::to_string(rows) + "x" + std::to_string(cols) +
                       " exceeds the static scratch: need min(rows, cols) <= 128 and rows*cols <= 262144");
        return DMUON_ERR_INVALID_ARG;
    }
    if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(wd) || lr < 0.0f || wd < 0.0f ||
        beta < 0.0f || beta >= 1.0f || ns_steps < 1 || ns_steps > DMUON_MAX_NS_STEPS) {
        set_last_error("dmuon_step_noalloc: need finite lr >= 0, wd >= 0, 0 <= beta < 1, 1 <= ns_steps <= 16");
        return DMUON_ERR_INVALID_ARG;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        set_last_error("dmuon_step_noalloc: no usable current device");
        return DMUON_ERR_CUDA;
    }
    float* scratch = nullptr;
    {
        // once per device and context, with that device current: the device
        // address of the static scratch (the host-side symbol is not a device
        // address)
        std::lock_guard<std::mutex> lock(g_mu);
        unsigned long long id = 0;
        if (!current_context_id(&id)) {
            set_last_error("dmuon_step_noalloc: cannot query the current CUDA context");
            return DMUON_ERR_CUDA;
        }
        if (id == 0 || !g_scratch[dev].ptr || g_scratch[dev].ctx_id != id) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                set_last_error(std::string("dmuon_step_noalloc: cudaGetSymbolAddress failed: ") +
                               cudaGetErrorString(e));
                return DMUON_ERR_CUDA;
            }
            // the lookup makes the device's primary context current if none was
            if (id == 0 && !current_context_id(&id)) {
                set_last_error("dmuon_step_noalloc: cannot query the current CUDA context");
                return DMUON_ERR_CUDA;
            }
            g_scratch[dev].ptr = static_cast<float*>(p);
            g_scratch[dev].ctx_id = id;
        }
        scratch = g_scratch[dev].ptr;
    }
    SmallArgs a;
    a.w = param;
    a.grad = grad;
    a.mom = momentum;
    a.scratch = scratch;
    a.rows = static_cast<int>(rows);
    a.cols = static_cast<int>(cols);
    a.transposed = rows > cols ? 1 : 0;
    a.m = static_cast<int>(rows < cols ? rows : cols);
    a.n = static_cast<int>(rows < cols ? cols : rows);
    a.dtype = dtype == DMUON_BF16 ? dmuon::ELEM_BF16 : dmuon::ELEM_F32;
    a.steps = ns_steps;
    a.beta = beta;
    a.decay = 1.0f - lr * wd;
    a.lrs = lr * static_cast<float>(std::sqrt(std::max(1.0, static_cast<double>(rows) / static_cast<double>(cols))));
    a.a = 3.4445f;
    a.b = -4.7750f;
    a.c = 2.0315f;
    a.eps = 1e-7f;
    muon_small_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_error(std::string("dmuon_step_noalloc: launch failed: ") + cudaGetErrorString(e));
        return DMUON_ERR_CUDA;
    }
    return DMUON_OK;
}
