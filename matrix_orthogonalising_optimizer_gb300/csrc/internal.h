// Internal structures shared by the planner, the runtime and the kernels of
// the batched Gram-space Newton-Schulz Muon step.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

namespace dmuon {

// ---------------------------------------------------------------- constants

// tcgen05 GEMM tile: 128 rows (TMEM lanes) x 256 columns, 128-byte K slabs.
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcSlabBytes = 128;  // one K slab row = one 128-byte swizzle row
constexpr int kTcStages = 6;
constexpr int kTcThreads = 384;    // warp 0 TMA, warp 1 MMA + TMEM, warps 2-3 idle, warps 4-11 epilogue
constexpr int kTcPair = 2;         // CTAs per cluster running one cta_group::2 MMA

// fp32 FFMA GEMM tile
constexpr int kSimtBM = 64;
constexpr int kSimtBN = 64;
constexpr int kSimtThreads = 256;

// momentum / pack tile over the original (rows x cols) matrix
constexpr int kMomTile = 64;
constexpr int kMomThreads = 256;
constexpr int kMomPartials = kMomThreads / 32;  // sum-of-squares partials per momentum tile (one per warp)
// flat momentum pass: a chunk of a matrix stored row after row, as many
// elements as a tile, streamed through shared memory by bulk copies
constexpr int kMomChunk = kMomTile * kMomTile;

constexpr int kMaxGroupsPerLaunch = 96;
constexpr int kMaxLaunchesPerWave = 1024;  // tile counters in the workspace, cleared per wave

enum ElemType : int32_t { ELEM_BF16 = 0, ELEM_F32 = 1 };
enum EpiMode : int32_t { EPI_STORE = 0, EPI_UPDATE = 1 };
enum AlphaSel : int32_t { ALPHA_ONE = 0, ALPHA_INV = 1, ALPHA_INV2 = 2 };

// Device status word values (first int32 of the workspace).
enum DevStatus : int32_t { DEV_OK = 0, DEV_TIMEOUT = 1 };

// ---------------------------------------------------------------- tables

// Per matrix of the plan, in bucket order ("slot").
struct MatInfo {
    void* x;            // packed u: m x ldx, row-major, transposed for tall matrices
    float* partials;    // sum-of-squares partials, kMomPartials per momentum tile
    int64_t ldx;        // elements
    int64_t tile_begin; // first momentum tile of this slot inside its wave
    int64_t gidx;       // index of the matrix in the caller's arrays
    int32_t rows, cols; // original shape
    int32_t tiles_c;    // momentum tiles along cols
    int32_t ntiles;     // momentum tiles of this matrix
    int32_t transposed; // rows > cols
    int32_t dtype;      // storage dtype of W, grad, momentum (ElemType)
    int32_t x_type;     // ElemType of the packed u
    float scale;        // update shape scale s
    int32_t flat;       // bf16, not transposed, cols a multiple of 8: u has the
                        // gradient's layout and the momentum pass streams the
                        // matrix as chunks of kMomChunk elements (ntiles counts
                        // chunks; tile_begin .. + ntiles is skipped by the tile pass)
    int32_t pad;
    int64_t flat_begin; // first chunk of this matrix among the wave's flat matrices
};

struct SlotScalars {
    float inv;   // 1 / (||u||_F + eps)
    float inv2;  // inv^2
};

// One batched product D[mat] = A[mat] (M x K) * B[mat] (K x N) with a fused
// epilogue.  A is K-major (row-major M x K).  The B operand is K-major (stored
// N x K) or MN-major (stored K x N).  Built on the host, read by the kernels.
struct GemmGroup {
    CUtensorMap tma_a;      // tcgen05 path: A as {K, M, batch}
    CUtensorMap tma_b;      // K-major {K, N, batch} or MN-major {N, K, batch}
    // raw views (fp32 FFMA path)
    const void* a;
    const void* b;
    int64_t a_bs, b_bs;     // batch strides, elements
    int32_t lda, ldb;
    int32_t a_type, b_type; // ElemType
    int32_t M, N, K, batch;
    int32_t b_mn_major;
    // K split into segments of kseg elements (a multiple of the 64-deep slab;
    // 0 = one segment): K slab j of segment t reads A at segment t % 2 and B
    // at segment t / 2 of their rows.  With operands stored as [hi | lo]
    // (bf16 x = hi + lo) and K = 3 kseg this accumulates hi*hi + lo*hi +
    // hi*lo; with K = 2 kseg and a plain B it accumulates (hi + lo) * B.
    int32_t kseg;
    int32_t sym;            // symmetric D: lower-triangle tiles, mirrored stores
    int32_t tiles_m, tiles_n, tiles_per_mat;
    // tcgen05 symmetric groups with m <= 128: matrices per 256 x 256 pair tile
    // (2 for m <= 128, 4 for m <= 64), laid block-diagonally -- CTA rank r
    // loads matrices mat + r pack/2 .. as its 128 rows of A and B, and block
    // (i, i) of the accumulator is matrix mat + i's product; 1 otherwise
    int32_t pack;
    int32_t ntiles;         // tiles of the whole group: tiles_per_mat * batch, or batch / pack rounded up
    int32_t slot_base;      // slot of batch entry 0
    // epilogue: v = alpha * (c_acc*acc + c_diag*[r==c] + c_aux*aux[r][c])
    int32_t mode;           // EpiMode
    int32_t alpha_sel;      // AlphaSel
    float c_acc, c_diag, c_aux;
    int32_t aux_type;       // ElemType
    int32_t aux_sym;        // aux is bitwise symmetric: read aux[c][r] (coalesced)
    int32_t aux_ld;
    const void* aux;
    int64_t aux_bs;
    // up to three stored copies of v (EPI_STORE), each with its own dtype
    void* out[3];
    int64_t out_bs[3];
    int32_t out_ld[3];
    int32_t out_type[3];
    int32_t out_mirror[3];  // symmetric D: also store the upper triangle of this output
    int32_t out_lo[3];      // bf16 output stored split: hi = bf16(v) at column c, lo = bf16(v - hi)
                            // at column out_lo + c of the same row (0 = plain)
};

// Passed by value to every GEMM launch.
struct LaunchList {
    const GemmGroup* groups;                 // device table base
    const MatInfo* infos;                    // device, indexed by slot
    const SlotScalars* scalars;              // device, indexed by slot
    void* const* params;                     // device, indexed by gidx
    int32_t* status;                         // device status word
    int32_t* counter;                        // tile counter of this launch (zero at launch)
    float lr, decay;                         // update: W = decay*W - lr*s*v
    int32_t n;                               // groups in this launch
    int32_t total_tiles;
    int32_t has_split;                       // some group stores split outputs (tcgen05 kernel instance)
    int32_t epi_sets;                        // tcgen05 epilogue: alternate tiles per warp set (set at launch)
    int32_t update;                          // the launch's products apply the W update (else they store)
    int32_t idx[kMaxGroupsPerLaunch];        // indices into `groups`
    int32_t begin[kMaxGroupsPerLaunch + 1];  // tile prefix
};

struct MomentumArgs {
    const MatInfo* infos;    // slots of the wave, first one at infos[0]
    SlotScalars* scalars;    // same slots
    const void* const* grads;
    void* const* moms;
    const int32_t* flat_slots;  // the wave's flat slots (relative to infos), ascending
    int32_t* status;         // device status word (a bounded wait that gave up)
    int32_t nslots;
    int32_t nflat;
    int64_t total_tiles;
    int64_t flat_chunks;
    float beta;
    int32_t nesterov;
    float eps;
};

// ---------------------------------------------------------------- per device

constexpr int kMaxCachedDevices = 64;

// A launch setting computed once per device with that device current (an
// occupancy figure, or a kernel attribute that must be set before the first
// launch on each device).  Thread-safe; devices beyond kMaxCachedDevices are
// computed on every call.
class PerDevice {
  public:
    template <typename F>
    cudaError_t get(int dev, int* out, F&& compute) {
        if (dev < 0 || dev >= kMaxCachedDevices) return compute(out);
        std::lock_guard<std::mutex> lock(mu_);
        if (!done_[dev]) {
            int v = 0;
            const cudaError_t e = compute(&v);
            if (e != cudaSuccess) return e;
            val_[dev] = v;
            done_[dev] = true;
        }
        *out = val_[dev];
        return cudaSuccess;
    }

  private:
    std::mutex mu_;
    int val_[kMaxCachedDevices] = {};
    bool done_[kMaxCachedDevices] = {};
};

// ---------------------------------------------------------------- launchers

cudaError_t launch_momentum_pack(const MomentumArgs& a, cudaStream_t s);
cudaError_t launch_momentum_flat(const MomentumArgs& a, cudaStream_t s);
cudaError_t launch_norm_finalize(const MomentumArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc(const LaunchList& l, int num_sms, cudaStream_t s);
cudaError_t launch_gemm_simt(const LaunchList& l, cudaStream_t s);
size_t gemm_tc_smem_bytes();

}  // namespace dmuon
