// Persistent batched GEMM on the 5th-generation tensor cores (sm_103a).
//
// The products of the Gram-space Newton-Schulz step (DMuon technical summary
// on gist.science, section 2.2): the Gram matrix X X^T formed SYRK-style
// (lower-triangle tiles only, mirrored in the epilogue), the m x m polynomial
// products -- all symmetric, so the same triangular schedule applies -- and
// the final Q X0 product fused with the Muon update.  Matrices of one shape
// bucket are batched as the third TMA coordinate, and one launch covers every
// group (bucket x product) of a phase, so small matrices share the machine
// (section 2.2 "batching").
//
// Layout: clusters of two CTAs (one CTA per SM), persistent over a dynamic
// schedule of 256 x 256 pair tiles taken in order from a per-launch counter.
// The pair runs one tcgen05.mma.cta_group::2 of M = 256, N = 256: CTA rank r
// holds rows 128 r .. 128 r + 127 of the A tile and columns 128 r ..
// 128 r + 127 of the B tile in its own shared memory, and receives rows
// 128 r .. of the 256 x 256 fp32 accumulator in its own TMEM.  A CTA thus
// stores 32 KB per 64-deep K slab (a lone 128 x 256 tile needs 48 KB), so the
// ring holds six stages.
//   warp 0      (both CTAs) one thread issues the CTA's TMA loads into a
//               6-stage ring; the bytes of both CTAs complete on the
//               leader's (rank 0) full barrier
//   warp 1      (both CTAs) allocates 512 TMEM columns as a pair; in the
//               leader one thread issues the MMAs (kind::f16, bf16 operands,
//               fp32 accumulation) into one of two 256-column accumulators
//               and commits to both CTAs' barriers
//   warps 2, 3  idle (they complete warpgroup 0, whose registers go to the
//               epilogue: setmaxnreg, 56 per thread against 224)
//   warps 4..11 (both CTAs) epilogue, two per TMEM lane quarter (128 columns
//               each): tcgen05.ld the accumulator (row per thread), apply the
//               fused epilogue, store; then release the accumulator to the
//               leader so the next tile's MMAs overlap this tile's epilogue.
// Operands use the 128-byte swizzle.  A is K-major (row-major M x K).  B is
// K-major (stored N x K: symmetric operands and the Gram product) or MN-major
// (stored K x N: the m x n iterate multiplied from the left).  A group may
// split K into parts (split-bf16 operands [hi | lo], see GemmGroup::kseg) and
// store its bf16 outputs split (the kernel instance with kSplit = true); a
// symmetric group of matrices with m <= 128 packs 2 or 4 of them
// block-diagonally into one pair tile (GemmGroup::pack).
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on expiry the
// waiting thread records DEV_TIMEOUT in the status word and leaves its loop,
// so a broken pipeline ends the kernel instead of hanging the GPU.  The
// per-stage ring waits (full, empty) only order the async proxy's copies and
// MMAs, which their mbarrier transactions already cover, and use CTA scope; a
// cluster-scope acquire on them cost about 10 % of the step.  The tile ring
// and the accumulator hand-off between the CTAs' threads use cluster scope;
// the epilogue warps' arrivals on them are relaxed (see their call sites).
#include <cuda_bf16.h>

#include <type_traits>

#include "epilogue.cuh"

namespace dmuon {
namespace {

constexpr int BM = kTcBM;
constexpr int BN = kTcBN;
constexpr int STAGES = kTcStages;
constexpr int SLAB_K = kTcSlabBytes / 2;        // 64 bf16 per 128-byte row
constexpr int UMMA_K = 16;                      // bf16 K per tcgen05.mma
constexpr int kPair = kTcPair;                  // CTAs per cluster sharing one MMA
constexpr int A_BYTES = BM * kTcSlabBytes;      // 16 KB: this CTA's 128 rows of A
constexpr int B_BYTES = (BN / kPair) * kTcSlabBytes;  // 16 KB: this CTA's 128 columns of B
constexpr int MN_BOX_BYTES = SLAB_K * 128;      // one MN-major box: 64 K-rows x 128 B
constexpr uint32_t STAGE_TX = kPair * (A_BYTES + B_BYTES);  // both CTAs' bytes, on the leader's barrier
constexpr uint32_t TMEM_COLS = 512;             // two 256-column accumulators
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kTileRing = 4;
constexpr int kTStageLd = 132;  // 128 W columns + 4 pad; 528-byte rows keep float4 reads aligned
static_assert(4 * 32 * 16 <= 16 * kTStageLd, "a half's stage holds four 32 x 16 diagonal slices");
// warpgroup 0 (warps 0-3): TMA, MMA and two idle warps; warpgroups 1-2:
// the epilogue
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = (kTcThreads - 32 * kEpiWarp0) / 32;
// Registers per thread after the split (setmaxnreg): warpgroup 0 gives
// back what its roles do not need, the epilogue takes it.  Per SM
// sub-partition (one warp of each warpgroup) 56 + 2 x 224 = 3 x 168, the
// launch's allocation, so the increase never waits for registers that are
// not there.
constexpr int kRegsLow = 56;
constexpr int kRegsEpi = 224;
static_assert(kTcThreads == 384 && kRegsLow + 2 * kRegsEpi <= 3 * 168, "register split must fit the launch");
// epilogue warps come in sets of four (one per TMEM lane quarter); each set
// takes an equal part of the 256 accumulator columns
constexpr int kColParts = kEpiWarps / 4;
static_assert(kEpiWarps % 4 == 0 && (kColParts == 1 || kColParts == 2), "4 or 8 epilogue warps");
// readers of a tile slot: the 8 epilogue warps of each CTA, the leader's MMA
// thread and the partner's producer
constexpr uint32_t kTileReaders = kPair * kEpiWarps + 2;
constexpr int CH = 16;                          // epilogue chunk: columns per tcgen05.ld
constexpr uint16_t kPairMask = (1u << kPair) - 1;

struct __align__(1024) Smem {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint64_t full[STAGES];       // leader only: both CTAs' loads of a stage landed
    uint64_t empty[STAGES];      // the pair's MMAs have read the stage (count 1)
    uint64_t acc_full[2];        // the accumulator is complete (count 1)
    uint64_t acc_empty[2];       // leader only: every epilogue warp of both CTAs is done
    uint64_t tile_full[kTileRing];   // a tile index is in tile_slot (count 1)
    uint64_t tile_empty[kTileRing];  // leader only: every reader of both CTAs is done
    int32_t tile_slot[kTileRing];
    uint32_t tmem_base;
    // transposed W update: a 16 x 128 chunk of v per epilogue group (column
    // half), padded rows (read as float4: 16-byte aligned); in store launches
    // four 32 x 16 slices per group, one per epilogue warp, stage diagonal chunks
    alignas(16) float tstage[2][CH * kTStageLd];
};

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes)
                 : "memory");
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

// Slow path of the bounded wait: polls for about 2 s of %globaltimer.
__device__ __forceinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, int32_t* status) {
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitNs) {
            atomicExch(status, DEV_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait for the phase of the given parity.  false = timed out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, status);
}

// TMA box load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, int32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Arrive without release ordering on an mbarrier of this or the partner CTA:
// for a signal that covers no memory operation of the arriving thread (an
// accumulator whose every tcgen05.ld has already completed).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive (release, cluster scope) on an mbarrier of this or the partner CTA.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait with cluster-scope acquire (the arrivals come from the partner).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int32_t* status) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitNs) {
            atomicExch(status, DEV_TIMEOUT);
            return false;
        }
    }
}

// All threads of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// A tensor map written by a host copy must be acquired by the tensormap proxy
// before TMA reads it.
__device__ __forceinline__ void tensormap_acquire(const CUtensorMap* map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.sys [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(map))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family format).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version
    d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
    return d;
}

// Instruction descriptor: kind::f16, bf16 A/B, fp32 D, M = 256 (the pair),
// N = 256.
__host__ __device__ constexpr uint32_t make_idesc(bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>((kPair * BM) >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at this offset in every CTA of `mask` once this
// thread's MMAs so far have completed.
__device__ __forceinline__ void umma_commit_mc(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            saddr(bar)),
        "h"(mask)
        : "memory");
}

// CH = 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[CH]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct TileCoord {
    int gi, mat, tm, tn;
};

// Dynamic schedule.  The pair's leader producer takes pair tiles from the
// launch's counter in order and publishes each index in a ring slot of both
// CTAs; readers wait for the slot, read it, and release it to the leader.
// Taking tiles in order keeps the pairs working on neighbouring tiles, whose
// operands are shared in L2 (a static round-robin lets the pairs drift apart
// over a long launch and thrash L2).  Returns the tile index, or a value
// >= total_tiles when the launch is out of tiles or a wait timed out.
__device__ __forceinline__ int wait_tile(uint64_t* full, const int32_t* slots, int k, int32_t* status, int total) {
    const int slot = k % kTileRing;
    const uint32_t ph = static_cast<uint32_t>(k / kTileRing) & 1u;
    if (!mbar_wait_cluster(&full[slot], ph, status)) return total;
    return *reinterpret_cast<const volatile int32_t*>(&slots[slot]);
}

// After every thread of the reader has read slot k: give it back to the leader.
__device__ __forceinline__ void release_tile(uint64_t* empty, int k) {
    mbar_arrive_cluster(mapa(saddr(&empty[k % kTileRing]), 0));
}

// The epilogue warps' form: every lane reads the slot with an acquire load,
// which orders its later operations after the read, and __syncwarp orders all
// lanes' reads before lane 0's arrive, so the arrive itself can be relaxed (a
// release would wait for the warp's global stores of the previous tile to
// drain at cluster scope).
__device__ __forceinline__ int wait_tile_acquire(uint64_t* full, const int32_t* slots, int k, int32_t* status,
                                                 int total) {
    const int slot = k % kTileRing;
    const uint32_t ph = static_cast<uint32_t>(k / kTileRing) & 1u;
    if (!mbar_wait_cluster(&full[slot], ph, status)) return total;
    int32_t t;
    asm volatile("ld.acquire.cluster.shared::cta.b32 %0, [%1];" : "=r"(t) : "r"(saddr(&slots[slot])) : "memory");
    return t;
}

// Static schedule over pair tiles: index -> (group, matrix, pair row, column
// tile).  A pair tile is 256 x 256; CTA rank r of the pair computes its rows
// 128 r .. 128 r + 127 (a 128 x 256 accumulator), and the two share the B
// tile.  Symmetric groups enumerate pair row i with column tiles 0 .. i, the
// lower triangle.
__device__ __forceinline__ TileCoord decode_tile(const LaunchList& L, int t) {
    TileCoord c;
    int gi = 0;
    while (gi + 1 < L.n && L.begin[gi + 1] <= t) ++gi;
    const GemmGroup& g = L.groups[L.idx[gi]];
    const int local = t - L.begin[gi];
    c.gi = gi;
    c.mat = local / g.tiles_per_mat * g.pack;  // packed groups: the tile's first matrix
    int idx = local % g.tiles_per_mat;
    if (g.sym) {
        int i = 0;
        while (idx >= i + 1) {
            idx -= i + 1;
            ++i;
        }
        c.tm = i;
        c.tn = idx;
    } else {
        // Panels of kPanel column tiles, pair rows inside a panel: a wave of
        // 76 pairs then covers about 10 x 8 pair tiles, whose A rows and B
        // columns stay in L2, instead of re-streaming all of B once per row.
        constexpr int kPanel = 8;
        const int panel_tiles = g.tiles_m * kPanel;
        const int panel = idx / panel_tiles;
        const int within = idx - panel * panel_tiles;
        const int width = min(kPanel, g.tiles_n - panel * kPanel);
        c.tm = within / width;
        c.tn = panel * kPanel + within % width;
    }
    return c;
}

// Warp-cooperative row segments.  After tcgen05.ld lane i of a warp holds row
// r0 + i, columns c0 .. c0+15: a 16-byte access per lane would then touch 32
// different rows (32 L2 requests, each for half a 32-byte sector of fp32 or
// bf16 data).  Regrouping the data between lanes first makes each access
// instruction cover whole row segments: bf16 rows (32 bytes) are swapped in
// halves between lanes i and i^1, so one instruction writes 16 full sectors;
// fp32 rows (64 bytes) are transposed as 4 x 4 blocks of 16 bytes inside each
// lane quad, so one instruction writes 8 rows x 64 contiguous bytes.  Loads
// use the same layouts in reverse.  All 32 lanes must call these; rows >= M
// are neither read (zero) nor written.
constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}

// 4 x 4 transpose of 16-byte blocks within each lane quad: block q of lane
// i (words 4q .. 4q+3) ends in block i of lane q.  Its own inverse.
template <typename T>
__device__ __forceinline__ void quad_transpose(T (&w)[16], int lane) {
#pragma unroll
    for (int s = 2; s >= 1; s >>= 1) {
        const bool hi = (lane & s) != 0;
#pragma unroll
        for (int q0 = 0; q0 < 4; ++q0) {
            if (q0 & s) continue;
            const int q1 = q0 | s;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const T send = hi ? w[4 * q0 + k] : w[4 * q1 + k];
                const T recv = __shfl_xor_sync(kFullMask, send, s);
                w[4 * q0 + k] = hi ? recv : w[4 * q0 + k];
                w[4 * q1 + k] = hi ? w[4 * q1 + k] : recv;
            }
        }
    }
}

// fp32 rows are transposed in v itself (no copy: the registers are scarce);
// `restore` transposes v back for later uses.
// A bf16 output stored split (lo > 0) writes its low parts lo elements
// further along each row, with the same lane exchange.
__device__ __forceinline__ void st_rows_bf16(char* base, int64_t ld, int r0, int c0, int lane, const float (&v)[CH],
                                             int M, bool low, int rmin) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        w[k] = low ? pack_bf16x2(lo_part(v[2 * k]), lo_part(v[2 * k + 1])) : pack_bf16x2(v[2 * k], v[2 * k + 1]);
    const bool odd = lane & 1;
    uint32_t d0[4], d1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t keep = odd ? w[4 + k] : w[k];
        const uint32_t recv = __shfl_xor_sync(kFullMask, odd ? w[k] : w[4 + k], 1);
        d0[k] = odd ? recv : keep;  // row (lane & ~1), half `odd`
        d1[k] = odd ? keep : recv;  // row (lane | 1),  half `odd`
    }
    const int ra = r0 + (lane & ~1);
    __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(base) + static_cast<int64_t>(ra) * ld + c0 + 8 * odd;
    if (ra < M && ra >= rmin) *reinterpret_cast<uint4*>(p) = make_uint4(d0[0], d0[1], d0[2], d0[3]);
    if (ra + 1 < M && ra + 1 >= rmin) *reinterpret_cast<uint4*>(p + ld) = make_uint4(d1[0], d1[1], d1[2], d1[3]);
}

// Rows below rmin are not stored (the upper half of a chunk right of the
// diagonal).
__device__ __forceinline__ void st_rows(char* base, int32_t type, int64_t ld, int r0, int c0, int lane,
                                        float (&v)[CH], int M, bool restore, int lo, int rmin = 0) {
    if (type == ELEM_BF16) {
        st_rows_bf16(base, ld, r0, c0, lane, v, M, false, rmin);
        if (lo) st_rows_bf16(base + 2 * static_cast<int64_t>(lo), ld, r0, c0, lane, v, M, true, rmin);
        return;
    }
    quad_transpose(v, lane);
    const int rq = r0 + (lane & ~3);
    float* p = reinterpret_cast<float*>(base) + static_cast<int64_t>(rq) * ld + c0 + 4 * (lane & 3);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (rq + j < M && rq + j >= rmin)
            *reinterpret_cast<float4*>(p + j * ld) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    if (restore) quad_transpose(v, lane);
}

__device__ __forceinline__ void ld_rows(const char* base, int32_t type, int64_t ld, int r0, int c0, int lane,
                                        float (&x)[CH], int M) {
    if (type == ELEM_BF16) {
        const bool odd = lane & 1;
        const int ra = r0 + (lane & ~1);
        const __nv_bfloat16* p =
            reinterpret_cast<const __nv_bfloat16*>(base) + static_cast<int64_t>(ra) * ld + c0 + 8 * odd;
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (ra < M) a = *reinterpret_cast<const uint4*>(p);
        if (ra + 1 < M) b = *reinterpret_cast<const uint4*>(p + ld);
        const uint32_t d0[4] = {a.x, a.y, a.z, a.w}, d1[4] = {b.x, b.y, b.z, b.w};
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t recv = __shfl_xor_sync(kFullMask, odd ? d0[k] : d1[k], 1);
            w[k] = odd ? recv : d0[k];
            w[4 + k] = odd ? d1[k] : recv;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 f = unpack_bf16x2(w[k]);
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    } else {
        const int rq = r0 + (lane & ~3);
        const float* p = reinterpret_cast<const float*>(base) + static_cast<int64_t>(rq) * ld + c0 + 4 * (lane & 3);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 q = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (rq + j < M) q = *reinterpret_cast<const float4*>(p + j * ld);
            x[4 * j] = q.x;
            x[4 * j + 1] = q.y;
            x[4 * j + 2] = q.z;
            x[4 * j + 3] = q.w;
        }
        quad_transpose(x, lane);
    }
}

// The epilogue works on this thread's row r, columns c0 .. c0+CH-1
// (tcgen05.ld leaves one row per thread).  Row segments move as 16-byte
// vectors, and so do the mirrored halves of symmetric results once transposed
// in registers (mirror_words); the mirrors of chunks on the diagonal or at a
// ragged edge, the symmetric aux reads and the transposed W update use the
// other orientation, where the warp's 32 lanes cover 32 consecutive rows and
// each access is coalesced.
//
// Inputs of a chunk (aux or W) do not depend on the accumulator, so they are
// loaded one chunk ahead: the first chunk's before the wait for the MMAs, the
// next chunk's before the current chunk's stores.

// CH elements of row r from columns c0.. of a row-major matrix (or of its
// transpose when by_col: element (r, c) read at [c][r]).
__device__ __forceinline__ void load_row(const char* base, int32_t type, int32_t ld, bool by_col, int r, int c0,
                                         int ncol, float (&x)[CH]) {
    if (by_col) {
#pragma unroll
        for (int j = 0; j < CH; ++j)
            x[j] = j < ncol ? load_elem(base, static_cast<int64_t>(c0 + j) * ld + r, type) : 0.0f;
    } else {
#pragma unroll
        for (int j = 0; j < CH; ++j)
            x[j] = j < ncol ? load_elem(base, static_cast<int64_t>(r) * ld + c0 + j, type) : 0.0f;
    }
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// At tile start, a whole mainloop before use: pull into L2 every W / aux line
// this thread's chunks will read (chunks c0, c0 + CH, ... of nch), so the
// epilogue's loads hit L2 instead of HBM.  By-column inputs (transposed W,
// symmetric aux) are row segments of 32 lanes, one line per input row.
__device__ __forceinline__ void prefetch_rows(const char* base, int32_t type, int32_t ld, bool by_col, int r,
                                              int r0, int lane, int c_first, int ncols, int M, int N) {
    const int es = type == ELEM_BF16 ? 2 : 4;
    if (!by_col) {
        if (r >= M) return;
        const int c_end = min(c_first + ncols, N);
        for (int c = c_first; c < c_end; c += 128 / es)
            prefetch_l2(base + (static_cast<int64_t>(r) * ld + c) * es);
    } else {
        if (r0 >= M) return;  // no valid row in this warp's 32 lanes
        for (int c = c_first + lane; c < min(c_first + ncols, N); c += 32)
            prefetch_l2(base + (static_cast<int64_t>(c) * ld + r0) * es);
    }
}

__device__ __forceinline__ void epi_prefetch(const EpiRegs& e, int r, int r0, int lane, int c_first, int ncols) {
    if (e.update()) {
        prefetch_rows(e.w, e.w_type(), e.w_cols, e.transposed(), r, r0, lane, c_first, ncols, e.M, e.N);
        if (e.aux) prefetch_rows(e.aux, e.aux_type(), e.aux_ld, e.aux_sym(), r, r0, lane, c_first, ncols, e.M, e.N);
    } else if (e.aux) {
        prefetch_rows(e.aux, e.aux_type(), e.aux_ld, e.aux_sym(), r, r0, lane, c_first, ncols, e.M, e.N);
    }
}

// Prefetched input of a chunk: W for the update, else the aux operand.
template <bool kUpd>
__device__ __forceinline__ void epi_load(const EpiRegs& e, int r, int r0, int lane, int c0, float (&x)[CH]) {
    if (r0 >= e.M || c0 >= e.N) return;  // warp-uniform
    const int ncol = min(CH, e.N - c0);
    const bool full = ncol == CH;
    const char* base;
    int32_t type, ld;
    bool by_col;
    bool vec;
    if (kUpd) {
        base = e.w;
        type = e.w_type();
        ld = e.w_cols;
        by_col = e.transposed();
        vec = full && e.w_vec();
    } else if (e.aux) {
        base = e.aux;
        type = e.aux_type();
        ld = e.aux_ld;
        by_col = e.aux_sym();
        vec = full;
    } else {
        return;
    }
    if (vec && !by_col) ld_rows(base, type, ld, r0, c0, lane, x, e.M);
    else if (r < e.M) load_row(base, type, ld, by_col, r, c0, ncol, x);
}

// Mirrored half of a 32 x 16 chunk that lies strictly below the diagonal (all
// its elements stored): element (r0 + lane, c0 + j) also goes to
// [c0 + j][r0 + lane].  A three-stage exchange inside each group of 8 lanes
// transposes the chunk in registers (the 8 x 8 blocks of each half of the
// columns, like quad_transpose one level deeper), so lane (g, t) =
// (lane / 8, lane % 8) ends with mirrored rows t and 8 + t, columns
// r0 + 8g .. r0 + 8g + 7, as two 16-byte bf16 pieces: two stores per lane
// instead of sixteen 2-byte ones; with `low`, the pieces hold the low bf16
// parts of a split output instead.  v is left as it is.  All 32 lanes must
// call this.
__device__ __forceinline__ void mirror_words(const float (&v)[CH], int lane, uint4 (&mw)[2], bool low) {
    float a[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) a[j] = v[j];
#pragma unroll
    for (int k = 4; k >= 1; k >>= 1) {
        const bool hi = (lane & k) != 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j0 = 0; j0 < 8; ++j0) {
                if (j0 & k) continue;
                const int i0 = 8 * h + j0, i1 = 8 * h + (j0 | k);
                const float send = hi ? a[i0] : a[i1];
                const float recv = __shfl_xor_sync(kFullMask, send, k);
                a[i0] = hi ? recv : a[i0];
                a[i1] = hi ? a[i1] : recv;
            }
        }
    }
    if (low) {
#pragma unroll
        for (int j = 0; j < CH; ++j) a[j] = lo_part(a[j]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
        mw[h] = make_uint4(pack_bf16x2(a[8 * h], a[8 * h + 1]), pack_bf16x2(a[8 * h + 2], a[8 * h + 3]),
                           pack_bf16x2(a[8 * h + 4], a[8 * h + 5]), pack_bf16x2(a[8 * h + 6], a[8 * h + 7]));
}

__device__ __forceinline__ void st_mirror(char* base, int64_t ld, int r0, int c0, int lane, const uint4 (&mw)[2]) {
    __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(base) + r0 + (lane >> 3) * 8;
    const int t = lane & 7;
    *reinterpret_cast<uint4*>(p + static_cast<int64_t>(c0 + t) * ld) = mw[0];
    *reinterpret_cast<uint4*>(p + static_cast<int64_t>(c0 + 8 + t) * ld) = mw[1];
}

// A whole 32 x 16 chunk of a symmetric result that touches the diagonal
// (c0 == r0: rows r0 .. r0+15 hold the 16 x 16 diagonal block, rows
// r0+16 .. r0+31 lie below it; c0 == r0 + 16: rows r0+16 .. hold the
// diagonal block, rows r0 .. r0+15 lie above it).  Instead of element-wise
// stores of the lower triangle and its mirror (one 2-byte store per lane and
// element, each to another row), the chunk is staged in `stg` (512 floats of
// shared memory owned by this warp, XOR-swizzled rows) and written back as
// 8-element row pieces, one per lane and pass, each a 16-byte (bf16) or two
// 16-byte (fp32) stores:
//   - rows of the chunk (all 32 for c0 == r0, the lower 16 otherwise), with
//     the diagonal block as the symmetric result holds it: element (r, c)
//     is acc[r][c] on and below the diagonal and acc[c][r] above it;
//   - for c0 == r0, the mirror of the rows below the block: rows c0 .. c0+15,
//     columns r0+16 .. r0+31.
// Every upper element is still the mirror of a lower one: the result stays
// bitwise symmetric.  All 32 lanes must call this.
__device__ __forceinline__ int stg_idx(int i, int j) { return i * CH + (j ^ (i & 15)); }

// 8 consecutive elements from (row r0 + i, column c0 + j0) of output o.
template <bool kSplit>
__device__ __forceinline__ void st_piece(const EpiRegs& e, int o, int64_t idx, const float (&w)[8]) {
    const int lo = kSplit ? e.out_lo[o] : 0;
    if (e.out_type(o) == ELEM_BF16) {
        __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(e.out[o]) + idx;
        *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                                                  pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
        if (lo)
            *reinterpret_cast<uint4*>(p + lo) =
                make_uint4(pack_bf16x2(lo_part(w[0]), lo_part(w[1])), pack_bf16x2(lo_part(w[2]), lo_part(w[3])),
                           pack_bf16x2(lo_part(w[4]), lo_part(w[5])), pack_bf16x2(lo_part(w[6]), lo_part(w[7])));
    } else {
        float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out[o]) + idx);
        p[0] = make_float4(w[0], w[1], w[2], w[3]);
        p[1] = make_float4(w[4], w[5], w[6], w[7]);
    }
}

template <bool kSplit>
__device__ __forceinline__ void epi_store_diag(const EpiRegs& e, int r0, int lane, int c0, const float (&v)[CH],
                                               float* stg) {
#pragma unroll
    for (int j = 0; j < CH; ++j) stg[stg_idx(lane, j)] = v[j];
    __syncwarp();
    const int d = c0 - r0;  // 0 or 16: the diagonal block's first row inside the chunk
    const int h = lane & 1;
    // rows: pass 1 for the block rows d .. d+15, pass 0 (c0 == r0 only) for rows 16 .. 31
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        if (pass == 0 && d != 0) continue;
        const int i = (pass == 0 ? 16 : d) + (lane >> 1);  // chunk row
        float w[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int j = 8 * h + t;  // chunk column; matrix column c0 + j vs row r0 + i
            w[t] = (pass == 1 && j + d > i) ? stg[stg_idx(j + d, i - d)] : stg[stg_idx(i, j)];
        }
#pragma unroll
        for (int o = 2; o >= 0; --o)
            if (e.out[o]) st_piece<kSplit>(e, o, static_cast<int64_t>(r0 + i) * e.out_ld[o] + c0 + 8 * h, w);
    }
    if (d == 0) {
        // mirrored row c0 + (lane >> 1), columns r0 + 16 + 8h .. : chunk rows 16 + 8h ..
        const int jj = lane >> 1, i0 = 16 + 8 * h;
        float w[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) w[t] = stg[stg_idx(i0 + t, jj)];
#pragma unroll
        for (int o = 2; o >= 0; --o)
            if (e.out[o] && e.out_mirror(o))
                st_piece<kSplit>(e, o, static_cast<int64_t>(c0 + jj) * e.out_ld[o] + r0 + i0, w);
    }
    __syncwarp();  // the stage is read before the next chunk writes it
}

// v (computed in place of the accumulator values) and, for the update, the new
// W (in place of the loaded W values), to keep the register footprint low.
// kSplit: the launch holds groups with split outputs (the other instance
// carries none of their code).
template <bool kSplit, bool kUpd>
__device__ __forceinline__ void epi_finish(const EpiRegs& e, int r, int r0, int lane, int c0, float (&v)[CH],
                                           float (&x)[CH], float* stg) {
    if (r0 >= e.M) return;  // warp-uniform: no row of this warp exists
    const bool valid = r < e.M;
    const int ncol = min(CH, e.N - c0);
    const bool full = ncol == CH;
    constexpr bool upd = kUpd;
    if (upd && e.aux) {
        // the update that also has an aux term (direct route: a X + B X) reads
        // the aux chunk here; x already holds W
        float a[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) a[j] = 0.0f;
        if (full && !e.aux_sym()) ld_rows(e.aux, e.aux_type(), e.aux_ld, r0, c0, lane, a, e.M);
        else if (valid) load_row(e.aux, e.aux_type(), e.aux_ld, e.aux_sym(), r, c0, ncol, a);
#pragma unroll
        for (int j = 0; j < CH; ++j) v[j] = epi_v(e, r, c0 + j, v[j], a[j]);
    } else {
#pragma unroll
        for (int j = 0; j < CH; ++j) v[j] = epi_v(e, r, c0 + j, v[j], upd ? 0.0f : x[j]);
    }

    if (!upd) {
        if (e.sym() && c0 + CH - 1 >= r0) {  // warp-uniform: the chunk reaches the warp's diagonal
            if (c0 >= r0 + 32) return;     // wholly above it: nothing of it is stored
            if (full && r0 + 32 <= e.M) {
                epi_store_diag<kSplit>(e, r0, lane, c0, v, stg);
                return;
            }
        }
        // every column of the chunk is stored directly in all 32 rows of the warp
        const bool coop = full && (!e.sym() || c0 + CH - 1 < r0);
        // whole 32-row chunk left of the diagonal block: bf16 mirrors built
        // once in registers (mirror_words), shared by every mirrored output
        const bool mfast = coop && e.sym() && r0 + 32 <= e.M;
        uint4 mw[2];
        bool have_mw = false;
        // last output first, and each output's mirror before its rows: an fp32
        // row store leaves v transposed unless something still needs it
#pragma unroll
        for (int o = 2; o >= 0; --o) {
            if (!e.out[o]) continue;
            const int lo = kSplit ? e.out_lo[o] : 0;
            if (e.out_mirror(o)) {
                if (mfast && e.out_type(o) == ELEM_BF16 && ((e.out_ld[o] | lo) & 7) == 0) {  // warp-uniform
                    if (!have_mw) {
                        mirror_words(v, lane, mw, false);
                        have_mw = true;
                    }
                    st_mirror(e.out[o], e.out_ld[o], r0, c0, lane, mw);
                    if (lo) {
                        // low parts in the same registers (the high parts are
                        // rebuilt for a later split output)
                        mirror_words(v, lane, mw, true);
                        st_mirror(e.out[o] + 2 * static_cast<int64_t>(lo), e.out_ld[o], r0, c0, lane, mw);
                        have_mw = false;
                    }
                } else if (valid) {
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        if (j < ncol && r > c0 + j) {
                            const int64_t i = static_cast<int64_t>(c0 + j) * e.out_ld[o] + r;
                            store_elem(e.out[o], i, e.out_type(o), v[j]);
                            if (lo) store_elem(e.out[o], i + lo, ELEM_BF16, lo_part(v[j]));
                        }
                }
            }
            if (coop) {
                st_rows(e.out[o], e.out_type(o), e.out_ld[o], r0, c0, lane, v, e.M, o > 0, lo);
            } else if (valid) {
                const int64_t rb = static_cast<int64_t>(r) * e.out_ld[o];
#pragma unroll
                for (int j = 0; j < CH; ++j)
                    if (j < ncol && (!e.sym() || r >= c0 + j)) {
                        store_elem(e.out[o], rb + c0 + j, e.out_type(o), v[j]);
                        if (lo) store_elem(e.out[o], rb + lo + c0 + j, ELEM_BF16, lo_part(v[j]));
                    }
            }
        }
        return;
    }
    // Muon update W = decay*W - lr*s*v in W's own orientation (x holds W)
    float (&w)[CH] = x;
#pragma unroll
    for (int j = 0; j < CH; ++j) w[j] = fmaf(-e.lrs, v[j], e.decay * x[j]);
    if (!e.transposed()) {
        const int64_t rb = static_cast<int64_t>(r) * e.w_cols;
        if (full && e.w_vec()) {
            st_rows(e.w, e.w_type(), e.w_cols, r0, c0, lane, w, e.M, false, 0);
        } else if (valid) {
#pragma unroll
            for (int j = 0; j < CH; ++j)
                if (j < ncol) store_elem(e.w, rb + c0 + j, e.w_type(), w[j]);
        }
    } else if (valid) {
#pragma unroll
        for (int j = 0; j < CH; ++j)
            if (j < ncol) store_elem(e.w, static_cast<int64_t>(c0 + j) * e.w_cols + r, e.w_type(), w[j]);
    }
}

// Transposed W update (tall matrices: D row r is W column r).  The four warps
// of a column half own 32 D rows each, so alone each could touch only 64 bytes
// of a W row at a time.  Instead they stage a 16 x 128 chunk of v in shared
// memory and each warp then updates 4 whole W row segments of 128 columns,
// 4 consecutive elements per lane (8- or 16-byte accesses).
__device__ __forceinline__ void named_bar(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(128) : "memory");
}

// Named barrier of the 128 threads of an epilogue group that also returns the AND
// of their predicates: the four warps take every loop exit together, so none
// is left waiting at a barrier the others no longer reach.
__device__ __forceinline__ bool named_bar_and(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(128)
        : "memory");
    return r != 0;
}

// W[c0 + 4q + i][wc .. wc+3] for i < 4 into w (rows beyond N, columns beyond M skipped).
__device__ __forceinline__ void tw_load(const EpiRegs& e, int c0, int q, int wc, float (&w)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = c0 + 4 * q + i;
        if (c >= e.N) continue;
        const int64_t base = static_cast<int64_t>(c) * e.w_cols + wc;
        if (wc + 3 < e.M) {
            if (e.w_type() == ELEM_BF16) {
                const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(e.w) + base);
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
                w[i][0] = f0.x; w[i][1] = f0.y; w[i][2] = f1.x; w[i][3] = f1.y;
            } else {
                const float4 f = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(e.w) + base);
                w[i][0] = f.x; w[i][1] = f.y; w[i][2] = f.z; w[i][3] = f.w;
            }
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (wc + t < e.M) w[i][t] = load_elem(e.w, base + t, e.w_type());
        }
    }
}

__device__ __forceinline__ void tw_store(const EpiRegs& e, int c0, int q, int wc, const float* stg, int lane,
                                         const float (&w)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = c0 + 4 * q + i;
        if (c >= e.N) continue;
        const float4 v = *reinterpret_cast<const float4*>(stg + (4 * q + i) * kTStageLd + 4 * lane);
        const float n0 = fmaf(-e.lrs, v.x, e.decay * w[i][0]);
        const float n1 = fmaf(-e.lrs, v.y, e.decay * w[i][1]);
        const float n2 = fmaf(-e.lrs, v.z, e.decay * w[i][2]);
        const float n3 = fmaf(-e.lrs, v.w, e.decay * w[i][3]);
        const int64_t base = static_cast<int64_t>(c) * e.w_cols + wc;
        if (wc + 3 < e.M) {
            if (e.w_type() == ELEM_BF16) {
                uint2 u;
                *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(n0, n1);
                *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(n2, n3);
                *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(e.w) + base) = u;
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(e.w) + base) = make_float4(n0, n1, n2, n3);
            }
        } else {
            const float n[4] = {n0, n1, n2, n3};
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (wc + t < e.M) store_elem(e.w, base + t, e.w_type(), n[t]);
        }
    }
}

template <bool kSplit, bool kUpd>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ LaunchList L) {
    extern __shared__ uint8_t smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&S.full[s], 1);   // the leader's expect_tx; the bytes of both CTAs
            mbar_init(&S.empty[s], 1);  // the leader's MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.acc_full[b], 1);
            // the epilogue warps that read one accumulator: all 8 per CTA
            // (column halves) or the 4 of one set (sets: alternate tiles)
            mbar_init(&S.acc_empty[b], kPair * (L.epi_sets ? 4 : kEpiWarps));
        }
        for (int i = 0; i < kTileRing; ++i) {
            mbar_init(&S.tile_full[i], 1);
            mbar_init(&S.tile_empty[i], kTileReaders);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        // one warp of each CTA: the same columns in both CTAs' TMEM
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&S.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the partner's barriers exist before any remote arrival targets them
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    const int rank = static_cast<int>(cluster_rank());
    const int total = L.total_tiles;
    // The launch may start while the previous kernel in the stream finishes
    // (programmatic dependent launch): the set-up above touches only this
    // CTA's shared memory and TMEM; global memory waits for that kernel's
    // completion and its writes.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Register split, warpgroup-uniform; each role's code sits inside the
    // branch of its own setmaxnreg, so it is compiled to that budget.
    if (warp < kEpiWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t stage = 0, phase = 0;
        uint32_t n_issued = 0;  // slabs issued so far (ring position n_issued % STAGES)
        bool ok = true;
        const uint32_t full0 = mapa(saddr(&S.full[0]), 0);  // the leader's barriers, 8 bytes apart
        for (int j = 0; j < L.n; ++j) {
            tensormap_acquire(&L.groups[L.idx[j]].tma_a);
            tensormap_acquire(&L.groups[L.idx[j]].tma_b);
        }
        // the leader takes tile indices one ahead, so the atomic's latency
        // hides behind the current tile's loads
        int t_next = rank == 0 ? atomicAdd(L.counter, 1) : 0;
        for (int k = 0; ok; ++k) {
            int t;
            if (rank == 0) {
                // publish the next tile in both CTAs' ring slot
                const int slot = k % kTileRing;
                const uint32_t ph = static_cast<uint32_t>(k / kTileRing) & 1u;
                if (!mbar_wait_cluster(&S.tile_empty[slot], ph ^ 1u, L.status)) {
                    ok = false;
                    break;
                }
                t = t_next < total ? t_next : total;
                if (t < total) t_next = atomicAdd(L.counter, 1);
                S.tile_slot[slot] = t;
                st_cluster_u32(mapa(saddr(&S.tile_slot[slot]), 1), t);
                mbar_arrive_cluster(mapa(saddr(&S.tile_full[slot]), 0));
                mbar_arrive_cluster(mapa(saddr(&S.tile_full[slot]), 1));
            } else {
                t = wait_tile(S.tile_full, S.tile_slot, k, L.status, total);
                release_tile(S.tile_empty, k);
            }
            if (t >= total) {
                // no tile left to claim: the next launch's CTAs may be placed
                // on SMs as this launch's CTAs leave them
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
                break;
            }
            const TileCoord tc = decode_tile(L, t);
            const GemmGroup* g = L.groups + L.idx[tc.gi];
            const int nkb = (g->K + SLAB_K - 1) / SLAB_K;
            const int b_col = tc.tn * BN + rank * (BN / kPair);  // this CTA's 128 columns of B
            // per-tile fields in registers (the waits' memory clobbers would
            // otherwise reload them from the group table for every slab)
            const int kseg = g->kseg;
            const bool b_mn = g->b_mn_major != 0;
            // packed group: CTA rank r holds matrices mat + r pack/2 .. (rows 0 ..)
            const int pk = g->pack;
            const int a_row = pk > 1 ? 0 : (2 * tc.tm + rank) * BM;
            const int b_row = pk > 1 ? 0 : b_col;
            const int zb = pk > 1 ? tc.mat + rank * (pk >> 1) : tc.mat;
            const CUtensorMap* map_a = &g->tma_a;
            const CUtensorMap* map_b = &g->tma_b;
            // K segment of the slab and its offset inside it (split operands:
            // segment t reads A's part t % 2 and B's part t / 2), advanced
            // without a division
            int seg = 0, within = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait(&S.empty[stage], phase ^ 1, L.status)) {
                    ok = false;
                    break;
                }
                if (rank == 0) mbar_expect_tx(&S.full[stage], STAGE_TX);
                ++n_issued;
                // own 128 rows of A and own 128 columns of B, counted on the
                // leader's barrier
                const uint32_t fb = full0 + stage * static_cast<uint32_t>(sizeof(uint64_t));
                // K coordinates of this slab in A and in B (no split: kseg = 0,
                // seg stays 0)
                const int ka = (seg & 1) * kseg + within, kbk = (seg >> 1) * kseg + within;
                within += SLAB_K;
                if (within == kseg) {
                    within = 0;
                    ++seg;
                }
                tma_load_3d_pair(S.a[stage], map_a, fb, ka, a_row, zb);
                if (!b_mn) {
                    tma_load_3d_pair(S.b[stage], map_b, fb, kbk, b_row, zb);
                } else {
#pragma unroll
                    for (int i = 0; i < BN / 64 / kPair; ++i)
                        tma_load_3d_pair(S.b[stage] + i * MN_BOX_BYTES, map_b, fb, b_col + 64 * i, kbk, tc.mat);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok) {
            // let copies already issued land before the CTA can exit (the
            // leader's barrier counts both CTAs' copies; the partner waits
            // for the leader at the final cluster barrier)
            if (rank == 0)
                for (uint32_t j = 1; j <= STAGES && j <= n_issued; ++j) {
                    const uint32_t q = n_issued - j;  // a slab issued last, at ring slot q % STAGES
                    mbar_wait(&S.full[q % STAGES], (q / STAGES) & 1u, L.status);
                }
        } else {
            // wait for the MMA's releases of the last ring round, so no
            // commit from the leader is still in flight towards this CTA
            // when the pair leaves through the final cluster barrier
            for (int i = 0; i < STAGES && ok; ++i) {
                ok = mbar_wait_cluster(&S.empty[stage], phase ^ 1, L.status);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ MMA issuer (leader)
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        int it = 0;
        // shared-memory descriptors of stage 0; a stage, and a 16-deep K step
        // inside it, only move the 14-bit start-address field (16-byte units),
        // which stays below its top for every shared-memory address.  This
        // thread alone feeds the pair's tensor cores and shares its scheduler
        // with two epilogue warps: its loop is kept short.
        const uint64_t a_desc0 = smem_desc(saddr(S.a[0]), 0, 1024);
        const uint64_t b_desc0_k = smem_desc(saddr(S.b[0]), 0, 1024);
        const uint64_t b_desc0_mn = smem_desc(saddr(S.b[0]), MN_BOX_BYTES, 1024);
        for (int k = 0; ok; ++k, ++it) {
            const int t = wait_tile(S.tile_full, S.tile_slot, k, L.status, total);
            release_tile(S.tile_empty, k);
            if (t >= total) break;
            const TileCoord tc = decode_tile(L, t);
            const GemmGroup* g = L.groups + L.idx[tc.gi];
            const int nkb = (g->K + SLAB_K - 1) / SLAB_K;
            const int buf = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait_cluster(&S.acc_empty[buf], (use & 1) ^ 1, L.status)) break;
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
            const bool bmn = g->b_mn_major != 0;
            const uint32_t idesc = make_idesc(bmn);
            const uint64_t b_desc0 = bmn ? b_desc0_mn : b_desc0_k;
            const uint64_t b_kstep = bmn ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait(&S.full[stage], phase, L.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad0 = a_desc0 + static_cast<uint64_t>(stage) * (A_BYTES >> 4);
                const uint64_t bd0 = b_desc0 + static_cast<uint64_t>(stage) * (B_BYTES >> 4);
#pragma unroll
                for (int kk = 0; kk < SLAB_K / UMMA_K; ++kk)
                    umma_bf16(d, ad0 + kk * ((UMMA_K * 2) >> 4), bd0 + kk * b_kstep, idesc, (kb | kk) != 0 ? 1u : 0u);
                umma_commit_mc(&S.empty[stage], kPairMask);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            // also on failure: the commit tracks every MMA issued so far, so the
            // epilogue's wait on it covers them before TMEM is released
            umma_commit_mc(&S.acc_full[buf], kPairMask);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        // ------------------------------------------------ epilogue
        // Two groups of four warps (one per TMEM lane quarter each).  Column
        // halves: both groups work on every tile, group h on its columns
        // 128 h .. 128 h + 127.  Sets (L.epi_sets, store launches with many
        // tiles per pair): group h takes the tiles k = h mod 2 -- accumulator
        // h -- whole, so one tile's setup and tail overlap the other's work.
        const int q = warp & 3;             // TMEM lane quarter this warp may access
        const int half = (warp - kEpiWarp0) / 4;  // the group: column half, or set
        const bool sets = L.epi_sets != 0;
        for (int k = 0;; ++k) {
            const int t = wait_tile_acquire(S.tile_full, S.tile_slot, k, L.status, total);
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa(saddr(&S.tile_empty[k % kTileRing]), 0));
            // The group leaves together (a wait that gave up counts for all
            // four): update launches' staged path has group barriers.  Store
            // launches have none, so with column halves each warp leaves on
            // its own; with sets the barrier also parks the warps of the set
            // that skips this tile (measured: faster than letting them run on)
            if (kUpd || sets) {
                if (!named_bar_and(1 + half, t < total)) break;
            } else if (t >= total) {
                break;
            }
            if (sets && (k & 1) != half) continue;
            const TileCoord tc = decode_tile(L, t);
            const GemmGroup& g = L.groups[L.idx[tc.gi]];
            const int buf = k & 1;
            const uint32_t use = static_cast<uint32_t>(k >> 1);
            const int tm = 2 * tc.tm + rank;  // this CTA's 128-row tile
            // this warp's matrix, first row, first column (matrix
            // coordinates) and accumulator column of its chunks
            const int part = sets ? BN : BN / kColParts, part0 = sets ? 0 : half * part;
            int mat = tc.mat, r0w = tm * BM + q * 32, cbase = tc.tn * BN + part0;
            int tcol0 = part0, maxch = part / CH, row_last = tm * BM + BM - 1;
            bool active = true;
            if (g.pack > 1) {
                // packed tile: diagonal block pm (mpad x mpad) is matrix
                // mat + pm; this warp's rows lie in block row / mpad, whose
                // columns lie in one column half (or in the set's tile)
                const int mpad = BN / g.pack, row = rank * BM + q * 32, pm = row / mpad;
                mat = tc.mat + pm;
                r0w = row - pm * mpad;
                cbase = 0;
                tcol0 = pm * mpad;
                maxch = mpad / CH;
                row_last = mpad - 1;
                active = (sets || pm * mpad / part == half) && mat < g.batch;
            }
            const EpiRegs e = load_epi(g, L, active ? mat : tc.mat);
            const int r = r0w + lane;
            // chunks of this warp that hold stored columns
            int nch = 0;
            for (int ch = 0; active && ch < maxch; ++ch) {
                const int c0 = cbase + ch * CH;
                if (c0 >= e.N || (e.sym() && !e.update() && c0 > row_last)) break;
                ++nch;
            }
            if (nch > 0) epi_prefetch(e, r, r0w, lane, cbase, nch * CH);
            // tall matrices' update through the staged path (the same four warps
            // of this half always see the same nch, so the named barriers match)
            const bool tpath = kUpd && e.transposed() && !e.aux && (e.w_cols % 4) == 0;
            if (tpath) {
                const int wc = tm * BM + 4 * lane;
                float* stg = S.tstage[half];
                float wn[4][4];
                if (nch > 0) tw_load(e, cbase, q, wc, wn);
                const bool ready = mbar_wait_cluster(&S.acc_full[buf], use & 1, L.status);
                if (!named_bar_and(1 + half, ready)) break;
                tc_fence_after();
                for (int kc = 0; kc < nch; ++kc) {
                    const int c0 = cbase + kc * CH;
                    float wcur[4][4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int t = 0; t < 4; ++t) wcur[i][t] = wn[i][t];
                    if (kc + 1 < nch) tw_load(e, c0 + CH, q, wc, wn);
                    float v[CH];
                    __syncwarp();
                    tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                  static_cast<uint32_t>(buf * BN + tcol0 + kc * CH), v);
#pragma unroll
                    for (int j = 0; j < CH; ++j) stg[j * kTStageLd + q * 32 + lane] = epi_v(e, r, c0 + j, v[j], 0.0f);
                    named_bar(1 + half);
                    tw_store(e, c0, q, wc, stg, lane, wcur);
                    named_bar(1 + half);  // the chunk is read before the next one is staged
                }
            } else {
            // this warp's 32 x 16 staging slice for diagonal chunks (the
            // transposed-update stage: a launch holds store groups or update
            // groups, never both)
            float* stg = S.tstage[half] + q * (32 * CH);
            // the chunk loop compiled per kind: stores, or the W update
            auto chunks = [&](auto upd_c) {
                constexpr bool kUpd = decltype(upd_c)::value;
                float xin[CH];
                if (nch > 0) epi_load<kUpd>(e, r, r0w, lane, cbase, xin);
                // a wait that gave up skips the tile's work but not the loop: the
                // group then leaves together at the next tile slot (the producer
                // stops publishing once its own waits give up)
                const bool ready = mbar_wait_cluster(&S.acc_full[buf], use & 1, L.status);
                tc_fence_after();
                for (int kc = 0; ready && kc < nch; ++kc) {
                    const int c0 = cbase + kc * CH;
                    float x[CH];
#pragma unroll
                    for (int j = 0; j < CH; ++j) x[j] = xin[j];
                    if (kc + 1 < nch) epi_load<kUpd>(e, r, r0w, lane, c0 + CH, xin);
                    float v[CH];
                    __syncwarp();
                    tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                  static_cast<uint32_t>(buf * BN + tcol0 + kc * CH), v);
                    epi_finish<kSplit, kUpd>(e, r, r0w, lane, c0, v, x, stg);
                }
            };
            chunks(std::integral_constant<bool, kUpd>{});
            }
            // Release the accumulator.  Each tcgen05.ld of it ended with
            // tcgen05.wait::ld before its values were used, so every read of
            // the TMEM columns is complete here; the arrive is relaxed: a
            // release would also wait for this warp's global stores to drain
            // at cluster scope (4-5 % of the step on short-K products), and
            // nothing that reuses the accumulator reads them.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa(saddr(&S.acc_empty[buf]), 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the partner may still read its shared memory
    // (the leader's MMAs) or arrive on its barriers
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

}  // namespace

size_t gemm_tc_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t launch_gemm_tc(const LaunchList& l, int num_sms, cudaStream_t s) {
    if (l.total_tiles <= 0) return cudaSuccess;
    static PerDevice max_pairs_per_device;
    const size_t smem = gemm_tc_smem_bytes();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel waits (griddepcontrol.wait)
    // for the previous kernel before its first global-memory access
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // the shared-memory attribute is set (on both instances), and the resident
    // pairs counted, once per device with that device current
    int max_pairs = 0;
    e = max_pairs_per_device.get(dev, &max_pairs, [&](int* out) {
        cudaError_t r = cudaFuncSetAttribute(gemm_tc_kernel<false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(gemm_tc_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(gemm_tc_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        if (r != cudaSuccess) return r;
        cudaLaunchConfig_t probe = cfg;
        probe.gridDim = dim3(num_sms / kPair * kPair);
        probe.numAttrs = 1;  // the cluster shape alone
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<false, false>, &probe);
        if (r != cudaSuccess) return r;
        *out = n > 0 ? n : num_sms / kPair;
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    const int pairs = l.total_tiles < max_pairs ? l.total_tiles : max_pairs;
    cfg.gridDim = dim3(pairs * kPair);
    // Epilogue layout.  Sets (each group of four warps takes alternate tiles
    // whole) for store launches with at least 8 tiles per pair; column halves
    // otherwise.  Measured: sets 4.5 % faster on 2 000 small matrices and
    // 1.5 % on the Llama-shaped set's Newton-Schulz phases, but 11 % slower on
    // its update launch and 2 % on sets of ~4 tiles per pair.
    LaunchList run = l;
    run.epi_sets = (!l.update && l.total_tiles >= 8 * pairs) ? 1 : 0;
    // three instances: store launches with and without split outputs, update
    // launches (which store nothing, so never split outputs)
    if (l.update) {
        if (l.has_split) return cudaErrorInvalidValue;
        return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<false, true>, run);
    }
    if (l.has_split) return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<true, false>, run);
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<false, false>, run);
}

}  // namespace dmuon
