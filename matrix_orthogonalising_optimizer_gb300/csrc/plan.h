// Host-side plan: shape buckets, waves, workspace layout and launch tables.
#pragma once

#include <cstdint>
#include <map>
#include <string>
#include <vector>

#include "dmuon.h"
#include "internal.h"

namespace dmuon {

enum BufKind : int {
    BUF_X0 = 0,  // packed u (direct route: iterate 0)
    BUF_X1,      // direct route: iterate 1
    BUF_RF,      // fp32 R (Gram) / fp32 A (direct)
    BUF_RB,      // operand R (Gram, tensor cores)
    BUF_P,       // P
    BUF_Q0,
    BUF_Q1,
    BUF_RP,      // R P
    BUF_AB,      // operand A (direct, tensor cores)
    BUF_BB,      // B = bA + cA^2 (direct)
    BUF_PART,    // sum-of-squares partials
    BUF_COUNT
};

struct Bucket {
    int32_t dtype = 0, route = 0, engine = 0, tile = DMUON_TILE_SINGLE;
    int64_t m = 0, n = 0;
    std::vector<int64_t> members;  // input indices, input order
    int64_t pmb = 0;               // per-matrix workspace bytes
    int64_t slot0 = 0;             // first slot (bucket order)
    int64_t buf_bytes[BUF_COUNT] = {};  // per-matrix bytes of each buffer (256-rounded), 0 = absent
    int32_t buf_type[BUF_COUNT] = {};   // ElemType of each buffer
};

struct Piece {
    int64_t bucket = 0, start = 0, count = 0;
    int64_t slot0 = 0;                 // first slot of the piece
    uint64_t off[BUF_COUNT] = {};      // byte offset of each buffer region inside the wave region
    std::vector<int32_t> tmpl;         // template kind -> group index (-1 = none)
};

struct Wave {
    std::vector<Piece> pieces;
    int64_t slot0 = 0, nslots = 0;
    uint64_t bytes = 0;
    int64_t mom_tiles = 0;    // momentum units of all slots (tile pass index)
    int64_t nflat = 0;        // flat slots (listed from the wave's slot0 in the flat table)
    int64_t flat_chunks = 0;  // momentum units of the flat slots (flat pass index)
    bool flat = false;        // the wave runs the flat momentum pass
};

struct Launch {
    int32_t kernel = 0;  // 0 = tcgen05, 1 = fp32 FFMA
    int32_t timer = 0;   // DMUON_TIMER_* of the phase
    LaunchList list{};
};

struct TimedLaunch {
    int32_t slots[2];
    void* ev0;
    void* ev1;
};

struct SlotHost {
    int64_t gidx = 0;
    int32_t rows = 0, cols = 0, transposed = 0, dtype = 0;
    int64_t bucket = 0, wave = 0, piece = 0, j = 0;  // j = index inside the piece
};

}  // namespace dmuon

struct dmuon_plan_s {
    // resolved options
    int32_t precision = DMUON_PREC_BF16;
    int32_t route_rule = DMUON_ROUTE_AUTO;
    float ns_a = 3.4445f, ns_b = -4.7750f, ns_c = 2.0315f;
    float eps = 1e-7f;
    int32_t scale_rule = DMUON_SCALE_ASPECT;
    int32_t nesterov = 1;
    int32_t small_m = 256;
    int32_t tile_rule = DMUON_TILE_PACKED;  // the plan's rule (AUTO resolved)
    uint64_t budget = 0;

    int64_t count = 0;
    std::vector<dmuon_shape_t> shapes;
    std::vector<dmuon::Bucket> buckets;
    std::vector<dmuon::Wave> waves;
    std::vector<dmuon::SlotHost> slots;  // bucket order

    // fixed region layout
    uint64_t off_status = 0, off_scalars = 0, off_infos = 0, off_ptrs = 0, off_groups = 0, off_counters = 0,
             off_flat = 0, off_waves = 0;
    int64_t num_groups = 0;
    uint64_t ws_bytes = 0;

    // bound state
    char* ws = nullptr;
    uint64_t ws_size = 0;
    int device = -1;
    int num_sms = 0;
    std::vector<dmuon::GemmGroup> groups;
    std::vector<int> group_kernel;        // per group: 0 tcgen05, 1 fp32 FFMA
    std::vector<const void*> cached_ptrs;  // params | grads | momenta
    std::map<int, std::vector<std::vector<dmuon::Launch>>> phase_cache;  // ns_steps -> per wave
    bool phase_error = false;              // a launch table broke an invariant (message set)

    // timing
    bool timing = false;
    std::vector<dmuon::TimedLaunch> pending;
    std::vector<void*> event_pool;
    size_t event_next = 0;
    double timer_ms[DMUON_TIMER_COUNT] = {};
    int64_t timer_launches[DMUON_TIMER_COUNT] = {};
};
