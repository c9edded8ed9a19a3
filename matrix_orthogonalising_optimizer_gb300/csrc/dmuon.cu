// C ABI of the batched Gram-space Newton-Schulz Muon step: planner,
// workspace layout, TMA tensor maps, launch tables and the step sequencer.
//
// The per-owner compute of DMuon (gist.science technical summary, section
// 2.2): Newton-Schulz in the m x m Gram space (G = X X^T, m <= n), formed
// SYRK-style, with matrices of like shape batched.  The planner turns a list
// of shapes into buckets (tall matrices transposed), packs buckets into waves
// that fit the workspace, and per wave records one launch per phase of the
// iteration covering every bucket, so launch count does not grow with the
// number of matrices.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "plan.h"

using namespace dmuon;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

uint64_t up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

int esz(int32_t t) { return t == ELEM_BF16 ? 2 : 4; }

// Row length of a split m x m operand [hi | lo]: two parts of m rounded up
// to the 64-deep K slab.
int64_t split_ld(int64_t m) { return 2 * static_cast<int64_t>(up(static_cast<uint64_t>(m), 64)); }

bool split_operand(int k) { return k == BUF_RB || k == BUF_P || k == BUF_Q0 || k == BUF_Q1 || k == BUF_RP; }

// The momentum pass streams a matrix flat when its packed u has the gradient's
// own layout (bf16 storage and operands, not transposed, rows on 16 bytes)
// and it is large enough for its record lookup to be amortised over many
// chunks (2^20 elements); and only in waves where such matrices hold at
// least kFlatWaveMin elements, since a second pass costs a launch and a tail.
// Measured on the Llama-3-8B-shaped set: its wide matrices at 90 % of HBM
// instead of 82 %; on sets of small matrices the extra pass was slower.
constexpr int64_t kFlatMatrixMin = int64_t(1) << 20;
constexpr int64_t kFlatWaveMin = int64_t(1) << 26;

bool flat_momentum(int32_t precision, int32_t dtype, int64_t rows, int64_t cols) {
    return precision == DMUON_PREC_BF16 && dtype == DMUON_BF16 && rows <= cols && cols % 8 == 0 &&
           rows * cols >= kFlatMatrixMin;
}

// Momentum work units of a matrix: chunks of kMomChunk elements (flat) or
// 64 x 64 tiles; either leaves kMomPartials sum-of-squares partials.
int64_t momentum_units(bool flat, int64_t rows, int64_t cols) {
    if (flat) return (rows * cols + kMomChunk - 1) / kMomChunk;
    return ((rows + kMomTile - 1) / kMomTile) * ((cols + kMomTile - 1) / kMomTile);
}

// ------------------------------------------------------------ template kinds

enum Tmpl : int {
    G_SYRK = 0, G_POLY0, G_POLY, G_Q01, G_Q10, G_RP0, G_RP, G_RUPD0, G_RUPD, G_FIN0, G_FIN1,
    D_SYRK0, D_SYRK_X0, D_SYRK_X1, D_A2, D_XUPD0, D_XUPD01, D_XUPD10, D_FIN0I, D_FIN0, D_FIN1,
    TMPL_COUNT
};

constexpr int kKernelTc = 0;
constexpr int kKernelSimt = 1;

// ------------------------------------------------------------ planning

void bucket_buffers(Bucket& b, int32_t precision) {
    const int64_t m = b.m, n = b.n;
    const int64_t ldn = static_cast<int64_t>(up(n, 8)), ldm = static_cast<int64_t>(up(m, 8));
    const int32_t xt = precision == DMUON_PREC_BF16 ? ELEM_BF16 : ELEM_F32;
    auto set = [&](int k, int64_t elems, int32_t t) {
        b.buf_bytes[k] = static_cast<int64_t>(up(static_cast<uint64_t>(elems * esz(t)), 256));
        b.buf_type[k] = t;
    };
    set(BUF_X0, m * ldn, xt);
    if (b.route == DMUON_BUCKET_GRAM) {
        if (b.engine == DMUON_ENGINE_TC_BF16) {
            // bf16 operands only: the polynomial's b R term reads the bf16 R
            // the products read
            for (int k : {BUF_RB, BUF_P, BUF_Q0, BUF_Q1, BUF_RP}) set(k, m * ldm, ELEM_BF16);
        } else if (b.engine == DMUON_ENGINE_TC_SPLIT) {
            // fp32 R (aux of P); split operands [hi | lo], each part a whole
            // number of 64-deep K slabs
            set(BUF_RF, m * ldm, ELEM_F32);
            for (int k : {BUF_RB, BUF_P, BUF_Q0, BUF_Q1, BUF_RP}) set(k, m * split_ld(m), ELEM_BF16);
        } else {
            // fp32 FFMA engine (the fp32 mode)
            for (int k : {BUF_RF, BUF_P, BUF_Q0, BUF_Q1, BUF_RP}) set(k, m * ldm, ELEM_F32);
        }
    } else {
        set(BUF_X1, m * ldn, xt);
        if (precision == DMUON_PREC_BF16) {  // bf16 A only: B's b A term reads it too
            set(BUF_AB, m * ldm, ELEM_BF16);
            set(BUF_BB, m * ldm, ELEM_BF16);
        } else {
            set(BUF_RF, m * ldm, ELEM_F32);
            set(BUF_BB, m * ldm, ELEM_F32);
        }
    }
    b.buf_bytes[BUF_PART] = static_cast<int64_t>(up(4 * kMomPartials * ((m + 63) / 64) * ((n + 63) / 64), 256));
    b.buf_type[BUF_PART] = ELEM_F32;
    b.pmb = 0;
    for (int k = 0; k < BUF_COUNT; ++k) b.pmb += b.buf_bytes[k];
}

float shape_scale(int32_t rule, int64_t rows, int64_t cols) {
    if (rule == DMUON_SCALE_RMS)
        return static_cast<float>(0.2 * std::sqrt(static_cast<double>(std::max(rows, cols))));
    return static_cast<float>(std::sqrt(std::max(1.0, static_cast<double>(rows) / static_cast<double>(cols))));
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
    if (g_encode) return DMUON_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return DMUON_OK;
}

// bf16 rank-3 view {dim0 (contiguous), dim1, batch}, 128-byte swizzle.
int encode_bf16(CUtensorMap* map, const void* base, int64_t dim0, int64_t dim1, int64_t batch, int64_t ld,
                int64_t bs, uint32_t box0, uint32_t box1, uint32_t box2) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(dim0), static_cast<cuuint64_t>(dim1),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(bs * 2)};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DMUON_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string(r) + ")");
    return DMUON_OK;
}

struct Operand {
    const void* p = nullptr;
    int32_t type = ELEM_BF16;
    int64_t ld = 0, bs = 0;  // elements
};

struct GroupSpec {
    int kernel = kKernelTc;
    Operand a, b;
    int64_t M = 0, N = 0, K = 0, batch = 0;
    int64_t kseg = 0;        // K segments (split operands); 0 = none
    int64_t a_k = 0, b_k = 0;  // K extent of A's / B's tensor map when it differs from K
    bool b_mn = false, sym = false;
    int32_t mode = EPI_STORE, alpha = ALPHA_ONE;
    float c_acc = 1.0f, c_diag = 0.0f, c_aux = 0.0f;
    Operand aux;
    bool aux_sym = false;
    Operand out[3];
    bool out_lower_only[3] = {false, false, false};  // symmetric D: skip the mirror of this output
    int64_t out_lo[3] = {0, 0, 0};                  // split bf16 output: offset of the low parts
    int64_t slot_base = 0;
};

int build_group(const GroupSpec& s, GemmGroup* g, int32_t tile) {
    std::memset(g, 0, sizeof(*g));
    g->a = s.a.p;
    g->b = s.b.p;
    g->a_bs = s.a.bs;
    g->b_bs = s.b.bs;
    g->lda = static_cast<int32_t>(s.a.ld);
    g->ldb = static_cast<int32_t>(s.b.ld);
    g->a_type = s.a.type;
    g->b_type = s.b.type;
    g->M = static_cast<int32_t>(s.M);
    g->N = static_cast<int32_t>(s.N);
    g->K = static_cast<int32_t>(s.K);
    g->batch = static_cast<int32_t>(s.batch);
    g->b_mn_major = s.b_mn ? 1 : 0;
    g->kseg = static_cast<int32_t>(s.kseg);
    g->sym = s.sym ? 1 : 0;
    g->slot_base = static_cast<int32_t>(s.slot_base);
    g->mode = s.mode;
    g->alpha_sel = s.alpha;
    g->c_acc = s.c_acc;
    g->c_diag = s.c_diag;
    g->c_aux = s.c_aux;
    g->aux = s.aux.p;
    g->aux_type = s.aux.type;
    g->aux_ld = static_cast<int32_t>(s.aux.ld);
    g->aux_bs = s.aux.bs;
    g->aux_sym = s.aux_sym ? 1 : 0;
    for (int o = 0; o < 3; ++o) {
        g->out[o] = const_cast<void*>(s.out[o].p);
        g->out_type[o] = s.out[o].type;
        g->out_ld[o] = static_cast<int32_t>(s.out[o].ld);
        g->out_bs[o] = s.out[o].bs;
        g->out_mirror[o] = s.sym && !s.out_lower_only[o] ? 1 : 0;
        g->out_lo[o] = static_cast<int32_t>(s.out_lo[o]);
    }
    g->pack = 1;
    if (s.kernel == kKernelTc) {
        // pair tiles: 256 rows (two CTAs of 128) x 256 columns
        const int64_t pair_rows = kTcPair * kTcBM;
        g->tiles_m = static_cast<int32_t>((s.M + pair_rows - 1) / pair_rows);
        g->tiles_n = static_cast<int32_t>((s.N + kTcBN - 1) / kTcBN);
        if (s.sym) {
            g->tiles_per_mat = g->tiles_m * (g->tiles_m + 1) / 2;
        } else {
            g->tiles_per_mat = g->tiles_m * g->tiles_n;
        }
        // small symmetric products: several matrices block-diagonally per tile
        if (s.sym && tile == DMUON_TILE_PACKED && s.M <= kTcBM) g->pack = s.M <= kTcBM / 2 ? 4 : 2;
        if (s.a.type != ELEM_BF16 || s.b.type != ELEM_BF16)
            return fail(DMUON_ERR_INVALID_ARG, "internal: tensor-core operands must be bf16");
        const int64_t ak = s.a_k ? s.a_k : s.K, bk = s.b_k ? s.b_k : s.K;
        // a CTA's 128 rows of A (and of K-major B): one matrix's rows, or two
        // 64-row matrices of a tile packed by four
        const uint32_t rows = g->pack == 4 ? kTcBM / 2 : kTcBM, mats = g->pack == 4 ? 2 : 1;
        int rc = encode_bf16(&g->tma_a, s.a.p, ak, s.M, s.batch, s.a.ld, s.a.bs, kTcSlabBytes / 2, rows, mats);
        if (rc) return rc;
        if (!s.b_mn)
            rc = encode_bf16(&g->tma_b, s.b.p, bk, s.N, s.batch, s.b.ld, s.b.bs, kTcSlabBytes / 2,
                             g->pack > 1 ? rows : kTcBN / kTcPair, mats);
        else
            rc = encode_bf16(&g->tma_b, s.b.p, s.N, bk, s.batch, s.b.ld, s.b.bs, 64, kTcSlabBytes / 2, 1);
        if (rc) return rc;
    } else {
        g->tiles_m = static_cast<int32_t>((s.M + kSimtBM - 1) / kSimtBM);
        g->tiles_n = static_cast<int32_t>((s.N + kSimtBN - 1) / kSimtBN);
        g->tiles_per_mat = s.sym ? g->tiles_m * (g->tiles_m + 1) / 2 : g->tiles_m * g->tiles_n;
    }
    g->ntiles = g->pack > 1 ? static_cast<int32_t>((s.batch + g->pack - 1) / g->pack)
                            : static_cast<int32_t>(g->tiles_per_mat * s.batch);
    return DMUON_OK;
}

// ------------------------------------------------------------ timing

void* take_event(dmuon_plan_s* h) {
    if (h->event_next == h->event_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        h->event_pool.push_back(e);
    }
    return h->event_pool[h->event_next++];
}

template <typename F>
cudaError_t timed(dmuon_plan_s* h, cudaStream_t s, int slot0, int slot1, F&& launch) {
    if (!h->timing) return launch();
    void* e0 = take_event(h);
    void* e1 = take_event(h);
    if (!e0 || !e1) return launch();
    cudaEventRecord(static_cast<cudaEvent_t>(e0), s);
    cudaError_t r = launch();
    cudaEventRecord(static_cast<cudaEvent_t>(e1), s);
    h->pending.push_back(TimedLaunch{{slot0, slot1}, e0, e1});
    return r;
}

int collect_timing(dmuon_plan_s* h) {
    for (const TimedLaunch& t : h->pending) {
        if (cudaEventSynchronize(static_cast<cudaEvent_t>(t.ev1)) != cudaSuccess)
            return fail(DMUON_ERR_CUDA, "event synchronise failed");
        float ms = 0.0f;
        cudaEventElapsedTime(&ms, static_cast<cudaEvent_t>(t.ev0), static_cast<cudaEvent_t>(t.ev1));
        for (int k = 0; k < 2; ++k) {
            if (t.slots[k] < 0) continue;
            h->timer_ms[t.slots[k]] += ms;
            h->timer_launches[t.slots[k]] += 1;
        }
    }
    h->pending.clear();
    h->event_next = 0;
    return DMUON_OK;
}

// ------------------------------------------------------------ phases

std::vector<std::vector<int>> gram_sequence(int T) {
    std::vector<std::vector<int>> seq;
    seq.push_back({G_SYRK});
    for (int k = 0; k < T; ++k) {
        seq.push_back({k == 0 ? G_POLY0 : G_POLY});
        std::vector<int> mid;
        if (k >= 1) mid.push_back((k - 1) % 2 == 0 ? G_Q01 : G_Q10);
        if (k < T - 1) mid.push_back(k == 0 ? G_RP0 : G_RP);
        if (!mid.empty()) seq.push_back(mid);
        if (k < T - 1) seq.push_back({k == 0 ? G_RUPD0 : G_RUPD});
    }
    seq.push_back({(T - 1) % 2 == 0 ? G_FIN0 : G_FIN1});
    return seq;
}

std::vector<std::vector<int>> direct_sequence(int T) {
    std::vector<std::vector<int>> seq;
    for (int k = 0; k < T; ++k) {
        const int src = k % 2;
        seq.push_back({k == 0 ? D_SYRK0 : (src == 0 ? D_SYRK_X0 : D_SYRK_X1)});
        seq.push_back({D_A2});
        if (k < T - 1) seq.push_back({k == 0 ? D_XUPD0 : (src == 0 ? D_XUPD01 : D_XUPD10)});
        else seq.push_back({k == 0 ? D_FIN0I : (src == 0 ? D_FIN0 : D_FIN1)});
    }
    return seq;
}

}  // namespace

namespace dmuon {
// The calling thread's error message, also for the other translation units.
void set_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace dmuon

static const std::vector<std::vector<Launch>>& launches_for(dmuon_plan_s* h, int T) {
    auto it = h->phase_cache.find(T);
    if (it != h->phase_cache.end()) return it->second;
    std::vector<std::vector<Launch>> per_wave;
    const std::vector<int>& gk = h->group_kernel;
    for (const Wave& w : h->waves) {
        std::vector<std::vector<std::vector<int>>> seqs;
        size_t L = 0;
        for (const Piece& p : w.pieces) {
            const Bucket& b = h->buckets[p.bucket];
            seqs.push_back(b.route == DMUON_BUCKET_GRAM ? gram_sequence(T) : direct_sequence(T));
            L = std::max(L, seqs.back().size());
        }
        std::vector<Launch> launches;
        for (size_t ph = 0; ph < L; ++ph) {
            std::vector<int> by_kernel[2];
            for (size_t pi = 0; pi < w.pieces.size(); ++pi) {
                const auto& seq = seqs[pi];
                const size_t shift = L - seq.size();
                if (ph < shift) continue;
                for (int tk : seq[ph - shift]) {
                    const int gi = w.pieces[pi].tmpl[tk];
                    if (gi >= 0) by_kernel[gk[gi]].push_back(gi);
                }
            }
            const int timer = ph == 0 ? DMUON_TIMER_SYRK : (ph == L - 1 ? DMUON_TIMER_FINAL : DMUON_TIMER_NS);
            for (int kern = 0; kern < 2; ++kern) {
                std::vector<int>& gs = by_kernel[kern];
                if (gs.empty()) continue;
                std::stable_sort(gs.begin(), gs.end(), [&](int x, int y) { return h->groups[x].K > h->groups[y].K; });
                for (size_t s0 = 0; s0 < gs.size(); s0 += kMaxGroupsPerLaunch) {
                    Launch la;
                    la.kernel = kern;
                    la.timer = timer;
                    LaunchList& l = la.list;
                    std::memset(&l, 0, sizeof(l));
                    const size_t e = std::min(gs.size(), s0 + kMaxGroupsPerLaunch);
                    int64_t tiles = 0;
                    for (size_t j = s0; j < e; ++j) {
                        const GemmGroup& g = h->groups[gs[j]];
                        l.idx[l.n] = gs[j];
                        l.begin[l.n] = static_cast<int32_t>(tiles);
                        if (g.out_lo[0] | g.out_lo[1] | g.out_lo[2]) l.has_split = 1;
                        tiles += g.ntiles;
                        ++l.n;
                    }
                    l.begin[l.n] = static_cast<int32_t>(tiles);
                    l.total_tiles = static_cast<int32_t>(tiles);
                    l.update = l.n > 0 && h->groups[l.idx[0]].mode == EPI_UPDATE ? 1 : 0;
                    // the tcgen05 kernel's shared stage serves the transposed
                    // update or diagonal store chunks: never both in one launch
                    for (int j = 1; j < l.n; ++j)
                        if (h->groups[l.idx[j]].mode != h->groups[l.idx[0]].mode) {
                            fail(DMUON_ERR_INVALID_ARG, "internal: a launch mixes update and store products");
                            h->phase_error = true;
                        }
                    char* ws = h->ws;
                    l.groups = reinterpret_cast<const GemmGroup*>(ws + h->off_groups);
                    l.infos = reinterpret_cast<const MatInfo*>(ws + h->off_infos);
                    l.scalars = reinterpret_cast<const SlotScalars*>(ws + h->off_scalars);
                    l.params = reinterpret_cast<void* const*>(ws + h->off_ptrs);
                    l.status = reinterpret_cast<int32_t*>(ws + h->off_status);
                    if (launches.size() < static_cast<size_t>(kMaxLaunchesPerWave))
                        l.counter = reinterpret_cast<int32_t*>(ws + h->off_counters) + launches.size();
                    launches.push_back(la);
                }
            }
        }
        per_wave.push_back(std::move(launches));
    }
    return h->phase_cache.emplace(T, std::move(per_wave)).first->second;
}

// ============================================================ C ABI

extern "C" {

const char* dmuon_last_error(void) { return g_last_error.c_str(); }

const char* dmuon_status_string(int status) {
    switch (status) {
        case DMUON_OK: return "ok";
        case DMUON_ERR_INVALID_ARG: return "invalid argument";
        case DMUON_ERR_ALIGN: return "pointer not 16-byte aligned";
        case DMUON_ERR_NO_WORKSPACE: return "no workspace bound";
        case DMUON_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case DMUON_ERR_CUDA: return "CUDA error";
        case DMUON_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case DMUON_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
        case DMUON_ERR_WORKSPACE_TOO_SMALL: return "workspace too small or misaligned";
        default: return "unknown status";
    }
}

dmuon_handle_t dmuon_plan_ex(const dmuon_shape_t* shapes, int64_t count, const dmuon_options_t* opt) {
    if (!shapes || count < 1) {
        fail(DMUON_ERR_INVALID_ARG, "shapes must be non-NULL and count >= 1");
        return nullptr;
    }
    dmuon_options_t o;
    std::memset(&o, 0, sizeof(o));
    if (opt) o = *opt;
    if (o.precision != DMUON_PREC_BF16 && o.precision != DMUON_PREC_FP32) {
        fail(DMUON_ERR_INVALID_ARG, "unknown precision mode");
        return nullptr;
    }
    if (o.route < DMUON_ROUTE_AUTO || o.route > DMUON_ROUTE_DIRECT) {
        fail(DMUON_ERR_INVALID_ARG, "unknown route rule");
        return nullptr;
    }
    if (o.scale_rule != DMUON_SCALE_ASPECT && o.scale_rule != DMUON_SCALE_RMS) {
        fail(DMUON_ERR_INVALID_ARG, "unknown scale rule");
        return nullptr;
    }
    if (!(o.eps >= 0.0f) || !std::isfinite(o.eps) || !std::isfinite(o.ns_a) || !std::isfinite(o.ns_b) ||
        !std::isfinite(o.ns_c) || (o.no_nesterov != 0 && o.no_nesterov != 1) ||
        o.tile_rule < DMUON_TILE_AUTO || o.tile_rule > DMUON_TILE_SINGLE) {
        fail(DMUON_ERR_INVALID_ARG, "bad option values");
        return nullptr;
    }
    auto* h = new dmuon_plan_s();
    h->precision = o.precision;
    h->route_rule = o.route;
    if (o.ns_a != 0.0f || o.ns_b != 0.0f || o.ns_c != 0.0f) {
        h->ns_a = o.ns_a;
        h->ns_b = o.ns_b;
        h->ns_c = o.ns_c;
    }
    if (o.eps != 0.0f) h->eps = o.eps;
    h->scale_rule = o.scale_rule;
    h->nesterov = o.no_nesterov ? 0 : 1;
    h->small_m = o.small_m == 0 ? 256 : o.small_m;
    h->tile_rule = o.tile_rule == DMUON_TILE_AUTO ? DMUON_TILE_PACKED : o.tile_rule;
    h->budget = o.workspace_budget;
    h->count = count;
    h->shapes.assign(shapes, shapes + count);

    // route of one matrix: its own rule, else the plan's; AUTO by shape
    auto resolve = [&](int32_t rule, int64_t m, int64_t n) {
        const bool small = h->small_m > 0 && m <= h->small_m;
        if (h->precision == DMUON_PREC_FP32) return rule == DMUON_ROUTE_DIRECT ? DMUON_BUCKET_DIRECT : DMUON_BUCKET_GRAM;
        if (rule == DMUON_ROUTE_GRAM) return DMUON_BUCKET_GRAM;
        if (rule == DMUON_ROUTE_DIRECT) return DMUON_BUCKET_DIRECT;
        return (n >= 3 * m || small) ? DMUON_BUCKET_GRAM : DMUON_BUCKET_DIRECT;
    };
    // tile rule of one matrix: its own, else the plan's; SINGLE where packing
    // does not apply
    auto resolve_tile = [&](int32_t own, int64_t m) {
        if (h->precision == DMUON_PREC_FP32 || m > kTcBM) return static_cast<int32_t>(DMUON_TILE_SINGLE);
        return own != DMUON_TILE_AUTO ? own : h->tile_rule;
    };
    std::map<std::tuple<int32_t, int64_t, int64_t, int32_t, int32_t>, std::vector<int64_t>> keyed;
    for (int64_t i = 0; i < count; ++i) {
        const dmuon_shape_t& s = shapes[i];
        if (s.rows < 1 || s.cols < 1 || s.rows > DMUON_MAX_DIM || s.cols > DMUON_MAX_DIM ||
            s.rows * s.cols >= DMUON_MAX_ELEMS || s.route < DMUON_ROUTE_AUTO || s.route > DMUON_ROUTE_DIRECT ||
            s.tile < DMUON_TILE_AUTO || s.tile > DMUON_TILE_SINGLE || s.reserved != 0) {
            fail(DMUON_ERR_INVALID_ARG, "shape " + std::to_string(i) + " out of range");
            delete h;
            return nullptr;
        }
        if (s.dtype != DMUON_BF16 && s.dtype != DMUON_FP32) {
            fail(DMUON_ERR_UNSUPPORTED_DTYPE, "shape " + std::to_string(i) + ": unknown dtype");
            delete h;
            return nullptr;
        }
        const int64_t m = std::min(s.rows, s.cols), n = std::max(s.rows, s.cols);
        const int32_t rule = s.route != DMUON_ROUTE_AUTO ? s.route : h->route_rule;
        keyed[std::make_tuple(s.dtype, m, n, static_cast<int32_t>(resolve(rule, m, n)), resolve_tile(s.tile, m))]
            .push_back(i);
    }
    int64_t slot = 0;
    for (auto& kv : keyed) {
        Bucket b;
        b.dtype = std::get<0>(kv.first);
        b.m = std::get<1>(kv.first);
        b.n = std::get<2>(kv.first);
        b.members = kv.second;
        const bool small = h->small_m > 0 && b.m <= h->small_m;
        b.route = std::get<3>(kv.first);
        b.tile = std::get<4>(kv.first);
        if (h->precision == DMUON_PREC_FP32) b.engine = DMUON_ENGINE_SIMT_FP32;
        else if (b.route == DMUON_BUCKET_GRAM && small) b.engine = DMUON_ENGINE_TC_SPLIT;
        else b.engine = DMUON_ENGINE_TC_BF16;
        bucket_buffers(b, h->precision);
        b.slot0 = slot;
        for (size_t j = 0; j < b.members.size(); ++j) {
            SlotHost sh;
            sh.gidx = b.members[j];
            const dmuon_shape_t& s = shapes[sh.gidx];
            sh.rows = static_cast<int32_t>(s.rows);
            sh.cols = static_cast<int32_t>(s.cols);
            sh.transposed = s.rows > s.cols ? 1 : 0;
            sh.dtype = s.dtype == DMUON_BF16 ? ELEM_BF16 : ELEM_F32;
            sh.bucket = static_cast<int64_t>(h->buckets.size());
            h->slots.push_back(sh);
        }
        slot += static_cast<int64_t>(b.members.size());
        h->buckets.push_back(std::move(b));
    }

    // waves
    std::vector<std::vector<std::tuple<int64_t, int64_t, int64_t>>> waves;
    if (h->budget == 0) {
        waves.emplace_back();
        for (size_t b = 0; b < h->buckets.size(); ++b)
            waves.back().emplace_back(static_cast<int64_t>(b), 0, static_cast<int64_t>(h->buckets[b].members.size()));
    } else {
        std::vector<std::tuple<int64_t, int64_t, int64_t>> cur;
        uint64_t used = 0;
        for (size_t b = 0; b < h->buckets.size(); ++b) {
            const uint64_t pmb = static_cast<uint64_t>(h->buckets[b].pmb);
            if (pmb > h->budget) {
                fail(DMUON_ERR_INVALID_ARG, "workspace budget smaller than one matrix of bucket " + std::to_string(b));
                delete h;
                return nullptr;
            }
            int64_t start = 0, left = static_cast<int64_t>(h->buckets[b].members.size());
            while (left > 0) {
                const int64_t fit = static_cast<int64_t>((h->budget - used) / pmb);
                if (fit == 0) {
                    waves.push_back(cur);
                    cur.clear();
                    used = 0;
                    continue;
                }
                const int64_t take = std::min(fit, left);
                cur.emplace_back(static_cast<int64_t>(b), start, take);
                used += static_cast<uint64_t>(take) * pmb;
                start += take;
                left -= take;
            }
        }
        if (!cur.empty()) waves.push_back(cur);
    }

    int64_t ngroups = 0;
    uint64_t max_wave = 0;
    for (size_t wi = 0; wi < waves.size(); ++wi) {
        Wave w;
        uint64_t cur = 0;
        int64_t tiles = 0, flat_elems = 0;
        for (size_t pi = 0; pi < waves[wi].size(); ++pi) {
            Piece p;
            std::tie(p.bucket, p.start, p.count) = waves[wi][pi];
            const Bucket& b = h->buckets[p.bucket];
            p.slot0 = b.slot0 + p.start;
            for (int k = 0; k < BUF_COUNT; ++k) {
                if (!b.buf_bytes[k]) continue;
                p.off[k] = cur;
                cur += static_cast<uint64_t>(p.count) * static_cast<uint64_t>(b.buf_bytes[k]);
            }
            for (int64_t j = 0; j < p.count; ++j) {
                SlotHost& sh = h->slots[p.slot0 + j];
                sh.wave = static_cast<int64_t>(wi);
                sh.piece = static_cast<int64_t>(pi);
                sh.j = j;
                if (flat_momentum(h->precision, shapes[sh.gidx].dtype, sh.rows, sh.cols))
                    flat_elems += static_cast<int64_t>(sh.rows) * sh.cols;
            }
            ngroups += b.route == DMUON_BUCKET_GRAM ? 11 : 10;
            w.pieces.push_back(p);
        }
        w.slot0 = w.pieces.front().slot0;
        w.nslots = 0;
        for (const Piece& p : w.pieces) w.nslots += p.count;
        w.flat = flat_elems >= kFlatWaveMin;
        for (int64_t s = w.slot0; s < w.slot0 + w.nslots; ++s) {
            const SlotHost& sh = h->slots[s];
            const bool fl = w.flat && flat_momentum(h->precision, shapes[sh.gidx].dtype, sh.rows, sh.cols);
            tiles += momentum_units(fl, sh.rows, sh.cols);
        }
        w.bytes = cur;
        w.mom_tiles = tiles;
        max_wave = std::max(max_wave, cur);
        h->waves.push_back(std::move(w));
    }
    h->num_groups = ngroups;
    const uint64_t nslots = static_cast<uint64_t>(h->slots.size());
    h->off_status = 0;
    h->off_scalars = 256;
    h->off_infos = h->off_scalars + up(nslots * sizeof(SlotScalars), 256);
    h->off_ptrs = h->off_infos + up(nslots * sizeof(MatInfo), 256);
    h->off_groups = h->off_ptrs + up(3 * static_cast<uint64_t>(count) * sizeof(void*), 256);
    h->off_counters = h->off_groups + up(static_cast<uint64_t>(ngroups) * sizeof(GemmGroup), 256);
    h->off_flat = h->off_counters + up(kMaxLaunchesPerWave * sizeof(int32_t), 256);
    h->off_waves = h->off_flat + up(nslots * sizeof(int32_t), 256);
    h->ws_bytes = h->off_waves + max_wave;
    return h;
}

dmuon_handle_t dmuon_plan(const dmuon_shape_t* shapes, int64_t count) { return dmuon_plan_ex(shapes, count, nullptr); }

void dmuon_destroy(dmuon_handle_t h) {
    if (!h) return;
    for (void* e : h->event_pool) cudaEventDestroy(static_cast<cudaEvent_t>(e));
    delete h;
}

int64_t dmuon_plan_num_buckets(dmuon_handle_t h) { return h ? static_cast<int64_t>(h->buckets.size()) : -1; }

int dmuon_plan_bucket(dmuon_handle_t h, int64_t i, dmuon_bucket_info_t* out) {
    if (!h || !out || i < 0 || i >= static_cast<int64_t>(h->buckets.size()))
        return fail(DMUON_ERR_INVALID_ARG, "bad bucket query");
    const Bucket& b = h->buckets[i];
    std::memset(out, 0, sizeof(*out));
    out->dtype = b.dtype;
    out->route = b.route;
    out->mm_engine = b.engine;
    out->tile = b.tile;
    out->m = b.m;
    out->n = b.n;
    out->count = static_cast<int64_t>(b.members.size());
    out->per_matrix_bytes = b.pmb;
    return DMUON_OK;
}

int dmuon_plan_bucket_members(dmuon_handle_t h, int64_t i, int64_t* out) {
    if (!h || !out || i < 0 || i >= static_cast<int64_t>(h->buckets.size()))
        return fail(DMUON_ERR_INVALID_ARG, "bad bucket query");
    const Bucket& b = h->buckets[i];
    std::copy(b.members.begin(), b.members.end(), out);
    return DMUON_OK;
}

int64_t dmuon_plan_num_waves(dmuon_handle_t h) { return h ? static_cast<int64_t>(h->waves.size()) : -1; }

int64_t dmuon_plan_wave_num_pieces(dmuon_handle_t h, int64_t w) {
    if (!h || w < 0 || w >= static_cast<int64_t>(h->waves.size())) return -1;
    return static_cast<int64_t>(h->waves[w].pieces.size());
}

int dmuon_plan_wave_piece(dmuon_handle_t h, int64_t w, int64_t p, int64_t* bucket, int64_t* start, int64_t* count) {
    if (!h || w < 0 || w >= static_cast<int64_t>(h->waves.size()) || p < 0 ||
        p >= static_cast<int64_t>(h->waves[w].pieces.size()) || !bucket || !start || !count)
        return fail(DMUON_ERR_INVALID_ARG, "bad wave query");
    const Piece& pc = h->waves[w].pieces[p];
    *bucket = pc.bucket;
    *start = pc.start;
    *count = pc.count;
    return DMUON_OK;
}

int dmuon_plan_flops(dmuon_handle_t h, int32_t ns_steps, double* out) {
    if (!h || !out || ns_steps < 1 || ns_steps > DMUON_MAX_NS_STEPS)
        return fail(DMUON_ERR_INVALID_ARG, "bad flops query");
    double total = 0.0, tc = 0.0;
    const double T = ns_steps;
    for (const Bucket& b : h->buckets) {
        const double m = static_cast<double>(b.m), n = static_cast<double>(b.n);
        const double cnt = static_cast<double>(b.members.size());
        double rect, cube;
        if (b.route == DMUON_BUCKET_GRAM) {
            rect = 3.0 * m * m * n;
            cube = (4.0 * T - 3.0) * m * m * m;
        } else {
            rect = T * 3.0 * m * m * n;
            cube = T * m * m * m;
        }
        total += cnt * (rect + cube);
        if (h->precision == DMUON_PREC_BF16) tc += cnt * (rect + (b.engine != DMUON_ENGINE_SIMT_FP32 ? cube : 0.0));
    }
    out[0] = total;
    out[1] = tc;
    return DMUON_OK;
}

int dmuon_plan_matrix_flops(dmuon_handle_t h, int32_t ns_steps, double* flops) {
    if (!h || !flops || ns_steps < 1 || ns_steps > DMUON_MAX_NS_STEPS)
        return fail(DMUON_ERR_INVALID_ARG, "bad per-matrix flops query");
    const double T = ns_steps;
    for (const Bucket& b : h->buckets) {
        const double m = static_cast<double>(b.m), n = static_cast<double>(b.n);
        const double f = b.route == DMUON_BUCKET_GRAM ? 3.0 * m * m * n + (4.0 * T - 3.0) * m * m * m
                                                      : T * (3.0 * m * m * n + m * m * m);
        for (int64_t gi : b.members) flops[gi] = f;
    }
    return DMUON_OK;
}

size_t dmuon_workspace_bytes(dmuon_handle_t h) { return h ? static_cast<size_t>(h->ws_bytes) : 0; }

int dmuon_bind_workspace(dmuon_handle_t h, void* dev_ptr, size_t bytes) {
    if (!h) return fail(DMUON_ERR_INVALID_ARG, "NULL handle");
    if (!dev_ptr || (reinterpret_cast<uintptr_t>(dev_ptr) & 255) != 0 || bytes < h->ws_bytes)
        return fail(DMUON_ERR_WORKSPACE_TOO_SMALL, "workspace must be 256-byte aligned and at least " +
                                                       std::to_string(h->ws_bytes) + " bytes");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(DMUON_ERR_CUDA, "no CUDA device");
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3)
        return fail(DMUON_ERR_UNSUPPORTED_DEVICE, "device is sm_" + std::to_string(major * 10 + minor) +
                                                      ", the kernels are built for sm_103a");
    int rc = get_encoder();
    if (rc) return rc;
    h->ws = static_cast<char*>(dev_ptr);
    h->ws_size = bytes;
    h->device = dev;
    h->num_sms = sms;
    h->phase_cache.clear();
    h->cached_ptrs.clear();

    char* ws = h->ws;
    char* wbase = ws + h->off_waves;
    auto buf = [&](const Piece& p, int k) -> Operand {
        const Bucket& b = h->buckets[p.bucket];
        Operand o;
        if (!b.buf_bytes[k]) return o;
        o.p = wbase + p.off[k];
        o.type = b.buf_type[k];
        o.bs = b.buf_bytes[k] / esz(o.type);
        const bool mm = !(k == BUF_X0 || k == BUF_X1 || k == BUF_PART);
        o.ld = static_cast<int64_t>(up(static_cast<uint64_t>(mm ? b.m : b.n), 8));
        if (b.engine == DMUON_ENGINE_TC_SPLIT && split_operand(k)) o.ld = split_ld(b.m);
        return o;
    };

    // per-slot info
    std::vector<MatInfo> infos(h->slots.size());
    for (size_t s = 0; s < h->slots.size(); ++s) {
        const SlotHost& sh = h->slots[s];
        const Piece& p = h->waves[sh.wave].pieces[sh.piece];
        const Bucket& b = h->buckets[sh.bucket];
        MatInfo& mi = infos[s];
        std::memset(&mi, 0, sizeof(mi));
        const Operand x = buf(p, BUF_X0);
        mi.x = const_cast<char*>(static_cast<const char*>(x.p)) + sh.j * b.buf_bytes[BUF_X0];
        mi.partials = reinterpret_cast<float*>(wbase + p.off[BUF_PART] + sh.j * b.buf_bytes[BUF_PART]);
        mi.ldx = x.ld;
        mi.gidx = sh.gidx;
        mi.rows = sh.rows;
        mi.cols = sh.cols;
        mi.tiles_c = (sh.cols + 63) / 64;
        mi.flat = h->waves[sh.wave].flat && flat_momentum(h->precision, h->shapes[sh.gidx].dtype, sh.rows, sh.cols);
        mi.ntiles = static_cast<int32_t>(momentum_units(mi.flat != 0, sh.rows, sh.cols));
        mi.transposed = sh.transposed;
        mi.dtype = sh.dtype;
        mi.x_type = x.type;
        mi.scale = shape_scale(h->scale_rule, sh.rows, sh.cols);
    }
    // per wave: the tile pass's index over all slots, the flat pass's over
    // the flat slots (listed, wave-relative, in the flat table)
    std::vector<int32_t> flat_list(h->slots.size());
    for (Wave& w : h->waves) {
        int64_t t = 0, f = 0;
        w.nflat = 0;
        for (int64_t s = w.slot0; s < w.slot0 + w.nslots; ++s) {
            infos[s].tile_begin = t;
            t += infos[s].ntiles;
            if (infos[s].flat) {
                infos[s].flat_begin = f;
                f += infos[s].ntiles;
                flat_list[w.slot0 + w.nflat++] = static_cast<int32_t>(s - w.slot0);
            }
        }
        w.flat_chunks = f;
    }

    // launch templates
    h->groups.assign(static_cast<size_t>(h->num_groups), GemmGroup{});
    std::vector<int>& gk = h->group_kernel;
    gk.assign(static_cast<size_t>(h->num_groups), kKernelTc);
    int64_t next = 0;
    const bool bf16 = h->precision == DMUON_PREC_BF16;
    for (Wave& w : h->waves) {
        for (Piece& p : w.pieces) {
            const Bucket& b = h->buckets[p.bucket];
            p.tmpl.assign(TMPL_COUNT, -1);
            const int64_t m = b.m, n = b.n;
            const int eng = b.engine == DMUON_ENGINE_SIMT_FP32 ? kKernelSimt : kKernelTc;
            // split engine: every m x m operand stored [hi | lo] (parts of sp
            // elements); an m x m product runs over K = 3 sp, the final over 2 sp
            const bool split = b.engine == DMUON_ENGINE_TC_SPLIT;
            const int64_t sp = split ? split_ld(m) / 2 : 0;
            auto add = [&](int kind, GroupSpec s) -> int {
                s.batch = p.count;
                s.slot_base = p.slot0;
                const int rc2 = build_group(s, &h->groups[next], b.tile);
                if (rc2) return rc2;
                gk[next] = s.kernel;
                p.tmpl[kind] = static_cast<int32_t>(next++);
                return DMUON_OK;
            };
            auto sym_spec = [&](int kernel, Operand a, Operand bb) {
                GroupSpec s;
                s.kernel = kernel;
                s.a = a;
                s.b = bb;
                s.M = m;
                s.N = m;
                s.K = m;
                s.sym = true;
                if (split) {
                    s.K = 3 * sp;
                    s.kseg = sp;
                    s.a_k = s.b_k = 2 * sp;
                }
                return s;
            };
            // split engine: the bf16 m x m outputs are stored [hi | lo]
            auto split_outputs = [&](GroupSpec& s) {
                if (!split) return;
                for (int o = 0; o < 3; ++o)
                    if (s.out[o].p && s.out[o].type == ELEM_BF16) s.out_lo[o] = sp;
            };
            if (b.route == DMUON_BUCKET_GRAM) {
                const Operand X0 = buf(p, BUF_X0), RF = buf(p, BUF_RF), RB = buf(p, BUF_RB), P = buf(p, BUF_P),
                              Q0 = buf(p, BUF_Q0), Q1 = buf(p, BUF_Q1), RP = buf(p, BUF_RP);
                const Operand Rop = eng == kKernelTc ? RB : RF;
                {  // R0 = inv^2 X X^T
                    GroupSpec s;
                    s.kernel = bf16 ? kKernelTc : kKernelSimt;
                    s.a = X0;
                    s.b = X0;
                    s.M = m;
                    s.N = m;
                    s.K = n;
                    s.sym = true;
                    s.alpha = ALPHA_INV2;
                    if (split) {
                        s.out[0] = RF;
                        s.out_lower_only[0] = true;  // fp32 R: only the next P's aux, lower triangle
                        s.out[1] = RB;
                    } else {
                        s.out[0] = eng == kKernelTc ? RB : RF;
                    }
                    split_outputs(s);
                    if ((rc = add(G_SYRK, s))) return rc;
                }
                for (int first = 1; first >= 0; --first) {  // P = aI + bR + cR^2
                    GroupSpec s = sym_spec(eng, Rop, Rop);
                    s.c_acc = h->ns_c;
                    s.c_diag = h->ns_a;
                    s.c_aux = h->ns_b;
                    // the b R term: fp32 R (FFMA engine: read transposed, coalesced;
                    // split engine: its lower triangle, read R[r][c], r >= c), or
                    // the bf16 R the products read (plain tensor-core engine)
                    s.aux = (eng == kKernelTc && !split) ? RB : RF;
                    s.aux_sym = eng != kKernelTc;
                    // P0 is also Q0: it is stored once, in Q0, where step 0's R P and
                    // R update read it
                    s.out[0] = first ? Q0 : P;
                    split_outputs(s);
                    if ((rc = add(first ? G_POLY0 : G_POLY, s))) return rc;
                }
                for (int dir = 0; dir < 2; ++dir) {  // Q <- P Q
                    GroupSpec s = sym_spec(eng, P, dir == 0 ? Q0 : Q1);
                    s.out[0] = dir == 0 ? Q1 : Q0;
                    split_outputs(s);
                    if ((rc = add(dir == 0 ? G_Q01 : G_Q10, s))) return rc;
                }
                for (int first = 1; first >= 0; --first) {  // R P (step 0: P0 held in Q0)
                    GroupSpec s = sym_spec(eng, Rop, first ? Q0 : P);
                    s.out[0] = RP;
                    split_outputs(s);
                    if ((rc = add(first ? G_RP0 : G_RP, s))) return rc;
                }
                for (int first = 1; first >= 0; --first) {  // R <- P (R P)
                    GroupSpec s = sym_spec(eng, first ? Q0 : P, RP);
                    if (split) {
                        s.out[0] = RF;
                        s.out_lower_only[0] = true;
                        s.out[1] = RB;
                    } else {
                        s.out[0] = eng == kKernelTc ? RB : RF;
                    }
                    split_outputs(s);
                    if ((rc = add(first ? G_RUPD0 : G_RUPD, s))) return rc;
                }
                for (int qb = 0; qb < 2; ++qb) {  // W update from inv * Q X
                    GroupSpec s;
                    s.kernel = bf16 ? kKernelTc : kKernelSimt;
                    s.a = qb == 0 ? Q0 : Q1;
                    s.b = X0;
                    s.b_mn = true;
                    s.M = m;
                    s.N = n;
                    s.K = m;
                    s.mode = EPI_UPDATE;
                    s.alpha = ALPHA_INV;
                    if (split) {  // (Q_hi + Q_lo) X0: K over both parts of Q, X0's rows twice
                        s.K = 2 * sp;
                        s.kseg = sp;
                        s.a_k = 2 * sp;
                        s.b_k = m;
                    }
                    if ((rc = add(qb == 0 ? G_FIN0 : G_FIN1, s))) return rc;
                }
            } else {
                const Operand X[2] = {buf(p, BUF_X0), buf(p, BUF_X1)};
                const Operand AF = buf(p, BUF_RF), AB = buf(p, BUF_AB), BB = buf(p, BUF_BB);
                const Operand Aop = eng == kKernelTc ? AB : AF;
                struct { int kind, src, alpha; } syrks[3] = {{D_SYRK0, 0, ALPHA_INV2}, {D_SYRK_X0, 0, ALPHA_ONE},
                                                           {D_SYRK_X1, 1, ALPHA_ONE}};
                for (auto& sk : syrks) {  // A = alpha X X^T
                    GroupSpec s;
                    s.kernel = eng;
                    s.a = X[sk.src];
                    s.b = X[sk.src];
                    s.M = m;
                    s.N = m;
                    s.K = n;
                    s.sym = true;
                    s.alpha = sk.alpha;
                    s.out[0] = eng == kKernelTc ? AB : AF;
                    if ((rc = add(sk.kind, s))) return rc;
                }
                {  // B = bA + cA^2
                    GroupSpec s = sym_spec(eng, Aop, Aop);
                    s.c_acc = h->ns_c;
                    s.c_aux = h->ns_b;
                    s.aux = eng == kKernelTc ? AB : AF;  // B's b A term: the A the product reads
                    s.aux_sym = eng != kKernelTc;
                    s.out[0] = BB;
                    if ((rc = add(D_A2, s))) return rc;
                }
                struct { int kind, src, alpha, mode; } ups[6] = {
                    {D_XUPD0, 0, ALPHA_INV, EPI_STORE}, {D_XUPD01, 0, ALPHA_ONE, EPI_STORE},
                    {D_XUPD10, 1, ALPHA_ONE, EPI_STORE}, {D_FIN0I, 0, ALPHA_INV, EPI_UPDATE},
                    {D_FIN0, 0, ALPHA_ONE, EPI_UPDATE},  {D_FIN1, 1, ALPHA_ONE, EPI_UPDATE}};
                for (auto& u : ups) {  // X' = alpha (a X + B X)
                    GroupSpec s;
                    s.kernel = eng;
                    s.a = BB;
                    s.b = X[u.src];
                    s.b_mn = true;
                    s.M = m;
                    s.N = n;
                    s.K = m;
                    s.mode = u.mode;
                    s.alpha = u.alpha;
                    s.c_aux = h->ns_a;
                    s.aux = X[u.src];
                    if (u.mode == EPI_STORE) s.out[0] = X[1 - u.src];
                    if ((rc = add(u.kind, s))) return rc;
                }
            }
        }
    }

    // split operands: the pad columns between m and each part's end are read
    // as K data by the products and written by nothing, so they are zeroed
    // once here
    for (const Wave& w : h->waves)
        for (const Piece& p : w.pieces) {
            const Bucket& b = h->buckets[p.bucket];
            if (b.engine != DMUON_ENGINE_TC_SPLIT || b.m % 64 == 0) continue;
            for (int k = 0; k < BUF_COUNT; ++k)
                if (split_operand(k) && b.buf_bytes[k] &&
                    cudaMemset(wbase + p.off[k], 0, static_cast<size_t>(p.count * b.buf_bytes[k])) != cudaSuccess)
                    return fail(DMUON_ERR_CUDA, "split operand clear failed");
        }

    // upload: status + tables
    if (cudaMemset(ws, 0, h->off_infos) != cudaSuccess ||
        cudaMemcpy(ws + h->off_infos, infos.data(), infos.size() * sizeof(MatInfo), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(ws + h->off_flat, flat_list.data(), flat_list.size() * sizeof(int32_t), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemset(ws + h->off_ptrs, 0, 3 * static_cast<size_t>(h->count) * sizeof(void*)) != cudaSuccess ||
        cudaMemcpy(ws + h->off_groups, h->groups.data(), h->groups.size() * sizeof(GemmGroup),
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return fail(DMUON_ERR_CUDA, std::string("table upload failed: ") + cudaGetErrorString(cudaGetLastError()));
    return DMUON_OK;
}

int dmuon_step(dmuon_handle_t h, void* const* params, const void* const* grads, void* const* momenta, float lr,
               float beta, float wd, int32_t ns_steps, void* stream) {
    return dmuon_step_ex(h, params, grads, momenta, lr, beta, wd, ns_steps, stream, nullptr);
}

int dmuon_step_ex(dmuon_handle_t h, void* const* params, const void* const* grads, void* const* momenta, float lr,
                  float beta, float wd, int32_t ns_steps, void* stream, void* params_ready) {
    if (!h) return fail(DMUON_ERR_INVALID_ARG, "NULL handle");
    if (!h->ws) return fail(DMUON_ERR_NO_WORKSPACE, "no workspace bound (dmuon_bind_workspace)");
    if (!params || !grads || !momenta) return fail(DMUON_ERR_INVALID_ARG, "NULL pointer array");
    if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(wd) || lr < 0.0f || wd < 0.0f ||
        beta < 0.0f || beta >= 1.0f)
        return fail(DMUON_ERR_INVALID_ARG, "need finite lr >= 0, wd >= 0, 0 <= beta < 1");
    if (ns_steps < 1 || ns_steps > DMUON_MAX_NS_STEPS)
        return fail(DMUON_ERR_INVALID_ARG, "ns_steps out of [1, " + std::to_string(DMUON_MAX_NS_STEPS) + "]");
    for (int64_t i = 0; i < h->count; ++i) {
        const void* ps[3] = {params[i], grads[i], momenta[i]};
        for (const void* p : ps) {
            if (!p) return fail(DMUON_ERR_INVALID_ARG, "NULL tensor pointer for matrix " + std::to_string(i));
            if (reinterpret_cast<uintptr_t>(p) & 15)
                return fail(DMUON_ERR_ALIGN, "tensor of matrix " + std::to_string(i) + " not 16-byte aligned");
        }
    }
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != h->device) return fail(DMUON_ERR_INVALID_ARG, "current device differs from the bound workspace's");
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // pointer table (params | grads | momenta), uploaded when it changes
    const size_t n = static_cast<size_t>(h->count);
    bool same = h->cached_ptrs.size() == 3 * n;
    for (size_t i = 0; same && i < n; ++i)
        same = h->cached_ptrs[i] == params[i] && h->cached_ptrs[n + i] == grads[i] &&
               h->cached_ptrs[2 * n + i] == momenta[i];
    if (!same) {
        h->cached_ptrs.resize(3 * n);
        for (size_t i = 0; i < n; ++i) {
            h->cached_ptrs[i] = params[i];
            h->cached_ptrs[n + i] = grads[i];
            h->cached_ptrs[2 * n + i] = momenta[i];
        }
        if (cudaMemcpyAsync(h->ws + h->off_ptrs, h->cached_ptrs.data(), 3 * n * sizeof(void*),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return fail(DMUON_ERR_CUDA, "pointer table upload failed");
    }

    const auto& per_wave = launches_for(h, ns_steps);
    if (h->phase_error) return DMUON_ERR_INVALID_ARG;
    void* const* dptr = reinterpret_cast<void* const*>(h->ws + h->off_ptrs);
    bool waited = params_ready == nullptr;
    const float decay = 1.0f - lr * wd;
    for (size_t wi = 0; wi < h->waves.size(); ++wi) {
        const Wave& w = h->waves[wi];
        MomentumArgs ma;
        std::memset(&ma, 0, sizeof(ma));
        ma.infos = reinterpret_cast<const MatInfo*>(h->ws + h->off_infos) + w.slot0;
        ma.scalars = reinterpret_cast<SlotScalars*>(h->ws + h->off_scalars) + w.slot0;
        ma.grads = reinterpret_cast<const void* const*>(dptr + n);
        ma.moms = dptr + 2 * n;
        ma.flat_slots = reinterpret_cast<const int32_t*>(h->ws + h->off_flat) + w.slot0;
        ma.status = reinterpret_cast<int32_t*>(h->ws + h->off_status);
        ma.nslots = static_cast<int32_t>(w.nslots);
        ma.nflat = static_cast<int32_t>(w.nflat);
        ma.total_tiles = w.mom_tiles;
        ma.flat_chunks = w.flat_chunks;
        ma.beta = beta;
        ma.nesterov = h->nesterov;
        ma.eps = h->eps;
        cudaError_t e = timed(h, s, DMUON_TIMER_MOMENTUM, -1, [&] {
            const cudaError_t r = launch_momentum_flat(ma, s);
            return r != cudaSuccess ? r : launch_momentum_pack(ma, s);
        });
        if (e == cudaSuccess) e = timed(h, s, DMUON_TIMER_NORM, -1, [&] { return launch_norm_finalize(ma, s); });
        if (e != cudaSuccess) return fail(DMUON_ERR_CUDA, std::string("momentum launch: ") + cudaGetErrorString(e));
        if (per_wave[wi].size() > static_cast<size_t>(kMaxLaunchesPerWave))
            return fail(DMUON_ERR_INVALID_ARG, "too many launches in one wave");
        // the tensor-core launches take tiles from per-launch counters
        e = cudaMemsetAsync(h->ws + h->off_counters, 0, per_wave[wi].size() * sizeof(int32_t), s);
        if (e != cudaSuccess) return fail(DMUON_ERR_CUDA, std::string("counter reset: ") + cudaGetErrorString(e));
        for (const Launch& la : per_wave[wi]) {
            if (!waited && la.timer == DMUON_TIMER_FINAL) {
                // the first launch that writes parameters: the caller may still
                // be reading them until params_ready
                e = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(params_ready), 0);
                if (e != cudaSuccess) return fail(DMUON_ERR_CUDA, std::string("wait on params_ready: ") +
                                                                     cudaGetErrorString(e));
                waited = true;
            }
            LaunchList l = la.list;
            l.lr = lr;
            l.decay = decay;
            if (la.kernel == kKernelTc)
                e = timed(h, s, la.timer, DMUON_TIMER_TC, [&] { return launch_gemm_tc(l, h->num_sms, s); });
            else
                e = timed(h, s, la.timer, DMUON_TIMER_SIMT, [&] { return launch_gemm_simt(l, s); });
            if (e != cudaSuccess) return fail(DMUON_ERR_CUDA, std::string("GEMM launch: ") + cudaGetErrorString(e));
        }
    }
    return DMUON_OK;
}

int dmuon_device_status(dmuon_handle_t h, void* stream) {
    if (!h || !h->ws) return fail(DMUON_ERR_NO_WORKSPACE, "no workspace bound");
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return fail(DMUON_ERR_CUDA, std::string("stream error: ") + cudaGetErrorString(cudaGetLastError()));
    int32_t v = 0;
    if (cudaMemcpy(&v, h->ws + h->off_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail(DMUON_ERR_CUDA, "status read failed");
    if (v != DEV_OK) {
        cudaMemset(h->ws + h->off_status, 0, sizeof(v));
        return fail(DMUON_ERR_DEVICE_TIMEOUT, "a device-side wait timed out");
    }
    return DMUON_OK;
}

int dmuon_set_timing(dmuon_handle_t h, int32_t enable) {
    if (!h) return fail(DMUON_ERR_INVALID_ARG, "NULL handle");
    int rc = collect_timing(h);
    if (rc) return rc;
    h->timing = enable != 0;
    for (int k = 0; k < DMUON_TIMER_COUNT; ++k) {
        h->timer_ms[k] = 0.0;
        h->timer_launches[k] = 0;
    }
    return DMUON_OK;
}

int dmuon_get_timing(dmuon_handle_t h, double* ms, int64_t* launches, int32_t n) {
    if (!h || n < 0) return fail(DMUON_ERR_INVALID_ARG, "bad timing query");
    int rc = collect_timing(h);
    if (rc) return rc;
    for (int k = 0; k < n && k < DMUON_TIMER_COUNT; ++k) {
        if (ms) ms[k] = h->timer_ms[k];
        if (launches) launches[k] = h->timer_launches[k];
    }
    return DMUON_OK;
}

int dmuon_debug_buffer(dmuon_handle_t h, int64_t wave, int64_t piece, int32_t which, uint64_t* offset, int64_t* ld,
                       int64_t* batch_stride, int32_t* elem_type) {
    if (!h || wave < 0 || wave >= static_cast<int64_t>(h->waves.size()) || piece < 0 ||
        piece >= static_cast<int64_t>(h->waves[wave].pieces.size()) || !offset || !ld || !batch_stride)
        return fail(DMUON_ERR_INVALID_ARG, "bad buffer query");
    const Piece& p = h->waves[wave].pieces[piece];
    const Bucket& b = h->buckets[p.bucket];
    int k = which == DMUON_BUF_X ? BUF_X0 : (which == DMUON_BUF_RF ? BUF_RF : -1);
    if (which == DMUON_BUF_R_OPERAND) k = b.buf_bytes[BUF_RB] ? BUF_RB : (b.buf_bytes[BUF_AB] ? BUF_AB : BUF_RF);
    if (k < 0 || !b.buf_bytes[k]) return fail(DMUON_ERR_INVALID_ARG, "unknown buffer");
    *offset = h->off_waves + p.off[k];
    *ld = static_cast<int64_t>(up(static_cast<uint64_t>(k == BUF_X0 ? b.n : b.m), 8));
    if (b.engine == DMUON_ENGINE_TC_SPLIT && split_operand(k)) *ld = split_ld(b.m);
    if (elem_type) *elem_type = b.buf_type[k] == ELEM_BF16 ? DMUON_BF16 : DMUON_FP32;
    *batch_stride = b.buf_bytes[k] / esz(b.buf_type[k]);
    return DMUON_OK;
}

}  // extern "C"
