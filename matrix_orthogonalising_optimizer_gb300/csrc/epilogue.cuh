// Fused GEMM epilogue shared by the tcgen05 and the fp32 FFMA kernels.
//
// Every product of the step ends in one formula per output element (r, c):
//   v = alpha * (c_acc * acc + c_diag * [r == c] + c_aux * aux[r][c])
// which covers the Newton-Schulz polynomial P = aI + bR + cR^2 (acc = R R,
// aux = R), the Gram product R0 = inv^2 X X^T, the direct-route iterate
// X' = alpha (a X + B X), and the plain products.  It then either stores v
// (fp32 and/or the operand dtype; symmetric results store the lower triangle
// and, for outputs read as operands, its mirror, so they are bitwise
// symmetric), or applies the Muon update
//   W = (1 - lr*wd) W - lr*s*v
// in W's own orientation (transposed back for tall matrices).
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace dmuon {

__device__ __forceinline__ int elem_size(int32_t t) { return t == ELEM_BF16 ? 2 : 4; }

__device__ __forceinline__ float load_elem(const void* p, int64_t i, int32_t t) {
    if (t == ELEM_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void store_elem(void* p, int64_t i, int32_t t, float v) {
    if (t == ELEM_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else static_cast<float*>(p)[i] = v;
}

// Per (group, matrix) pointers and scalars, resolved once per tile.
struct EpiCtx {
    float alpha;
    float lrs;           // lr * s for the update
    const void* aux;
    void* out[3];
    void* w;
    int32_t w_type;
    int32_t w_cols;
    int32_t transposed;
};

__device__ __forceinline__ EpiCtx make_epi_ctx(const GemmGroup& g, const LaunchList& L, int mat) {
    EpiCtx c;
    const int slot = g.slot_base + mat;
    const SlotScalars sc = L.scalars[slot];
    c.alpha = g.alpha_sel == ALPHA_INV ? sc.inv : (g.alpha_sel == ALPHA_INV2 ? sc.inv2 : 1.0f);
    c.aux = g.aux ? static_cast<const char*>(g.aux) + mat * g.aux_bs * elem_size(g.aux_type) : nullptr;
#pragma unroll
    for (int o = 0; o < 3; ++o)
        c.out[o] = g.out[o] ? static_cast<char*>(g.out[o]) + mat * g.out_bs[o] * elem_size(g.out_type[o]) : nullptr;
    c.w = nullptr;
    c.lrs = 0.0f;
    c.w_type = ELEM_BF16;
    c.w_cols = 0;
    c.transposed = 0;
    if (g.mode == EPI_UPDATE) {
        const MatInfo& mi = L.infos[slot];
        c.w = L.params[mi.gidx];
        c.w_type = mi.dtype;
        c.w_cols = mi.cols;
        c.transposed = mi.transposed;
        c.lrs = L.lr * mi.scale;
    }
    return c;
}

// Epilogue parameters of one tile, held in registers (the group table lives in
// global memory, and stores through generic pointers would otherwise force
// the compiler to reload every field after each store).
// The one-bit properties share one word (registers are the epilogue's
// scarce resource).
enum EpiFlag : uint32_t {
    F_UPDATE = 1u << 0,      // EPI_UPDATE (else EPI_STORE)
    F_SYM = 1u << 1,         // symmetric result
    F_AUX_F32 = 1u << 2,     // aux dtype fp32 (else bf16)
    F_AUX_SYM = 1u << 3,     // aux read transposed
    F_W_F32 = 1u << 4,       // W dtype fp32 (else bf16)
    F_TRANSPOSED = 1u << 5,  // W stored transposed (tall matrix)
    F_W_VEC = 1u << 6,       // W rows start on 16 bytes
    F_OUT_F32 = 1u << 8,     // << o: output o is fp32 (else bf16)
    F_OUT_MIRROR = 1u << 12, // << o: output o also stores the mirrored half
};

struct EpiRegs {
    const char* aux;
    char* out[3];
    char* w;
    float alpha, c_acc, c_diag, c_aux, lrs, decay;
    int32_t M, N, aux_ld, w_cols;
    uint32_t flags;
    int32_t out_ld[3], out_lo[3];
    __device__ __forceinline__ bool update() const { return flags & F_UPDATE; }
    __device__ __forceinline__ bool sym() const { return flags & F_SYM; }
    __device__ __forceinline__ int32_t aux_type() const { return flags & F_AUX_F32 ? ELEM_F32 : ELEM_BF16; }
    __device__ __forceinline__ bool aux_sym() const { return flags & F_AUX_SYM; }
    __device__ __forceinline__ int32_t w_type() const { return flags & F_W_F32 ? ELEM_F32 : ELEM_BF16; }
    __device__ __forceinline__ bool transposed() const { return flags & F_TRANSPOSED; }
    __device__ __forceinline__ bool w_vec() const { return flags & F_W_VEC; }
    __device__ __forceinline__ int32_t out_type(int o) const { return flags & (F_OUT_F32 << o) ? ELEM_F32 : ELEM_BF16; }
    __device__ __forceinline__ bool out_mirror(int o) const { return flags & (F_OUT_MIRROR << o); }
};

__device__ __forceinline__ EpiRegs load_epi(const GemmGroup& g, const LaunchList& L, int mat) {
    const EpiCtx c = make_epi_ctx(g, L, mat);
    EpiRegs e;
    e.aux = static_cast<const char*>(c.aux);
    uint32_t f = 0;
#pragma unroll
    for (int o = 0; o < 3; ++o) {
        e.out[o] = static_cast<char*>(c.out[o]);
        e.out_ld[o] = g.out_ld[o];
        if (g.out_type[o] == ELEM_F32) f |= F_OUT_F32 << o;
        if (g.sym && g.out_mirror[o]) f |= F_OUT_MIRROR << o;
        e.out_lo[o] = g.out_lo[o];
    }
    e.w = static_cast<char*>(c.w);
    e.alpha = c.alpha;
    e.c_acc = g.c_acc;
    e.c_diag = g.c_diag;
    e.c_aux = g.c_aux;
    e.lrs = c.lrs;
    e.decay = L.decay;
    e.M = g.M;
    e.N = g.N;
    e.aux_ld = g.aux_ld;
    e.w_cols = c.w_cols;
    if (g.mode == EPI_UPDATE) f |= F_UPDATE;
    if (g.sym) f |= F_SYM;
    if (g.aux_type == ELEM_F32) f |= F_AUX_F32;
    if (g.aux_sym) f |= F_AUX_SYM;
    if (c.w_type == ELEM_F32) f |= F_W_F32;
    if (c.transposed) f |= F_TRANSPOSED;
    // 16-byte row access to W needs every row start on 16 bytes
    if (c.w && ((static_cast<int64_t>(c.w_cols) * (c.w_type == ELEM_BF16 ? 2 : 4)) % 16 == 0)) f |= F_W_VEC;
    e.flags = f;
    return e;
}

// The low bf16 part of v: v - bf16(v), exact in fp32, so hi + lo carries v
// to about 16 significant bits.
__device__ __forceinline__ float lo_part(float v) { return v - __bfloat162float(__float2bfloat16_rn(v)); }

// Element i of output o (and, for a split output, its low part out_lo
// elements further along the row).
__device__ __forceinline__ void store_out(const EpiRegs& e, int o, int64_t i, float v) {
    store_elem(e.out[o], i, e.out_type(o), v);
    if (e.out_lo[o]) store_elem(e.out[o], i + e.out_lo[o], ELEM_BF16, lo_part(v));
}

// Same formula, same operation order as epi_value (epilogue.cuh).
__device__ __forceinline__ float epi_v(const EpiRegs& e, int r, int c, float acc, float aux) {
    float t = e.c_acc * acc;
    if (r == c) t += e.c_diag;
    if (e.aux) t = fmaf(e.c_aux, aux, t);
    return e.alpha * t;
}

// Element (r, col), r < M, col < N, with the parameters in registers: the
// per-element path of the fp32 FFMA kernel (same formula as the chunked
// tensor-core epilogue).
__device__ __forceinline__ void epi_element_regs(const EpiRegs& e, int r, int col, float acc) {
    if (!e.update() && e.sym() && r < col) return;
    float aux = 0.0f;
    if (e.aux) {
        const int64_t i = e.aux_sym() ? static_cast<int64_t>(col) * e.aux_ld + r : static_cast<int64_t>(r) * e.aux_ld + col;
        aux = load_elem(e.aux, i, e.aux_type());
    }
    const float v = epi_v(e, r, col, acc, aux);
    if (e.update()) {
        const int64_t wi = e.transposed() ? static_cast<int64_t>(col) * e.w_cols + r
                                        : static_cast<int64_t>(r) * e.w_cols + col;
        const float w = load_elem(e.w, wi, e.w_type());
        store_elem(e.w, wi, e.w_type(), fmaf(-e.lrs, v, e.decay * w));
        return;
    }
#pragma unroll
    for (int o = 0; o < 3; ++o) {
        if (!e.out[o]) continue;
        store_out(e, o, static_cast<int64_t>(r) * e.out_ld[o] + col, v);
        if (e.out_mirror(o) && r > col) store_out(e, o, static_cast<int64_t>(col) * e.out_ld[o] + r, v);
    }
}

}  // namespace dmuon
