// Fused GEMM epilogue shared by the tcgen05 and the fp32 FFMA kernels.
//
// Every product of the step ends in one formula per output element (r, c):
//   v = alpha * (c_acc * acc + c_diag * [r == c] + c_aux * aux[r][c])
// which covers the Newton-Schulz polynomial P = aI + bR + cR^2 (acc = R R,
// aux = R), the Gram product R0 = inv^2 X X^T, the direct-route iterate
// X' = alpha (a X + B X), and the plain products.  It then either stores v
// (fp32 and/or the operand dtype; symmetric results store the lower triangle
// and its mirror, so they are bitwise symmetric), or applies the Muon update
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

__device__ __forceinline__ float epi_aux(const GemmGroup& g, const EpiCtx& c, int r, int col) {
    if (!c.aux) return 0.0f;
    const int64_t i = g.aux_sym ? static_cast<int64_t>(col) * g.aux_ld + r
                                : static_cast<int64_t>(r) * g.aux_ld + col;
    return load_elem(c.aux, i, g.aux_type);
}

// The one per-element formula; every path computes it in this order.
__device__ __forceinline__ float epi_value(const GemmGroup& g, const EpiCtx& c, int r, int col,
                                           float acc, float aux) {
    float t = g.c_acc * acc;
    if (r == col) t += g.c_diag;
    if (c.aux) t = fmaf(g.c_aux, aux, t);
    return c.alpha * t;
}

__device__ __forceinline__ void epi_write(const GemmGroup& g, const EpiCtx& c, int i, int j, float v) {
#pragma unroll
    for (int o = 0; o < 3; ++o)
        if (c.out[o]) store_elem(c.out[o], static_cast<int64_t>(i) * g.out_ld[o] + j, g.out_type[o], v);
}

__device__ __forceinline__ void epi_update(const LaunchList& L, const EpiCtx& c, int r, int col, float v) {
    const int64_t wi = c.transposed ? static_cast<int64_t>(col) * c.w_cols + r
                                    : static_cast<int64_t>(r) * c.w_cols + col;
    const float w = load_elem(c.w, wi, c.w_type);
    store_elem(c.w, wi, c.w_type, fmaf(-c.lrs, v, L.decay * w));
}

// Element (r, col) with r < M, col < N.
__device__ __forceinline__ void epi_element(const GemmGroup& g, const EpiCtx& c, const LaunchList& L,
                                            int r, int col, float acc) {
    if (g.mode == EPI_STORE && g.sym && r < col) return;
    const float v = epi_value(g, c, r, col, acc, epi_aux(g, c, r, col));
    if (g.mode == EPI_UPDATE) {
        epi_update(L, c, r, col, v);
        return;
    }
    epi_write(g, c, r, col, v);
    if (g.sym && r > col) epi_write(g, c, col, r, v);
}

}  // namespace dmuon
