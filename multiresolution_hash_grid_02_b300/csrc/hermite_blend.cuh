// Hermite-NGP blends of one (point, level) on one thread, shared by the
// generic forward and the fused encoder + SIREN forward.
//
// "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
// 关键设计 1 (tensor-product Hermite bases, dx^|alpha| scaling) and 关键设计 2
// (gradient and Laplacian from the bases' derivatives).  Separable: contract
// axis 0, then axis 1 (then axis 2), carrying value, d/dx_0 and d2/dx_0^2
// partial sums.
#pragma once

#include "hg_device.cuh"
#include "hg_params.h"

namespace hg {

// Separable 2D blend of one feature: q[corner][alpha].
__device__ __forceinline__ void blend2(const float (&q)[4][4], const Basis1& b0, const Basis1& b1, float& g,
                                       float (&dg)[3], float& lap) {
    g = 0.f, dg[0] = 0.f, dg[1] = 0.f, lap = 0.f;
#pragma unroll
    for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
        for (int a1 = 0; a1 < 2; ++a1) {
            float s = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                for (int a0 = 0; a0 < 2; ++a0) {
                    const float c = q[v0 + 2 * v1][a0 + 2 * a1];
                    s = fmaf(c, b0.w[v0][a0], s);
                    s1 = fmaf(c, b0.d1[v0][a0], s1);
                    s2 = fmaf(c, b0.d2[v0][a0], s2);
                }
            g = fmaf(s, b1.w[v1][a1], g);
            dg[0] = fmaf(s1, b1.w[v1][a1], dg[0]);
            dg[1] = fmaf(s, b1.d1[v1][a1], dg[1]);
            lap = fmaf(s2, b1.w[v1][a1], lap);
            lap = fmaf(s, b1.d2[v1][a1], lap);
        }
}

// blend2 for both features at once: q[corner][alpha] holds the (feature 0,
// feature 1) coefficient pairs, o[] accumulates (gamma, d/dx0, d/dx1, lap)
// pairs.  Each f32x2 operation is the scalar blend2's operation on both
// features (the same order, the same roundings), so the results are
// bit-identical to blend2's, with half the FMA instructions.
__device__ __forceinline__ void blend2_f2(const uint64_t (&q)[4][4], const Basis1& b0, const Basis1& b1,
                                          uint64_t (&o)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = 0ull;  // (+0.0f, +0.0f)
#pragma unroll
    for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
        for (int a1 = 0; a1 < 2; ++a1) {
            uint64_t s = 0ull, s1 = 0ull, s2 = 0ull;
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                for (int a0 = 0; a0 < 2; ++a0) {
                    const uint64_t c = q[v0 + 2 * v1][a0 + 2 * a1];
                    s = f2_fma(c, f2_dup(b0.w[v0][a0]), s);
                    s1 = f2_fma(c, f2_dup(b0.d1[v0][a0]), s1);
                    s2 = f2_fma(c, f2_dup(b0.d2[v0][a0]), s2);
                }
            const uint64_t w = f2_dup(b1.w[v1][a1]);
            o[0] = f2_fma(s, w, o[0]);
            o[1] = f2_fma(s1, w, o[1]);
            o[2] = f2_fma(s, f2_dup(b1.d1[v1][a1]), o[2]);
            o[3] = f2_fma(s2, w, o[3]);
            o[3] = f2_fma(s, f2_dup(b1.d2[v1][a1]), o[3]);
        }
}

// Separable 3D blend of one feature.
__device__ __forceinline__ void blend3(const float (&q)[8][8], const Basis1& b0, const Basis1& b1,
                                       const Basis1& b2, float& g, float (&dg)[3], float& lap) {
    g = 0.f, dg[0] = 0.f, dg[1] = 0.f, dg[2] = 0.f, lap = 0.f;
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2)
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2) {
            float A = 0.f, B = 0.f, C = 0.f, Dl = 0.f;
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
                for (int a1 = 0; a1 < 2; ++a1) {
                    float s = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
                    for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                        for (int a0 = 0; a0 < 2; ++a0) {
                            const float c = q[v0 + 2 * v1 + 4 * v2][a0 + 2 * a1 + 4 * a2];
                            s = fmaf(c, b0.w[v0][a0], s);
                            s1 = fmaf(c, b0.d1[v0][a0], s1);
                            s2 = fmaf(c, b0.d2[v0][a0], s2);
                        }
                    A = fmaf(s, b1.w[v1][a1], A);
                    B = fmaf(s1, b1.w[v1][a1], B);
                    C = fmaf(s, b1.d1[v1][a1], C);
                    Dl = fmaf(s2, b1.w[v1][a1], Dl);
                    Dl = fmaf(s, b1.d2[v1][a1], Dl);
                }
            g = fmaf(A, b2.w[v2][a2], g);
            dg[0] = fmaf(B, b2.w[v2][a2], dg[0]);
            dg[1] = fmaf(C, b2.w[v2][a2], dg[1]);
            dg[2] = fmaf(A, b2.d1[v2][a2], dg[2]);
            lap = fmaf(Dl, b2.w[v2][a2], lap);
            lap = fmaf(A, b2.d2[v2][a2], lap);
        }
}

// One (point n, level l) of a packed [L][T][2^d][F] table with F = 2, on
// one thread: the 2^d corner rows read whole (vector loads), then the
// separable blend of each feature (2D: both features at once, blend2_f2) --
// the arithmetic of the generic forward's packed path, so the results are
// bit-identical to it.  g[f], dg[f][j] and
// lap[f]: gamma, d gamma / d x_j and the Laplacian of feature f.
template <int D, typename TT>
__device__ __forceinline__ void encode_item_f2(const FwdParams& p, int64_t n, int l, float (&g)[2],
                                               float (&dg)[2][3], float (&lap)[2]) {
    constexpr int V = 1 << D, FC = 2;
    const Level& lv = p.c.lv[l];
    uint32_t c[D];
    float t[D];
    Basis1 B[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }
    constexpr int ROW = V * FC * static_cast<int>(sizeof(TT));
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
    RowRegs<ROW> rows[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        uint32_t gv[D];
#pragma unroll
        for (int i = 0; i < D; ++i) gv[i] = c[i] + ((v >> i) & 1u);
        const uint32_t id = vertex_index<D>(gv, lv, lv.dense & 1u, p.c.tmask[0]);
        load_row<ROW>(base + static_cast<int64_t>(id) * p.tab.rs[0], rows[v]);
    }
    if constexpr (D == 2) {
        uint64_t q[V][V], o[4];
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int a = 0; a < V; ++a)
                q[v][a] = f2_pack(row_elem<TT, ROW>(rows[v], packed_slot<D>(a) * FC),
                                  row_elem<TT, ROW>(rows[v], packed_slot<D>(a) * FC + 1));
        blend2_f2(q, B[0], B[1], o);
        f2_unpack(o[0], g[0], g[1]);
        f2_unpack(o[1], dg[0][0], dg[1][0]);
        f2_unpack(o[2], dg[0][1], dg[1][1]);
        f2_unpack(o[3], lap[0], lap[1]);
        dg[0][2] = dg[1][2] = 0.f;
    } else {
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            float q[V][V];
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int a = 0; a < V; ++a) q[v][a] = row_elem<TT, ROW>(rows[v], packed_slot<D>(a) * FC + f);
            blend3(q, B[0], B[1], B[2], g[f], dg[f], lap[f]);
        }
    }
}

}  // namespace hg
