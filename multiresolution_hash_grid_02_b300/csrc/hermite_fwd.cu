// Hermite-NGP forward: gamma, grad gamma and the Laplacian (or the full
// Hessian) of every (point, level) in one pass.
//
// "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
// 关键设计 1 (the encoding equation with tensor-product Hermite bases and the
// dx^|alpha| scaling) and 关键设计 2 (the factorised derivative and the
// second derivative of the bases).
//
// Mapping: one thread per (point, level); grid.y = level, so the blocks of
// one level run together and that level's table stays resident in L2 while
// every point gathers from it.  The blend is separable: contract axis 0, then
// axis 1 (then axis 2), carrying value, d/dx_0 and d2/dx_0^2 partial sums, so
// a 3D level costs ~600 FMA for F = 2 instead of ~1300 for the direct sum.
// The full-Hessian variant (HESS) splits the second-order partial sums by
// axis pair instead of adding them into one Laplacian term.
#include <cuda_runtime.h>

#include <algorithm>

#include "hermite_blend.cuh"
#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;

// Separable 2D blend with the full Hessian h = (xx, xy, yy).
__device__ __forceinline__ void blend2h(const float (&q)[4][4], const Basis1& b0, const Basis1& b1, float& g,
                                        float (&dg)[3], float (&h)[6]) {
    g = 0.f, dg[0] = 0.f, dg[1] = 0.f, h[0] = 0.f, h[1] = 0.f, h[2] = 0.f;
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
            h[0] = fmaf(s2, b1.w[v1][a1], h[0]);
            h[1] = fmaf(s1, b1.d1[v1][a1], h[1]);
            h[2] = fmaf(s, b1.d2[v1][a1], h[2]);
        }
}

// Separable 3D blend with the full Hessian h = (xx, xy, xz, yy, yz, zz).
// Per (v2, a2) the axis-0/1 contraction carries six sums: A (value),
// B (d/dx0), C (d/dx1), D00 (d2/dx0^2), D11 (d2/dx1^2), E01 (d2/dx0 dx1);
// axis 2 then supplies w, w' or w'' to each output.
__device__ __forceinline__ void blend3h(const float (&q)[8][8], const Basis1& b0, const Basis1& b1,
                                        const Basis1& b2, float& g, float (&dg)[3], float (&h)[6]) {
    g = 0.f, dg[0] = 0.f, dg[1] = 0.f, dg[2] = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) h[k] = 0.f;
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2)
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2) {
            float A = 0.f, B = 0.f, C = 0.f, D00 = 0.f, D11 = 0.f, E01 = 0.f;
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
                    D00 = fmaf(s2, b1.w[v1][a1], D00);
                    D11 = fmaf(s, b1.d2[v1][a1], D11);
                    E01 = fmaf(s1, b1.d1[v1][a1], E01);
                }
            g = fmaf(A, b2.w[v2][a2], g);
            dg[0] = fmaf(B, b2.w[v2][a2], dg[0]);
            dg[1] = fmaf(C, b2.w[v2][a2], dg[1]);
            dg[2] = fmaf(A, b2.d1[v2][a2], dg[2]);
            h[0] = fmaf(D00, b2.w[v2][a2], h[0]);
            h[1] = fmaf(E01, b2.w[v2][a2], h[1]);
            h[2] = fmaf(B, b2.d1[v2][a2], h[2]);
            h[3] = fmaf(D11, b2.w[v2][a2], h[3]);
            h[4] = fmaf(C, b2.d1[v2][a2], h[4]);
            h[5] = fmaf(A, b2.d2[v2][a2], h[5]);
        }
}

// Kernel: D dims, FC features per pass, TT table element type, VEC = packed
// interleaved rows read whole with vector loads (requires F == FC), HESS =
// full Hessian instead of the Laplacian.
template <int D, int FC, typename TT, bool VEC, bool HESS>
__global__ void __launch_bounds__(kBlock) hermite_fwd_kernel(const __grid_constant__ FwdParams p) {
    constexpr int V = 1 << D, P = D * (D + 1) / 2;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const bool active = (p.c.level_mask >> l) & 1u;

    float x[D];
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = __ldg(p.coords + n * D + i);

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(x[i], lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }

    // vertex indices: one per corner (VEC) or one per (order, corner)
    constexpr int NK = VEC ? 1 : D + 1;
    uint32_t idx[NK][V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        uint32_t g[D];
#pragma unroll
        for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
#pragma unroll
        for (int k = 0; k < NK; ++k) idx[k][v] = vertex_index<D>(g, lv, (lv.dense >> k) & 1u, p.c.tmask[k]);
    }

    if constexpr (D == 2 && VEC && FC == 2 && !HESS) {
        // packed 2D rows, both features per f32x2 operation (blend2_f2: bit-identical to blend2)
        float g[2] = {0.f, 0.f}, dg[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, lap[2] = {0.f, 0.f};
        if (active) {
            constexpr int ROW = V * FC * static_cast<int>(sizeof(TT));
            const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
            RowRegs<ROW> rows[V];
#pragma unroll
            for (int v = 0; v < V; ++v) load_row<ROW>(base + static_cast<int64_t>(idx[0][v]) * p.tab.rs[0], rows[v]);
            uint64_t q2[V][V], o[4];
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int a = 0; a < V; ++a)
                    q2[v][a] = f2_pack(row_elem<TT, ROW>(rows[v], packed_slot<D>(a) * FC),
                                       row_elem<TT, ROW>(rows[v], packed_slot<D>(a) * FC + 1));
            blend2_f2(q2, B[0], B[1], o);
            f2_unpack(o[0], g[0], g[1]);
            f2_unpack(o[1], dg[0][0], dg[1][0]);
            f2_unpack(o[2], dg[0][1], dg[1][1]);
            f2_unpack(o[3], lap[0], lap[1]);
        }
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f;
            __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, g[f]);
            if (p.dgamma) {
#pragma unroll
                for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, dg[f][j]);
            }
            if (p.lap) __stcs(p.lap + n * p.c.sn + lf * p.c.sf, lap[f]);
        }
    } else {
        for (int f0 = 0; f0 < F; f0 += FC) {
            float q[FC][V][V];
            if (active) {
                if constexpr (VEC) {
                    constexpr int ROW = V * FC * static_cast<int>(sizeof(TT));
                    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
                    RowRegs<ROW> rows[V];
#pragma unroll
                    for (int v = 0; v < V; ++v) load_row<ROW>(base + static_cast<int64_t>(idx[0][v]) * p.tab.rs[0], rows[v]);
#pragma unroll
                    for (int v = 0; v < V; ++v)
#pragma unroll
                        for (int a = 0; a < V; ++a)
#pragma unroll
                            for (int f = 0; f < FC; ++f) q[f][v][a] = row_elem<TT, ROW>(rows[v], packed_slot<D>(a) * FC + f);
                } else {
#pragma unroll
                    for (int v = 0; v < V; ++v)
#pragma unroll
                        for (int a = 0; a < V; ++a) {
                            const int k = alpha_order(a);
                            const TT* e = static_cast<const TT*>(p.tab.ptr[k]) + l * p.tab.ls[k] +
                                          static_cast<int64_t>(idx[k][v]) * p.tab.rs[k] + bucket_slot<D>(a) * F + f0;
#pragma unroll
                            for (int f = 0; f < FC; ++f) q[f][v][a] = to_f32<TT>(e[f]);
                        }
                }
            }
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                float g = 0.f, dg[3] = {0.f, 0.f, 0.f}, lap = 0.f, h[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (active) {
                    if constexpr (HESS) {
                        if constexpr (D == 2) {
                            blend2h(q[f], B[0], B[1], g, dg, h);
                        } else {
                            blend3h(q[f], B[0], B[1], B[D - 1], g, dg, h);
                        }
                    } else if constexpr (D == 2) {
                        blend2(q[f], B[0], B[1], g, dg, lap);
                    } else {
                        blend3(q[f], B[0], B[1], B[D - 1], g, dg, lap);
                    }
                }
                const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
                __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, g);
                if (p.dgamma) {
#pragma unroll
                    for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, dg[j]);
                }
                if constexpr (HESS) {
#pragma unroll
                    for (int k = 0; k < P; ++k) __stcs(p.hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, h[k]);
                } else if (p.lap) {
                    __stcs(p.lap + n * p.c.sn + lf * p.c.sf, lap);
                }
            }
        }
    }
}

// Contribution of one packed slot (multi-index alpha, with the weights
// W0..W2 of its per-axis orders) to the 3D outputs, for both features at
// once (the 4D lane-quad forward blends its axis-3 slices with these): c[v] is the slot's (feature 0, feature 1) coefficient pair at corner
// v = v0 + 2 v1 + 4 v2; o[] accumulates (gamma, d/dx0, d/dx1, d/dx2, lap)
// pairs.  The same separable order as blend3, restricted to one alpha.
__device__ __forceinline__ void unit_blend3_f2(const uint64_t (&c)[8], const AxisW2& W0, const AxisW2& W1,
                                               const AxisW2& W2, uint64_t (&o)[5]) {
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2) {
        uint64_t A, B, C, Dl;
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1) {
            const uint64_t c0 = c[2 * v1 + 4 * v2], c1 = c[1 + 2 * v1 + 4 * v2];
            const uint64_t s = f2_fma(c0, W0.w[0], f2_mul(c1, W0.w[1]));
            const uint64_t s1 = f2_fma(c0, W0.d1[0], f2_mul(c1, W0.d1[1]));
            const uint64_t s2 = f2_fma(c0, W0.d2[0], f2_mul(c1, W0.d2[1]));
            if (v1 == 0) {
                A = f2_mul(s, W1.w[0]);
                B = f2_mul(s1, W1.w[0]);
                C = f2_mul(s, W1.d1[0]);
                Dl = f2_fma(s, W1.d2[0], f2_mul(s2, W1.w[0]));
            } else {
                A = f2_fma(s, W1.w[1], A);
                B = f2_fma(s1, W1.w[1], B);
                C = f2_fma(s, W1.d1[1], C);
                Dl = f2_fma(s2, W1.w[1], Dl);
                Dl = f2_fma(s, W1.d2[1], Dl);
            }
        }
        o[0] = f2_fma(A, W2.w[v2], o[0]);
        o[1] = f2_fma(B, W2.w[v2], o[1]);
        o[2] = f2_fma(C, W2.w[v2], o[2]);
        o[3] = f2_fma(A, W2.d1[v2], o[3]);
        o[4] = f2_fma(Dl, W2.w[v2], o[4]);
        o[4] = f2_fma(A, W2.d2[v2], o[4]);
    }
}

// unit_blend3_f2 with the full Hessian: o[] accumulates (gamma, d/dx0,
// d/dx1, d/dx2, xx, xy, xz, yy, yz, zz) pairs, in the order of blend3h.
__device__ __forceinline__ void unit_blend3_f2_hess(const uint64_t (&c)[8], const AxisW2& W0, const AxisW2& W1,
                                                    const AxisW2& W2, uint64_t (&o)[10]) {
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2) {
        uint64_t A, B, C, D00, D11, E01;
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1) {
            const uint64_t c0 = c[2 * v1 + 4 * v2], c1 = c[1 + 2 * v1 + 4 * v2];
            const uint64_t s = f2_fma(c0, W0.w[0], f2_mul(c1, W0.w[1]));
            const uint64_t s1 = f2_fma(c0, W0.d1[0], f2_mul(c1, W0.d1[1]));
            const uint64_t s2 = f2_fma(c0, W0.d2[0], f2_mul(c1, W0.d2[1]));
            if (v1 == 0) {
                A = f2_mul(s, W1.w[0]);
                B = f2_mul(s1, W1.w[0]);
                C = f2_mul(s, W1.d1[0]);
                D00 = f2_mul(s2, W1.w[0]);
                D11 = f2_mul(s, W1.d2[0]);
                E01 = f2_mul(s1, W1.d1[0]);
            } else {
                A = f2_fma(s, W1.w[1], A);
                B = f2_fma(s1, W1.w[1], B);
                C = f2_fma(s, W1.d1[1], C);
                D00 = f2_fma(s2, W1.w[1], D00);
                D11 = f2_fma(s, W1.d2[1], D11);
                E01 = f2_fma(s1, W1.d1[1], E01);
            }
        }
        o[0] = f2_fma(A, W2.w[v2], o[0]);
        o[1] = f2_fma(B, W2.w[v2], o[1]);
        o[2] = f2_fma(C, W2.w[v2], o[2]);
        o[3] = f2_fma(A, W2.d1[v2], o[3]);
        o[4] = f2_fma(D00, W2.w[v2], o[4]);
        o[5] = f2_fma(E01, W2.w[v2], o[5]);
        o[6] = f2_fma(B, W2.d1[v2], o[6]);
        o[7] = f2_fma(D11, W2.w[v2], o[7]);
        o[8] = f2_fma(C, W2.d1[v2], o[8]);
        o[9] = f2_fma(A, W2.d2[v2], o[9]);
    }
}

// Lane-pair blend of a packed 3D F = 2 row split by the order along axis 2.
// After pair_exchange, lane h of a pair holds, for every corner v = v0 + 2 v1
// + 4 v2, the (feature 0, feature 1) coefficient pairs q[v][i] of the four
// multi-indices alpha = (i & 1, i >> 1, h): the whole separable contraction
// over (v0, a0) and (v1, a1) runs inside the lane (axis-0 sums s, s1, s2 for
// each (v1, a1, v2); axis-1 sums per v2), and axis 2 contributes only its
// order-h weights w2.  o[] accumulates (gamma, d/dx0, d/dx1, d/dx2, lap)
// pairs, or with HESS (gamma, d/dx0, d/dx1, d/dx2, xx, xy, xz, yy, yz, zz);
// gamma and the gradient take the same operations in both variants.  The
// lane's partial outputs (alpha_2 = h) of the pair add up to the encoding.
// 148 f32x2 operations per lane (164 with HESS), against 224 for a blend of
// each slot on its own (3D, 2^21 points, 16 levels: 2.34 -> 2.12 ms).
template <bool HESS>
__device__ __forceinline__ void blend3_pair_a2(const uint64_t (&q)[8][4], const Basis1& b0, const Basis1& b1,
                                               const AxisW& w2, uint64_t (&o)[HESS ? 10 : 5]) {
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2) {
        uint64_t A, B, C, Dl, D00, D11, E01;
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
            for (int a1 = 0; a1 < 2; ++a1) {
                uint64_t s, s1, s2;
#pragma unroll
                for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                    for (int a0 = 0; a0 < 2; ++a0) {
                        const uint64_t c = q[v0 + 2 * v1 + 4 * v2][a0 + 2 * a1];
                        if (v0 == 0 && a0 == 0) {
                            s = f2_mul(c, f2_dup(b0.w[0][0]));
                            s1 = f2_mul(c, f2_dup(b0.d1[0][0]));
                            s2 = f2_mul(c, f2_dup(b0.d2[0][0]));
                        } else {
                            s = f2_fma(c, f2_dup(b0.w[v0][a0]), s);
                            s1 = f2_fma(c, f2_dup(b0.d1[v0][a0]), s1);
                            s2 = f2_fma(c, f2_dup(b0.d2[v0][a0]), s2);
                        }
                    }
                const uint64_t w = f2_dup(b1.w[v1][a1]), d1 = f2_dup(b1.d1[v1][a1]), d2 = f2_dup(b1.d2[v1][a1]);
                if (v1 == 0 && a1 == 0) {
                    A = f2_mul(s, w);
                    B = f2_mul(s1, w);
                    C = f2_mul(s, d1);
                    if constexpr (HESS) {
                        D00 = f2_mul(s2, w);
                        D11 = f2_mul(s, d2);
                        E01 = f2_mul(s1, d1);
                    } else {
                        Dl = f2_fma(s, d2, f2_mul(s2, w));
                    }
                } else {
                    A = f2_fma(s, w, A);
                    B = f2_fma(s1, w, B);
                    C = f2_fma(s, d1, C);
                    if constexpr (HESS) {
                        D00 = f2_fma(s2, w, D00);
                        D11 = f2_fma(s, d2, D11);
                        E01 = f2_fma(s1, d1, E01);
                    } else {
                        Dl = f2_fma(s2, w, Dl);
                        Dl = f2_fma(s, d2, Dl);
                    }
                }
            }
        const uint64_t w = f2_dup(w2.w[v2]), d1 = f2_dup(w2.d1[v2]), d2 = f2_dup(w2.d2[v2]);
        o[0] = f2_fma(A, w, o[0]);
        o[1] = f2_fma(B, w, o[1]);
        o[2] = f2_fma(C, w, o[2]);
        o[3] = f2_fma(A, d1, o[3]);
        if constexpr (HESS) {
            o[4] = f2_fma(D00, w, o[4]);
            o[5] = f2_fma(E01, w, o[5]);
            o[6] = f2_fma(B, d1, o[6]);
            o[7] = f2_fma(D11, w, o[7]);
            o[8] = f2_fma(C, d1, o[8]);
            o[9] = f2_fma(A, d2, o[9]);
        } else {
            o[4] = f2_fma(Dl, w, o[4]);
            o[4] = f2_fma(A, d2, o[4]);
        }
    }
}

// Packed 3D slots (f, fx, fy, fz | fxy, fxz, fyz, fxyz): lane h of a pair
// loads half h of each corner row.  Swapping fz (lane 0, position 3) with
// fxy (lane 1, position 0) leaves lane h with the four multi-indices of
// order h along axis 2, at position i = a0 + 2 a1 -- the layout
// blend3_pair_a2 reads.
__device__ __forceinline__ void pair_exchange(unsigned mask, int h, uint64_t (&q)[8][4]) {
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const uint64_t x = h ? q[v][0] : q[v][3];
        const uint64_t y = __shfl_xor_sync(mask, x, 1);
        if (h) q[v][0] = y;
        else q[v][3] = y;
    }
}

// Half-row h of a packed 3D F = 2 row (slots 4h..4h+3, both features) as
// four (feature 0, feature 1) pairs: one 256-bit load for fp32 rows, one
// 128-bit load widened exactly for fp16 rows.
template <typename TT>
__device__ __forceinline__ void load_half_row(const TT* e, uint64_t (&q)[4]) {
    if constexpr (sizeof(TT) == 4) {
        ld_nc_v4b64(e, q);
    } else {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(e));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            q[i] = f2_pack(f.x, f.y);
        }
    }
}

// Lane-pair split for packed 3D F = 2 rows (64 bytes fp32, 32 bytes fp16).
// Lane h of a pair reads the half h of every corner row with one load, so
// one warp instruction covers whole rows (one L1 wavefront per row); one
// slot swap per corner (pair_exchange) then gives lane h the multi-indices
// of order h along axis 2, which it blends with the full separable
// contraction (blend3_pair_a2).  The two features travel as packed pairs
// through f32x2 FMAs (the weights are shared).  The encoding is linear in
// theta, so the pair's partial outputs add up: a reduce-scatter leaves
// feature h's outputs on lane h, which stores them.
// Two 256-thread blocks per SM (at most 128 registers): without the bound
// the full-Hessian variant takes 130 and runs one block per SM (3D, 2^21
// points: 3.87 ms against 2.59 ms bounded; the Laplacian variant also gains
// 4%, 2.31 -> 2.22 ms).
template <typename TT, bool HESS>
__global__ void __launch_bounds__(kBlock, 2) hermite_fwd_pair3_kernel(const __grid_constant__ FwdParams p) {
    constexpr int D = 3, V = 8, S = 4, NO = HESS ? 10 : 5;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = (static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x) >> 1;
    const int lane = threadIdx.x & 1;
    if (n >= p.c.n) return;  // both lanes of a pair share n
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const int64_t lf = static_cast<int64_t>(l) * F + lane;
    if (!((p.c.level_mask >> l) & 1u)) {
        __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, 0.f);
        if (p.dgamma) {
#pragma unroll
            for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, 0.f);
        }
        if constexpr (HESS) {
#pragma unroll
            for (int k = 0; k < 6; ++k) __stcs(p.hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, 0.f);
        } else if (p.lap) {
            __stcs(p.lap + n * p.c.sn + lf * p.c.sf, 0.f);
        }
        return;
    }

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
    const uint64_t keep = l2_evict_last_policy();  // the coordinates, re-read by every level's pass
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(ldg_hint(p.coords + n * D + i, keep), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }
    // half-row h of corner v: 4 slots x (f0, f1) = four 64-bit pairs
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0] + lane * (S * 2);
    uint64_t q[V][S];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const uint32_t g[D] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u)};
        const uint32_t id = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
        load_half_row<TT>(base + static_cast<int64_t>(id) * p.tab.rs[0], q[v]);
    }
    const unsigned mask = __activemask();
    pair_exchange(mask, lane, q);
    uint64_t o[NO];
#pragma unroll
    for (int k = 0; k < NO; ++k) o[k] = 0ull;  // (+0.0f, +0.0f)
    blend3_pair_a2<HESS>(q, B[0], B[1], axis_pick(B[2], lane), o);
    // reduce-scatter across the pair: lane h keeps feature h
    float r[NO];
#pragma unroll
    for (int k = 0; k < NO; ++k) {
        float x, y;
        f2_unpack(o[k], x, y);
        const float mine = lane ? y : x;
        const float other = lane ? x : y;
        r[k] = mine + __shfl_xor_sync(mask, other, 1);
    }
    __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, r[0]);
    if (p.dgamma) {
#pragma unroll
        for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, r[1 + j]);
    }
    if constexpr (HESS) {
#pragma unroll
        for (int k = 0; k < 6; ++k) __stcs(p.hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, r[4 + k]);
    } else if (p.lap) {
        __stcs(p.lap + n * p.c.sn + lf * p.c.sf, r[4]);
    }
}

// Asynchronous 16-byte copies global -> shared (L2 only), and their groups.
__device__ __forceinline__ void async_copy16(void* dst, const void* src) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

constexpr int kPipeBlock = 128;  // threads of a pipelined CTA: 64 points per batch

// The lane-pair forward of hermite_fwd_pair3_kernel, pipelined: persistent
// CTAs walk the batches of one level; each lane copies its eight half-rows
// of the next batch into a private shared-memory slot with cp.async while it
// blends the current batch, so gathers overlap arithmetic without holding
// registers.  Slots are [stage][corner][16-byte chunk][thread], so a warp's
// copies and reads cover consecutive 16-byte words (no bank conflicts); a
// lane reads only what it copied, so its own wait suffices.  Lanes past the
// last point copy the last point's rows and store nothing.  The slot swap
// and the blend are hermite_fwd_pair3_kernel's, so the outputs are
// bit-identical.
// Used for fp16 tables, whose half-row is one 16-byte copy: 3D fp16 workload
// (2^23 points, 10 active levels) 6.55 -> 5.63 ms, full Hessian 7.11 -> 6.95
// ms.  An fp32 half-row (32 bytes) takes two 16-byte copies, i.e. twice the
// L2 requests of one 256-bit load, and the kernel is bound by them: the 3D
// fp32 workload ran 2.26 -> 4.26 ms, so fp32 stays on the unpipelined kernel.
template <typename TT, bool HESS>
__global__ void __launch_bounds__(kPipeBlock) hermite_fwd_pipe3_kernel(const __grid_constant__ FwdParams p) {
    constexpr int D = 3, V = 8, S = 4, NO = HESS ? 10 : 5;
    constexpr int CH = S * 2 * static_cast<int>(sizeof(TT)) / 16;  // 16-byte chunks per half-row
    constexpr int PB = kPipeBlock / 2;                                 // points per batch
    extern __shared__ uint4 slots[];                                   // [2][V][CH][kPipeBlock]
    const int l = p.c.lvl[blockIdx.y];
    const int lane = threadIdx.x & 1;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const int64_t lf = static_cast<int64_t>(l) * F + lane;
    const int64_t batches = (p.c.n + PB - 1) / PB;
    if (!((p.c.level_mask >> l) & 1u)) {
        for (int64_t b = blockIdx.x; b < batches; b += gridDim.x) {
            const int64_t n = b * PB + (threadIdx.x >> 1);
            if (n >= p.c.n) continue;
            __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, 0.f);
            if (p.dgamma) {
#pragma unroll
                for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, 0.f);
            }
            if constexpr (HESS) {
#pragma unroll
                for (int k = 0; k < 6; ++k) __stcs(p.hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, 0.f);
            } else if (p.lap) {
                __stcs(p.lap + n * p.c.sn + lf * p.c.sf, 0.f);
            }
        }
        return;
    }
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0] + lane * (S * 2);
    auto point_of = [&](int64_t b) {
        const int64_t n = b * PB + (threadIdx.x >> 1);
        return n < p.c.n ? n : p.c.n - 1;
    };
    auto issue = [&](int64_t b, int st) {
        const int64_t n = point_of(b);
        uint32_t c[D];
        float t[D];
#pragma unroll
        for (int i = 0; i < D; ++i) locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const uint32_t g[D] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u)};
            const uint32_t id = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
            const TT* e = base + static_cast<int64_t>(id) * p.tab.rs[0];
#pragma unroll
            for (int ch = 0; ch < CH; ++ch)
                async_copy16(&slots[((st * V + v) * CH + ch) * kPipeBlock + threadIdx.x], e + ch * (16 / sizeof(TT)));
        }
    };
    int64_t b = blockIdx.x;
    if (b < batches) issue(b, 0);
    async_commit();
    int st = 0;
    for (; b < batches; b += gridDim.x) {
        if (b + gridDim.x < batches) issue(b + gridDim.x, st ^ 1);
        async_commit();
        async_wait<1>();  // this lane's copies of batch b have landed
        const int64_t n = b * PB + (threadIdx.x >> 1);
        uint32_t c[D];
        float t[D];
        Basis1 B[D];
#pragma unroll
        for (int i = 0; i < D; ++i) {
            locate(__ldg(p.coords + point_of(b) * D + i), lv, c[i], t[i]);
            B[i] = hermite_basis(t[i], lv);
        }
        uint64_t q[V][S];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            if constexpr (sizeof(TT) == 4) {
#pragma unroll
                for (int ch = 0; ch < CH; ++ch) {
                    const uint4 r = slots[((st * V + v) * CH + ch) * kPipeBlock + threadIdx.x];
                    q[v][2 * ch] = f2_pack(__uint_as_float(r.x), __uint_as_float(r.y));
                    q[v][2 * ch + 1] = f2_pack(__uint_as_float(r.z), __uint_as_float(r.w));
                }
            } else {
                const uint4 r = slots[(st * V + v) * kPipeBlock + threadIdx.x];
                const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
                    q[v][i] = f2_pack(f.x, f.y);
                }
            }
        }
        pair_exchange(0xffffffffu, lane, q);
        uint64_t o[NO];
#pragma unroll
        for (int k = 0; k < NO; ++k) o[k] = 0ull;  // (+0.0f, +0.0f)
        blend3_pair_a2<HESS>(q, B[0], B[1], axis_pick(B[2], lane), o);
        float r[NO];
#pragma unroll
        for (int k = 0; k < NO; ++k) {
            float x, y;
            f2_unpack(o[k], x, y);
            const float mine = lane ? y : x;
            const float other = lane ? x : y;
            r[k] = mine + __shfl_xor_sync(0xffffffffu, other, 1);
        }
        if (n < p.c.n) {
            __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, r[0]);
            if (p.dgamma) {
#pragma unroll
                for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, r[1 + j]);
            }
            if constexpr (HESS) {
#pragma unroll
                for (int k = 0; k < 6; ++k) __stcs(p.hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, r[4 + k]);
            } else if (p.lap) {
                __stcs(p.lap + n * p.c.sn + lf * p.c.sf, r[4]);
            }
        }
        st ^= 1;
    }
    async_wait<0>();
}

// 4D (space-time) forward, any layout and F: one thread per (point, level),
// one feature at a time.  The 4D blend is a sum over the four axis-3
// slices (corner side v3, basis order a3): each slice is a 3D blend of the
// 8 x 8 coefficients with v3 and alpha_3 fixed, and its outputs take the
// axis-3 weight w, w' or w'' (the product rule of the tensor basis):
//   gamma += G w,  d/dx_j += dG_j w (j < 3),  d/dx_3 += G w',
//   lap += lap3 w + G w'',
//   Hessian: the slice's (i, j < 3) entries times w, (j, 3) entries dG_j w',
//   (3, 3) entry G w''.
// Element loads: the 256 coefficients of a (point, level, feature) are read
// one slice (64) at a time.
template <typename TT, bool HESS>
__global__ void __launch_bounds__(kBlock) hermite_fwd4_kernel(const __grid_constant__ FwdParams p) {
    constexpr int D = 4, P = 10;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const bool active = (p.c.level_mask >> l) & 1u;

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }
    for (int f = 0; f < F; ++f) {
        float g = 0.f, dg[4] = {0.f, 0.f, 0.f, 0.f}, lap = 0.f, h[P];
#pragma unroll
        for (int k = 0; k < P; ++k) h[k] = 0.f;
        if (active) {
#pragma unroll 1
            for (int v3 = 0; v3 < 2; ++v3) {
                // indices of the slice's 8 corners in the five order tables
                uint32_t idx[8][5];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint32_t gv[D] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u),
                                            c[3] + static_cast<uint32_t>(v3)};
#pragma unroll
                    for (int k = 0; k <= D; ++k) idx[v][k] = vertex_index<D>(gv, lv, (lv.dense >> k) & 1u, p.c.tmask[k]);
                }
#pragma unroll
                for (int a3 = 0; a3 < 2; ++a3) {
                    float q[8][8];
#pragma unroll
                    for (int v = 0; v < 8; ++v)
#pragma unroll
                        for (int a = 0; a < 8; ++a) {
                            const int alpha = a + 8 * a3, k = alpha_order(alpha);
                            const TT* e = static_cast<const TT*>(p.tab.ptr[k]) + l * p.tab.ls[k] +
                                          static_cast<int64_t>(idx[v][k]) * p.tab.rs[k] + bucket_slot<D>(alpha) * F + f;
                            q[v][a] = to_f32<TT>(*e);
                        }
                    const float w = B[3].w[v3][a3], w1 = B[3].d1[v3][a3], w2 = B[3].d2[v3][a3];
                    float sg, sdg[3];
                    if constexpr (HESS) {
                        float sh[6];
                        blend3h(q, B[0], B[1], B[2], sg, sdg, sh);
                        h[0] = fmaf(sh[0], w, h[0]);
                        h[1] = fmaf(sh[1], w, h[1]);
                        h[2] = fmaf(sh[2], w, h[2]);
                        h[3] = fmaf(sdg[0], w1, h[3]);
                        h[4] = fmaf(sh[3], w, h[4]);
                        h[5] = fmaf(sh[4], w, h[5]);
                        h[6] = fmaf(sdg[1], w1, h[6]);
                        h[7] = fmaf(sh[5], w, h[7]);
                        h[8] = fmaf(sdg[2], w1, h[8]);
                        h[9] = fmaf(sg, w2, h[9]);
                    } else {
                        float sl;
                        blend3(q, B[0], B[1], B[2], sg, sdg, sl);
                        lap = fmaf(sl, w, fmaf(sg, w2, lap));
                    }
                    g = fmaf(sg, w, g);
#pragma unroll
                    for (int j = 0; j < 3; ++j) dg[j] = fmaf(sdg[j], w, dg[j]);
                    dg[3] = fmaf(sg, w1, dg[3]);
                }
            }
        }
        const int64_t lf = static_cast<int64_t>(l) * F + f;
        __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, g);
        if (p.dgamma) {
#pragma unroll
            for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, dg[j]);
        }
        if constexpr (HESS) {
#pragma unroll
            for (int k = 0; k < P; ++k) __stcs(p.hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, h[k]);
        } else if (p.lap) {
            __stcs(p.lap + n * p.c.sn + lf * p.c.sf, lap);
        }
    }
}

// Reduce-scatter of NV per-lane partial sums over the 4 lanes of an item
// (lanes 4i..4i+3 of the warp, all present in `mask`): lane (b1, b0) ends
// with the sums of flat entries b1*NV/2 + b0*NV/4 + k, k < NV/4.  Index
// choices are compile-time; the lane bits only select between two values.
template <int NV>
__device__ __forceinline__ void reduce_scatter4(unsigned mask, int lane, const float (&x)[NV], float (&y)[NV / 4]) {
    static_assert(NV % 4 == 0, "pad to a multiple of 4");
    constexpr int H = NV / 2, Q = NV / 4;
    const bool b1 = lane & 2, b0 = lane & 1;
    float z[H];
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const float mine = b1 ? x[k + H] : x[k], other = b1 ? x[k] : x[k + H];
        z[k] = mine + __shfl_xor_sync(mask, other, 2);
    }
#pragma unroll
    for (int k = 0; k < Q; ++k) {
        const float mine = b0 ? z[k + Q] : z[k], other = b0 ? z[k] : z[k + Q];
        y[k] = mine + __shfl_xor_sync(mask, other, 1);
    }
}

// Store flat output entry j = 2 * o + f of a 4D F = 2 item: o = 0 gamma,
// 1..4 d/dx_0..3, 5 the Laplacian (or 5..14 the Hessian entries).
template <bool HESS>
__device__ __forceinline__ void store4(const FwdParams& p, int64_t n, int l, int j, float v) {
    const int o = j >> 1;
    const int64_t lf = static_cast<int64_t>(l) * 2 + (j & 1);
    if (o == 0) {
        __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, v);
    } else if (o <= 4) {
        if (p.dgamma) __stcs(p.dgamma + n * p.c.dsn + (o - 1) * p.c.dsj + lf * p.c.dsf, v);
    } else if (HESS) {
        if (o < 15) __stcs(p.hess + n * p.c.hsn + (o - 5) * p.c.hsq + lf * p.c.hsf, v);
    } else if (o == 5 && p.lap) {
        __stcs(p.lap + n * p.c.sn + lf * p.c.sf, v);
    }
}

// Lane-quad forward for packed 4D F = 2 rows (128 bytes fp32, 64 bytes
// fp16).  Lane g of a quad reads the quarter g of every corner row (slots
// 4g..4g+3, both features: one 256-bit or 128-bit load), so one warp load
// covers whole rows.  The 16 corners are taken as two axis-3 halves: each
// half is blended over axes 0-2 with the 3D unit blend (f32x2, both
// features at once) and folded into the 4D outputs with the axis-3 weight of
// the slot's order along axis 3 (w, w' or w'', as in hermite_fwd4_kernel).
// A reduce-scatter over the quad leaves each lane a quarter of the outputs.
// Two blocks per SM (128 registers, a few spilled words): 5.39 ms on the 4D
// workload (2^20 points), against 6.53 ms at one block without spills.
template <typename TT, bool HESS>
__global__ void __launch_bounds__(kBlock, 2) hermite_fwd_quad4_kernel(const __grid_constant__ FwdParams p) {
    constexpr int D = 4, G = 4, S = 4, NO = HESS ? 15 : 6, NV = (2 * NO + 3) / 4 * 4;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t first = (static_cast<int64_t>(blockIdx.x) * kBlock + (threadIdx.x & ~31u)) / G;
    const int64_t n = (static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x) / G;
    const int lane = threadIdx.x % G;
    if (n >= p.c.n) return;  // all four lanes share n
    const unsigned mask = item_lanes<G>(first, p.c.n);
    const Level& lv = p.c.lv[l];
    float x[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) x[k] = 0.f;
    if ((p.c.level_mask >> l) & 1u) {
        uint32_t c[D];
        float t[D];
        Basis1 B[D];
#pragma unroll
        for (int i = 0; i < D; ++i) {
            locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
            B[i] = hermite_basis(t[i], lv);
        }
        const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0] + lane * (S * 2);
        uint64_t o[NO];
#pragma unroll
        for (int k = 0; k < NO; ++k) o[k] = 0ull;
#pragma unroll
        for (int v3 = 0; v3 < 2; ++v3) {
            uint64_t q[8][S];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint32_t g[D] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u),
                                       c[3] + static_cast<uint32_t>(v3)};
                const uint32_t id = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
                load_half_row<TT>(base + static_cast<int64_t>(id) * p.tab.rs[0], q[v]);
            }
#pragma unroll
            for (int u = 0; u < S; ++u) {
                const AxisW2 W0 = axis_dup(unit_axis<D, G>(B[0], lane, u, 0));
                const AxisW2 W1 = axis_dup(unit_axis<D, G>(B[1], lane, u, 1));
                const AxisW2 W2 = axis_dup(unit_axis<D, G>(B[2], lane, u, 2));
                const AxisW W3 = unit_axis<D, G>(B[3], lane, u, 3);
                const uint64_t w = f2_dup(W3.w[v3]), w1 = f2_dup(W3.d1[v3]), w2 = f2_dup(W3.d2[v3]);
                uint64_t cv[8];
#pragma unroll
                for (int v = 0; v < 8; ++v) cv[v] = q[v][u];
                if constexpr (HESS) {
                    uint64_t s3[10];
#pragma unroll
                    for (int k = 0; k < 10; ++k) s3[k] = 0ull;
                    unit_blend3_f2_hess(cv, W0, W1, W2, s3);  // gamma, d0..d2, xx xy xz yy yz zz
                    o[0] = f2_fma(s3[0], w, o[0]);
#pragma unroll
                    for (int j = 1; j < 4; ++j) o[j] = f2_fma(s3[j], w, o[j]);
                    o[4] = f2_fma(s3[0], w1, o[4]);
                    // 4D Hessian (o[5..14]): xx xy xz xw yy yz yw zz zw ww
                    o[5] = f2_fma(s3[4], w, o[5]);
                    o[6] = f2_fma(s3[5], w, o[6]);
                    o[7] = f2_fma(s3[6], w, o[7]);
                    o[8] = f2_fma(s3[1], w1, o[8]);
                    o[9] = f2_fma(s3[7], w, o[9]);
                    o[10] = f2_fma(s3[8], w, o[10]);
                    o[11] = f2_fma(s3[2], w1, o[11]);
                    o[12] = f2_fma(s3[9], w, o[12]);
                    o[13] = f2_fma(s3[3], w1, o[13]);
                    o[14] = f2_fma(s3[0], w2, o[14]);
                } else {
                    uint64_t s3[5] = {0ull, 0ull, 0ull, 0ull, 0ull};
                    unit_blend3_f2(cv, W0, W1, W2, s3);       // gamma, d0..d2, lap over axes 0-2
                    o[0] = f2_fma(s3[0], w, o[0]);
#pragma unroll
                    for (int j = 1; j < 4; ++j) o[j] = f2_fma(s3[j], w, o[j]);
                    o[4] = f2_fma(s3[0], w1, o[4]);
                    o[5] = f2_fma(s3[4], w, f2_fma(s3[0], w2, o[5]));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < NO; ++k) f2_unpack(o[k], x[2 * k], x[2 * k + 1]);
    }
    float y[NV / 4];
    reduce_scatter4<NV>(mask, lane, x, y);
    const int j0 = (lane >> 1) * (NV / 2) + (lane & 1) * (NV / 4);
#pragma unroll
    for (int k = 0; k < NV / 4; ++k) store4<HESS>(p, n, l, j0 + k, y[k]);
}

template <int D, int FC, typename TT, bool VEC, bool HESS>
cudaError_t launch(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    hermite_fwd_kernel<D, FC, TT, VEC, HESS><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, int FC, typename TT, bool HESS>
cudaError_t pick_vec(const FwdParams& p, bool vec, cudaStream_t s) {
    return vec ? launch<D, FC, TT, true, HESS>(p, s) : launch<D, FC, TT, false, HESS>(p, s);
}

template <int D, typename TT, bool HESS>
cudaError_t pick_fc(const FwdParams& p, int fc, bool vec, cudaStream_t s) {
    return fc == 2 ? pick_vec<D, 2, TT, HESS>(p, vec, s) : pick_vec<D, 1, TT, HESS>(p, vec, s);
}

template <typename TT, bool HESS>
cudaError_t launch_pair3(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n * 2 + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    hermite_fwd_pair3_kernel<TT, HESS><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

// One wave of persistent pipelined CTAs per level (level-major dispatch: the
// first wave walks level 0's batches while the next level's CTAs wait).  The
// SM count and the occupancy are read for the current device on every call
// (host-side queries of a few microseconds), so nothing is cached between
// calls, threads or devices.
template <typename TT, bool HESS>
cudaError_t launch_pipe3(const FwdParams& p, cudaStream_t s) {
    constexpr int kSmem = 2 * 8 * (4 * 2 * static_cast<int>(sizeof(TT)) / 16) * kPipeBlock * 16;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hermite_fwd_pipe3_kernel<TT, HESS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hermite_fwd_pipe3_kernel<TT, HESS>, kPipeBlock,
                                                          kSmem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t batches = (p.c.n + kPipeBlock / 2 - 1) / (kPipeBlock / 2);
    const int64_t ctas = std::min<int64_t>(batches, static_cast<int64_t>(sms) * per_sm);
    dim3 grid(static_cast<unsigned>(ctas), static_cast<unsigned>(p.c.nlvl));
    hermite_fwd_pipe3_kernel<TT, HESS><<<grid, kPipeBlock, kSmem, s>>>(p);
    return cudaGetLastError();
}

template <typename TT, bool HESS>
cudaError_t launch4(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    hermite_fwd4_kernel<TT, HESS><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename TT, bool HESS>
cudaError_t launch_quad4(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n * 4 + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    hermite_fwd_quad4_kernel<TT, HESS><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <bool HESS>
cudaError_t dispatch(const FwdParams& p, int fc, bool vec, int dtype, cudaStream_t s) {
    if (p.c.d == 4 && vec && p.c.F == 2)
        return dtype == HG_F16 ? launch_quad4<__half, HESS>(p, s) : launch_quad4<float, HESS>(p, s);
    if (p.c.d == 4) return dtype == HG_F16 ? launch4<__half, HESS>(p, s) : launch4<float, HESS>(p, s);
    if (vec && p.c.d == 3 && p.c.F == 2)
        return dtype == HG_F16 ? launch_pipe3<__half, HESS>(p, s) : launch_pair3<float, HESS>(p, s);
    if (p.c.d == 2)
        return dtype == HG_F16 ? pick_fc<2, __half, HESS>(p, fc, vec, s) : pick_fc<2, float, HESS>(p, fc, vec, s);
    return dtype == HG_F16 ? pick_fc<3, __half, HESS>(p, fc, vec, s) : pick_fc<3, float, HESS>(p, fc, vec, s);
}

}  // namespace

int launch_hermite_fwd(const FwdParams& p, int fc, bool vec, int dtype, bool hess, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return hess ? dispatch<true>(p, fc, vec, dtype, s) : dispatch<false>(p, fc, vec, dtype, s);
}

}  // namespace hg
