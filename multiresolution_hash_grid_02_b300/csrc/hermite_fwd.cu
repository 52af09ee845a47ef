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

#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;

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

// Contribution of one packed slot (multi-index alpha, with the weights
// W0..W2 of its per-axis orders) to the 3D outputs, for both features at
// once: c[v] is the slot's (feature 0, feature 1) coefficient pair at corner
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
// one warp instruction covers whole rows (one L1 wavefront per row), and
// blends the four slots of that half.  The two features travel as packed
// pairs through f32x2 FMAs (the weights are shared).  The encoding is linear
// in theta, so the pair's partial outputs add up: a reduce-scatter leaves
// feature h's outputs on lane h, which stores them.
// Two 256-thread blocks per SM (at most 128 registers): without the bound
// the full-Hessian variant takes 130 and runs one block per SM (3D, 2^21
// points: 3.87 ms against 2.59 ms bounded; the Laplacian variant also gains
// 4%, 2.31 -> 2.22 ms).
template <typename TT, bool HESS>
__global__ void __launch_bounds__(kBlock, 2) hermite_fwd_pair3_kernel(const __grid_constant__ FwdParams p) {
    constexpr int D = 3, V = 8, G = 2, S = 4, NO = HESS ? 10 : 5;
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
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
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
    uint64_t o[NO];
#pragma unroll
    for (int k = 0; k < NO; ++k) o[k] = 0ull;  // (+0.0f, +0.0f)
#pragma unroll
    for (int u = 0; u < S; ++u) {
        const AxisW2 W0 = axis_dup(unit_axis<D, G>(B[0], lane, u, 0));
        const AxisW2 W1 = axis_dup(unit_axis<D, G>(B[1], lane, u, 1));
        const AxisW2 W2 = axis_dup(unit_axis<D, G>(B[2], lane, u, 2));
        uint64_t cv[V];
#pragma unroll
        for (int v = 0; v < V; ++v) cv[v] = q[v][u];
        if constexpr (HESS) {
            unit_blend3_f2_hess(cv, W0, W1, W2, o);
        } else {
            unit_blend3_f2(cv, W0, W1, W2, o);
        }
    }
    // reduce-scatter across the pair: lane h keeps feature h
    const unsigned mask = __activemask();
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

template <bool HESS>
cudaError_t dispatch(const FwdParams& p, int fc, bool vec, int dtype, cudaStream_t s) {
    if (vec && p.c.d == 3 && p.c.F == 2)
        return dtype == HG_F16 ? launch_pair3<__half, HESS>(p, s) : launch_pair3<float, HESS>(p, s);
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
