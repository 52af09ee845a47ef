// Hermite-NGP backward: scatter-add the coefficient gradients of every
// (point, level) into the order-bucketed gradient tables.
//
// "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
// 整体框架 (the flowchart's backward pass updates the hash coefficients theta)
// and 关键设计 1 (the encoding is linear in theta, so the backward is the
// transpose of the forward's blend).  Colliding entries add their gradients
// ("英偉達將訓練 NeRF 模型從 5 小時縮至 5 秒", the hashed levels).
//
// Mapping as in the forward (one thread per (point, level), grid.y = level,
// so a level's gradient table stays resident in L2 while it is accumulated).
// The transpose runs the separable blend backwards (axis 2, then 1, then 0)
// and yields all 2^d x 2^d coefficient gradients of a feature in registers;
// the packed layout then issues one 16-byte vector RED per four floats.
// The full-Hessian variant (HESS) takes the upstream gradient of every
// second derivative instead of the Laplacian's, and transposes the
// forward's split second-order sums.
#include <cuda_runtime.h>

#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;

// Transposed 2D blend: upstream (gg, gd[0..1], gl) -> qb[corner][alpha].
__device__ __forceinline__ void blend2_t(float gg, const float (&gd)[3], float gl, const Basis1& b0,
                                         const Basis1& b1, float (&qb)[4][4]) {
#pragma unroll
    for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
        for (int a1 = 0; a1 < 2; ++a1) {
            const float s = fmaf(gg, b1.w[v1][a1], fmaf(gd[1], b1.d1[v1][a1], gl * b1.d2[v1][a1]));
            const float s1 = gd[0] * b1.w[v1][a1];
            const float s2 = gl * b1.w[v1][a1];
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                for (int a0 = 0; a0 < 2; ++a0)
                    qb[v0 + 2 * v1][a0 + 2 * a1] = fmaf(s, b0.w[v0][a0], fmaf(s1, b0.d1[v0][a0], s2 * b0.d2[v0][a0]));
        }
}

// Transposed 3D blend.
__device__ __forceinline__ void blend3_t(float gg, const float (&gd)[3], float gl, const Basis1& b0,
                                         const Basis1& b1, const Basis1& b2, float (&qb)[8][8]) {
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2)
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2) {
            const float A = fmaf(gg, b2.w[v2][a2], fmaf(gd[2], b2.d1[v2][a2], gl * b2.d2[v2][a2]));
            const float B = gd[0] * b2.w[v2][a2];
            const float C = gd[1] * b2.w[v2][a2];
            const float Dl = gl * b2.w[v2][a2];
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
                for (int a1 = 0; a1 < 2; ++a1) {
                    const float s = fmaf(A, b1.w[v1][a1], fmaf(C, b1.d1[v1][a1], Dl * b1.d2[v1][a1]));
                    const float s1 = B * b1.w[v1][a1];
                    const float s2 = Dl * b1.w[v1][a1];
#pragma unroll
                    for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                        for (int a0 = 0; a0 < 2; ++a0)
                            qb[v0 + 2 * v1 + 4 * v2][a0 + 2 * a1 + 4 * a2] =
                                fmaf(s, b0.w[v0][a0], fmaf(s1, b0.d1[v0][a0], s2 * b0.d2[v0][a0]));
                }
        }
}

// Transposed 2D blend with the full Hessian: upstream (gg, gd[0..1],
// gh = (xx, xy, yy)) -> qb[corner][alpha].
__device__ __forceinline__ void blend2h_t(float gg, const float (&gd)[3], const float (&gh)[6], const Basis1& b0,
                                          const Basis1& b1, float (&qb)[4][4]) {
#pragma unroll
    for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
        for (int a1 = 0; a1 < 2; ++a1) {
            const float s = fmaf(gg, b1.w[v1][a1], fmaf(gd[1], b1.d1[v1][a1], gh[2] * b1.d2[v1][a1]));
            const float s1 = fmaf(gd[0], b1.w[v1][a1], gh[1] * b1.d1[v1][a1]);
            const float s2 = gh[0] * b1.w[v1][a1];
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                for (int a0 = 0; a0 < 2; ++a0)
                    qb[v0 + 2 * v1][a0 + 2 * a1] = fmaf(s, b0.w[v0][a0], fmaf(s1, b0.d1[v0][a0], s2 * b0.d2[v0][a0]));
        }
}

// Transposed 3D blend with the full Hessian, gh = (xx, xy, xz, yy, yz, zz):
// the adjoints of the forward's sums A, B, C, D00, D11, E01 per (v2, a2),
// then of s, s1, s2 per (v1, a1).
__device__ __forceinline__ void blend3h_t(float gg, const float (&gd)[3], const float (&gh)[6], const Basis1& b0,
                                          const Basis1& b1, const Basis1& b2, float (&qb)[8][8]) {
#pragma unroll
    for (int v2 = 0; v2 < 2; ++v2)
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2) {
            const float A = fmaf(gg, b2.w[v2][a2], fmaf(gd[2], b2.d1[v2][a2], gh[5] * b2.d2[v2][a2]));
            const float B = fmaf(gd[0], b2.w[v2][a2], gh[2] * b2.d1[v2][a2]);
            const float C = fmaf(gd[1], b2.w[v2][a2], gh[4] * b2.d1[v2][a2]);
            const float D00 = gh[0] * b2.w[v2][a2];
            const float D11 = gh[3] * b2.w[v2][a2];
            const float E01 = gh[1] * b2.w[v2][a2];
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1)
#pragma unroll
                for (int a1 = 0; a1 < 2; ++a1) {
                    const float s = fmaf(A, b1.w[v1][a1], fmaf(C, b1.d1[v1][a1], D11 * b1.d2[v1][a1]));
                    const float s1 = fmaf(B, b1.w[v1][a1], E01 * b1.d1[v1][a1]);
                    const float s2 = D00 * b1.w[v1][a1];
#pragma unroll
                    for (int v0 = 0; v0 < 2; ++v0)
#pragma unroll
                        for (int a0 = 0; a0 < 2; ++a0)
                            qb[v0 + 2 * v1 + 4 * v2][a0 + 2 * a1 + 4 * a2] =
                                fmaf(s, b0.w[v0][a0], fmaf(s1, b0.d1[v0][a0], s2 * b0.d2[v0][a0]));
                }
        }
}

// One upstream value.  With the full Hessian (twice the upstream bytes) the
// upstream values are loaded evict-first: read once, they should not push the
// level's gradient rows and the coordinates out of the L2 (3D workload: 4.13
// -> 3.94 ms).  The Laplacian backward keeps default caching: with the hints
// its DRAM reads drop from 2.05 to 1.79 GB per launch, but the L2, not DRAM,
// bounds it, and it ran 2 % slower (3.31 against 3.23 ms).
template <bool HESS>
__device__ __forceinline__ float ld_upstream(const float* a, uint64_t once) {
    if constexpr (HESS) return ldg_hint(a, once);
    return __ldg(a);
}

// Upstream gradients of one (point, level, feature): gamma, grad, and the
// Laplacian's (gl) or, under HESS, every Hessian entry's (gh[0..P-1]).
template <int D, bool HESS>
__device__ __forceinline__ void load_upstream(const BwdParams& p, int64_t n, int64_t lf, float& gg, float (&gd)[3],
                                              float& gl, float (&gh)[6]) {
    const uint64_t once = HESS ? l2_evict_first_policy() : 0ull;
    gg = p.g_gamma ? ld_upstream<HESS>(p.g_gamma + n * p.c.sn + lf * p.c.sf, once) : 0.f;
#pragma unroll
    for (int j = 0; j < 3; ++j)
        gd[j] = (p.g_dgamma && j < D) ? ld_upstream<HESS>(p.g_dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, once)
                                      : 0.f;
    gl = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) gh[k] = 0.f;
    if constexpr (HESS) {
        if (p.g_hess) {
#pragma unroll
            for (int k = 0; k < D * (D + 1) / 2; ++k)
                gh[k] = ld_upstream<HESS>(p.g_hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, once);
        }
    } else {
        gl = p.g_lap ? ld_upstream<HESS>(p.g_lap + n * p.c.sn + lf * p.c.sf, once) : 0.f;
    }
}

template <int D, int FC, bool VEC, bool HESS>
__global__ void __launch_bounds__(kBlock) hermite_bwd_kernel(const __grid_constant__ BwdParams p) {
    constexpr int V = 1 << D;
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }

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
        float qb[FC][V][V];
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
            float gg, gd[3], gl, gh[6];
            load_upstream<D, HESS>(p, n, lf, gg, gd, gl, gh);
            if constexpr (HESS) {
                if constexpr (D == 2) {
                    blend2h_t(gg, gd, gh, B[0], B[1], qb[f]);
                } else {
                    blend3h_t(gg, gd, gh, B[0], B[1], B[D - 1], qb[f]);
                }
            } else if constexpr (D == 2) {
                blend2_t(gg, gd, gl, B[0], B[1], qb[f]);
            } else {
                blend3_t(gg, gd, gl, B[0], B[1], B[D - 1], qb[f]);
            }
        }
        if constexpr (VEC) {
            // packed row: [slot][FC] floats, 16-byte aligned, length V*FC (a multiple of 4)
            float* row0 = p.grad.ptr[0] + l * p.grad.ls[0];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                float r[V * FC];
#pragma unroll
                for (int a = 0; a < V; ++a)
#pragma unroll
                    for (int f = 0; f < FC; ++f) r[packed_slot<D>(a) * FC + f] = qb[f][v][a];
                float* dst = row0 + static_cast<int64_t>(idx[0][v]) * p.grad.rs[0];
#pragma unroll
                for (int i = 0; i < V * FC; i += 4) red_add_v4(dst + i, r[i], r[i + 1], r[i + 2], r[i + 3]);
            }
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int a = 0; a < V; ++a) {
                    const int k = alpha_order(a);
                    float* e = p.grad.ptr[k] + l * p.grad.ls[k] + static_cast<int64_t>(idx[k][v]) * p.grad.rs[k] +
                               bucket_slot<D>(a) * F + f0;
#pragma unroll
                    for (int f = 0; f < FC; ++f) red_add_f32(e + f, qb[f][v][a]);
                }
        }
    }
}

// Transposed blend of one packed slot (one alpha, weights W0..W1[..W2]) of
// one feature: qb[v] = d(loss)/d theta at corner v, from the upstream
// gradients (gg, gd[], gl).  The same separable order as blend3_t / blend2_t,
// restricted to one alpha.
template <int D>
__device__ __forceinline__ void unit_blend_t(float gg, const float (&gd)[3], float gl, const AxisW& W0,
                                             const AxisW& W1, const AxisW& W2, float (&qb)[1 << D]) {
    if constexpr (D == 3) {
#pragma unroll
        for (int v2 = 0; v2 < 2; ++v2) {
            const float A = fmaf(gg, W2.w[v2], fmaf(gd[2], W2.d1[v2], gl * W2.d2[v2]));
            const float B = gd[0] * W2.w[v2];
            const float C = gd[1] * W2.w[v2];
            const float Dl = gl * W2.w[v2];
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1) {
                const float s = fmaf(A, W1.w[v1], fmaf(C, W1.d1[v1], Dl * W1.d2[v1]));
                const float s1 = B * W1.w[v1];
                const float s2 = Dl * W1.w[v1];
#pragma unroll
                for (int v0 = 0; v0 < 2; ++v0)
                    qb[v0 + 2 * v1 + 4 * v2] = fmaf(s, W0.w[v0], fmaf(s1, W0.d1[v0], s2 * W0.d2[v0]));
            }
        }
    } else {
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1) {
            const float s = fmaf(gg, W1.w[v1], fmaf(gd[1], W1.d1[v1], gl * W1.d2[v1]));
            const float s1 = gd[0] * W1.w[v1];
            const float s2 = gl * W1.w[v1];
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0) qb[v0 + 2 * v1] = fmaf(s, W0.w[v0], fmaf(s1, W0.d1[v0], s2 * W0.d2[v0]));
        }
    }
}

// The same transposed blend for both features at once (F = 2): the upstream
// gradients are (feature 0, feature 1) pairs, the weights are shared, and
// each f32x2 operation is exactly the two fp32 operations above.
template <int D>
__device__ __forceinline__ void unit_blend_t_f2(uint64_t gg, const uint64_t (&gd)[3], uint64_t gl, const AxisW2& W0,
                                                const AxisW2& W1, const AxisW2& W2, uint64_t (&qb)[1 << D]) {
    if constexpr (D == 3) {
#pragma unroll
        for (int v2 = 0; v2 < 2; ++v2) {
            const uint64_t A = f2_fma(gg, W2.w[v2], f2_fma(gd[2], W2.d1[v2], f2_mul(gl, W2.d2[v2])));
            const uint64_t B = f2_mul(gd[0], W2.w[v2]);
            const uint64_t C = f2_mul(gd[1], W2.w[v2]);
            const uint64_t Dl = f2_mul(gl, W2.w[v2]);
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1) {
                const uint64_t s = f2_fma(A, W1.w[v1], f2_fma(C, W1.d1[v1], f2_mul(Dl, W1.d2[v1])));
                const uint64_t s1 = f2_mul(B, W1.w[v1]);
                const uint64_t s2 = f2_mul(Dl, W1.w[v1]);
#pragma unroll
                for (int v0 = 0; v0 < 2; ++v0)
                    qb[v0 + 2 * v1 + 4 * v2] = f2_fma(s, W0.w[v0], f2_fma(s1, W0.d1[v0], f2_mul(s2, W0.d2[v0])));
            }
        }
    } else {
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1) {
            const uint64_t s = f2_fma(gg, W1.w[v1], f2_fma(gd[1], W1.d1[v1], f2_mul(gl, W1.d2[v1])));
            const uint64_t s1 = f2_mul(gd[0], W1.w[v1]);
            const uint64_t s2 = f2_mul(gl, W1.w[v1]);
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0)
                qb[v0 + 2 * v1] = f2_fma(s, W0.w[v0], f2_fma(s1, W0.d1[v0], f2_mul(s2, W0.d2[v0])));
        }
    }
}

// unit_blend_t with the full Hessian (gh in the order of blend2h_t /
// blend3h_t).
template <int D>
__device__ __forceinline__ void unit_blend_t_hess(float gg, const float (&gd)[3], const float (&gh)[6],
                                                  const AxisW& W0, const AxisW& W1, const AxisW& W2,
                                                  float (&qb)[1 << D]) {
    if constexpr (D == 3) {
#pragma unroll
        for (int v2 = 0; v2 < 2; ++v2) {
            const float A = fmaf(gg, W2.w[v2], fmaf(gd[2], W2.d1[v2], gh[5] * W2.d2[v2]));
            const float B = fmaf(gd[0], W2.w[v2], gh[2] * W2.d1[v2]);
            const float C = fmaf(gd[1], W2.w[v2], gh[4] * W2.d1[v2]);
            const float D00 = gh[0] * W2.w[v2];
            const float D11 = gh[3] * W2.w[v2];
            const float E01 = gh[1] * W2.w[v2];
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1) {
                const float s = fmaf(A, W1.w[v1], fmaf(C, W1.d1[v1], D11 * W1.d2[v1]));
                const float s1 = fmaf(B, W1.w[v1], E01 * W1.d1[v1]);
                const float s2 = D00 * W1.w[v1];
#pragma unroll
                for (int v0 = 0; v0 < 2; ++v0)
                    qb[v0 + 2 * v1 + 4 * v2] = fmaf(s, W0.w[v0], fmaf(s1, W0.d1[v0], s2 * W0.d2[v0]));
            }
        }
    } else {
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1) {
            const float s = fmaf(gg, W1.w[v1], fmaf(gd[1], W1.d1[v1], gh[2] * W1.d2[v1]));
            const float s1 = fmaf(gd[0], W1.w[v1], gh[1] * W1.d1[v1]);
            const float s2 = gh[0] * W1.w[v1];
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0) qb[v0 + 2 * v1] = fmaf(s, W0.w[v0], fmaf(s1, W0.d1[v0], s2 * W0.d2[v0]));
        }
    }
}

// The same for both features at once (F = 2), as unit_blend_t_f2.
template <int D>
__device__ __forceinline__ void unit_blend_t_hess_f2(uint64_t gg, const uint64_t (&gd)[3], const uint64_t (&gh)[6],
                                                     const AxisW2& W0, const AxisW2& W1, const AxisW2& W2,
                                                     uint64_t (&qb)[1 << D]) {
    if constexpr (D == 3) {
#pragma unroll
        for (int v2 = 0; v2 < 2; ++v2) {
            const uint64_t A = f2_fma(gg, W2.w[v2], f2_fma(gd[2], W2.d1[v2], f2_mul(gh[5], W2.d2[v2])));
            const uint64_t B = f2_fma(gd[0], W2.w[v2], f2_mul(gh[2], W2.d1[v2]));
            const uint64_t C = f2_fma(gd[1], W2.w[v2], f2_mul(gh[4], W2.d1[v2]));
            const uint64_t D00 = f2_mul(gh[0], W2.w[v2]);
            const uint64_t D11 = f2_mul(gh[3], W2.w[v2]);
            const uint64_t E01 = f2_mul(gh[1], W2.w[v2]);
#pragma unroll
            for (int v1 = 0; v1 < 2; ++v1) {
                const uint64_t s = f2_fma(A, W1.w[v1], f2_fma(C, W1.d1[v1], f2_mul(D11, W1.d2[v1])));
                const uint64_t s1 = f2_fma(B, W1.w[v1], f2_mul(E01, W1.d1[v1]));
                const uint64_t s2 = f2_mul(D00, W1.w[v1]);
#pragma unroll
                for (int v0 = 0; v0 < 2; ++v0)
                    qb[v0 + 2 * v1 + 4 * v2] = f2_fma(s, W0.w[v0], f2_fma(s1, W0.d1[v0], f2_mul(s2, W0.d2[v0])));
            }
        }
    } else {
#pragma unroll
        for (int v1 = 0; v1 < 2; ++v1) {
            const uint64_t s = f2_fma(gg, W1.w[v1], f2_fma(gd[1], W1.d1[v1], f2_mul(gh[2], W1.d2[v1])));
            const uint64_t s1 = f2_fma(gd[0], W1.w[v1], f2_mul(gh[1], W1.d1[v1]));
            const uint64_t s2 = f2_mul(gh[0], W1.w[v1]);
#pragma unroll
            for (int v0 = 0; v0 < 2; ++v0)
                qb[v0 + 2 * v1] = f2_fma(s, W0.w[v0], f2_fma(s1, W0.d1[v0], f2_mul(s2, W0.d2[v0])));
        }
    }
}

// Lane-split backward for packed fp32 gradient rows of 32 or 64 bytes: G
// lanes share one (point, level); lane g owns the 16-byte chunk g of every
// corner row (S = 2^D/G slots x FC features = 4 floats), computes the
// gradients of those slots, and issues one red.global.add.v4.f32 per corner,
// so one warp instruction reduces into whole rows.
// Four 256-thread blocks per SM (64 registers): the run-aggregation branch,
// rarely taken on random points, must not cost occupancy on the common path.
// The full-Hessian variant (twice the upstream values) spills a few words to
// local memory at this bound; on B300 that costs less than the occupancy it
// keeps (3D, 2^21 points: 4.08 ms at four blocks, 4.42 at three, 5.98 at two).
template <int D, int FC, int G, bool HESS>
__global__ void __launch_bounds__(kBlock, 4) hermite_bwd_split_kernel(const __grid_constant__ BwdParams p) {
    constexpr int V = 1 << D, S = V / G;
    static_assert(S * FC == 4, "one 16-byte chunk per lane");
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int64_t n = (static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x) / G;
    const int lane = threadIdx.x % G;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
    // the coordinates, re-read by every level's pass: evict-last with the full Hessian (see load_upstream)
    const uint64_t keep = HESS ? l2_evict_last_policy() : 0ull;
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(HESS ? ldg_hint(p.coords + n * D + i, keep) : __ldg(p.coords + n * D + i), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }
    float gg[FC], gl[FC], gd[FC][3], gh[FC][6];
#pragma unroll
    for (int f = 0; f < FC; ++f) load_upstream<D, HESS>(p, n, static_cast<int64_t>(l) * F + f, gg[f], gd[f], gl[f], gh[f]);
    float r[V][4];
#pragma unroll
    for (int u = 0; u < S; ++u) {
        const AxisW W0 = unit_axis<D, G>(B[0], lane, u, 0);
        const AxisW W1 = unit_axis<D, G>(B[1], lane, u, 1);
        const AxisW W2 = unit_axis<D, G>(B[D - 1], lane, u, D - 1);
        if constexpr (FC == 2) {
            const uint64_t gd2[3] = {f2_pack(gd[0][0], gd[1][0]), f2_pack(gd[0][1], gd[1][1]),
                                     f2_pack(gd[0][2], gd[1][2])};
            uint64_t qb[V];
            if constexpr (HESS) {
                uint64_t gh2[6];
#pragma unroll
                for (int k = 0; k < 6; ++k) gh2[k] = f2_pack(gh[0][k], gh[1][k]);
                unit_blend_t_hess_f2<D>(f2_pack(gg[0], gg[1]), gd2, gh2, axis_dup(W0), axis_dup(W1), axis_dup(W2),
                                        qb);
            } else {
                unit_blend_t_f2<D>(f2_pack(gg[0], gg[1]), gd2, f2_pack(gl[0], gl[1]), axis_dup(W0), axis_dup(W1),
                                   axis_dup(W2), qb);
            }
#pragma unroll
            for (int v = 0; v < V; ++v) f2_unpack(qb[v], r[v][u * FC], r[v][u * FC + 1]);
        } else {
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                float qb[V];
                if constexpr (HESS) {
                    unit_blend_t_hess<D>(gg[f], gd[f], gh[f], W0, W1, W2, qb);
                } else {
                    unit_blend_t<D>(gg[f], gd[f], gl[f], W0, W1, W2, qb);
                }
#pragma unroll
                for (int v = 0; v < V; ++v) r[v][u * FC + f] = qb[v];
            }
        }
    }
    // consecutive points in one cell (coherent inputs) add up before the RED
    const unsigned active =
        item_lanes<G>((static_cast<int64_t>(blockIdx.x) * kBlock + (threadIdx.x & ~31u)) / G, p.c.n);
    if (!run_aggregate<D, G, V * 4>(active, c, reinterpret_cast<float(&)[V * 4]>(r))) return;
    float* row0 = p.grad.ptr[0] + l * p.grad.ls[0] + lane * 4;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        uint32_t g[D];
#pragma unroll
        for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
        const uint32_t id = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
        red_add_v4(row0 + static_cast<int64_t>(id) * p.grad.rs[0], r[v][0], r[v][1], r[v][2], r[v][3]);
    }
}

constexpr int kPrivBlock = 512;

// Privatised backward for small one-to-one levels.  A CTA owns (level, a
// chunk of points, 16-byte row part g): it accumulates its points' gradients
// for part g of every row of the level in shared memory (shared atomics,
// contention resolved on chip), then adds the part into the gradient table
// with one red.global.add.v4.f32 per row that received anything.  Without it
// the coarsest levels -- a few hundred to a few thousand rows hit by millions
// of points -- serialise on the same L2 addresses.  Each contribution is the
// split kernel's (part g plays lane g).
template <int D, int FC, int G, bool HESS>
__global__ void __launch_bounds__(kPrivBlock) hermite_bwd_priv_kernel(const __grid_constant__ BwdParams p) {
    constexpr int V = 1 << D, S = V / G;
    static_assert(S * FC == 4, "one 16-byte part per row");
    extern __shared__ float4 sacc[];
    const int l = p.priv.lvl[blockIdx.y];
    const uint32_t rows = p.priv.rows[blockIdx.y];
    const int part = blockIdx.z;
    for (uint32_t i = threadIdx.x; i < rows; i += kPrivBlock) sacc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    float* sf = reinterpret_cast<float*>(sacc);
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * p.priv.chunk;
    const int64_t n1 = min(n0 + p.priv.chunk, p.c.n);
    for (int64_t n = n0 + threadIdx.x; n < n1; n += kPrivBlock) {
        uint32_t c[D];
        float t[D];
        Basis1 B[D];
#pragma unroll
        for (int i = 0; i < D; ++i) {
            locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
            B[i] = hermite_basis(t[i], lv);
        }
        float gg[FC], gl[FC], gd[FC][3], gh[FC][6];
#pragma unroll
        for (int f = 0; f < FC; ++f)
            load_upstream<D, HESS>(p, n, static_cast<int64_t>(l) * F + f, gg[f], gd[f], gl[f], gh[f]);
        float r[V][4];
#pragma unroll
        for (int u = 0; u < S; ++u) {
            const AxisW W0 = unit_axis<D, G>(B[0], part, u, 0);
            const AxisW W1 = unit_axis<D, G>(B[1], part, u, 1);
            const AxisW W2 = unit_axis<D, G>(B[D - 1], part, u, D - 1);
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                float qb[V];
                if constexpr (HESS) {
                    unit_blend_t_hess<D>(gg[f], gd[f], gh[f], W0, W1, W2, qb);
                } else {
                    unit_blend_t<D>(gg[f], gd[f], gl[f], W0, W1, W2, qb);
                }
#pragma unroll
                for (int v = 0; v < V; ++v) r[v][u * FC + f] = qb[v];
            }
        }
        const unsigned active = item_lanes<1>(n - (threadIdx.x & 31), n1);
        if (run_aggregate<D, 1, V * 4>(active, c, reinterpret_cast<float(&)[V * 4]>(r))) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                uint32_t g[D];
#pragma unroll
                for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
                float* a = sf + 4 * vertex_index<D>(g, lv, true, 0u);
#pragma unroll
                for (int j = 0; j < 4; ++j) atomicAdd(a + j, r[v][j]);
            }
        }
    }
    __syncthreads();
    float* row0 = p.grad.ptr[0] + l * p.grad.ls[0] + part * 4;
    for (uint32_t i = threadIdx.x; i < rows; i += kPrivBlock) {
        const float4 a = sacc[i];
        if (a.x != 0.f || a.y != 0.f || a.z != 0.f || a.w != 0.f)
            red_add_v4(row0 + static_cast<int64_t>(i) * p.grad.rs[0], a.x, a.y, a.z, a.w);
    }
}

// 4D (space-time) backward, any layout and F: the transpose of
// hermite_fwd4_kernel.  Per axis-3 slice (v3, a3) the upstream gradients
// are folded with the axis-3 weights into the upstream of a 3D slice blend,
//   gamma:  g_gamma w + g_dgamma_3 w' + (g_lap | g_hess_33) w''
//   d/dx_j: g_dgamma_j w [+ g_hess_j3 w']                (j < 3)
//   second: g_lap w  |  g_hess_ij w                       (i, j < 3)
// and the 3D transposed blend gives that slice's 64 coefficient gradients,
// added one element at a time.
template <bool HESS>
__global__ void __launch_bounds__(kBlock) hermite_bwd4_kernel(const __grid_constant__ BwdParams p) {
    constexpr int D = 4;
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }
    for (int f = 0; f < F; ++f) {
        const int64_t lf = static_cast<int64_t>(l) * F + f;
        const float gg = p.g_gamma ? __ldg(p.g_gamma + n * p.c.sn + lf * p.c.sf) : 0.f;
        float gd[4];
#pragma unroll
        for (int j = 0; j < D; ++j) gd[j] = p.g_dgamma ? __ldg(p.g_dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf) : 0.f;
        float gl = 0.f, gh[10];
#pragma unroll
        for (int k = 0; k < 10; ++k) gh[k] = 0.f;
        if constexpr (HESS) {
            if (p.g_hess) {
#pragma unroll
                for (int k = 0; k < 10; ++k) gh[k] = __ldg(p.g_hess + n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf);
            }
        } else {
            gl = p.g_lap ? __ldg(p.g_lap + n * p.c.sn + lf * p.c.sf) : 0.f;
        }
#pragma unroll 1
        for (int v3 = 0; v3 < 2; ++v3) {
#pragma unroll
            for (int a3 = 0; a3 < 2; ++a3) {
                const float w = B[3].w[v3][a3], w1 = B[3].d1[v3][a3], w2 = B[3].d2[v3][a3];
                float qb[8][8];
                if constexpr (HESS) {
                    // 4D Hessian entries: xx xy xz xw yy yz yw zz zw ww
                    const float sg = fmaf(gg, w, fmaf(gd[3], w1, gh[9] * w2));
                    const float sd[3] = {fmaf(gd[0], w, gh[3] * w1), fmaf(gd[1], w, gh[6] * w1),
                                         fmaf(gd[2], w, gh[8] * w1)};
                    const float sh[6] = {gh[0] * w, gh[1] * w, gh[2] * w, gh[4] * w, gh[5] * w, gh[7] * w};
                    blend3h_t(sg, sd, sh, B[0], B[1], B[2], qb);
                } else {
                    const float sg = fmaf(gg, w, fmaf(gd[3], w1, gl * w2));
                    const float sd[3] = {gd[0] * w, gd[1] * w, gd[2] * w};
                    blend3_t(sg, sd, gl * w, B[0], B[1], B[2], qb);
                }
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint32_t gv[D] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u),
                                            c[3] + static_cast<uint32_t>(v3)};
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        const int alpha = a + 8 * a3, k = alpha_order(alpha);
                        const uint32_t id = vertex_index<D>(gv, lv, (lv.dense >> k) & 1u, p.c.tmask[k]);
                        float* e = p.grad.ptr[k] + l * p.grad.ls[k] + static_cast<int64_t>(id) * p.grad.rs[k] +
                                   bucket_slot<D>(alpha) * F + f;
                        red_add_f32(e, qb[v][a]);
                    }
                }
            }
        }
    }
}

// Lane-octet backward for packed 4D F = 2 fp32 gradient rows (128 bytes):
// lane g of an octet owns the 16-byte chunk g of every corner row (slots 2g
// and 2g+1, both features) and issues one red.global.add.v4.f32 per corner,
// so one warp RED covers four whole rows.  Per axis-3 half (v3) and slot the
// upstream gradients are folded with the slot's axis-3 weight into the
// upstream of a 3D slice, whose transposed unit blend (f32x2) gives the 8
// corners' contributions -- the transpose of hermite_fwd_quad4_kernel.
// Consecutive points of one cell add up in the warp first.
// Two blocks per SM (128 registers, no spills): measured on the 4D workload
// (2^20 points) 6.67 ms, against 7.87 ms at three blocks and 10.39 ms at
// four (80 / 64 registers with 140 / 276 bytes of spills).
template <bool HESS>
__global__ void __launch_bounds__(kBlock, 2) hermite_bwd_oct4_kernel(const __grid_constant__ BwdParams p) {
    constexpr int D = 4, G = 8, S = 2;
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int64_t n = (static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x) / G;
    const int lane = threadIdx.x % G;
    if (n >= p.c.n) return;
    const Level& lv = p.c.lv[l];

    uint32_t c[D];
    float t[D];
    Basis1 B[D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
        B[i] = hermite_basis(t[i], lv);
    }
    // upstream gradients of both features as (f0, f1) pairs
    auto up = [&](const float* a, int64_t at, int64_t fstride) {
        return a ? f2_pack(__ldg(a + at), __ldg(a + at + fstride)) : 0ull;
    };
    const int64_t lf = static_cast<int64_t>(l) * 2;
    const uint64_t gg = up(p.g_gamma, n * p.c.sn + lf * p.c.sf, p.c.sf);
    uint64_t gd[4];
#pragma unroll
    for (int j = 0; j < D; ++j) gd[j] = up(p.g_dgamma, n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, p.c.dsf);
    uint64_t gs[HESS ? 10 : 1];  // the Laplacian's, or the 4D Hessian's xx xy xz xw yy yz yw zz zw ww
    if constexpr (HESS) {
#pragma unroll
        for (int k = 0; k < 10; ++k) gs[k] = up(p.g_hess, n * p.c.hsn + k * p.c.hsq + lf * p.c.hsf, p.c.hsf);
    } else {
        gs[0] = up(p.g_lap, n * p.c.sn + lf * p.c.sf, p.c.sf);
    }
    const unsigned active =
        item_lanes<G>((static_cast<int64_t>(blockIdx.x) * kBlock + (threadIdx.x & ~31u)) / G, p.c.n);
    float* row0 = p.grad.ptr[0] + l * p.grad.ls[0] + lane * 4;
#pragma unroll
    for (int v3 = 0; v3 < 2; ++v3) {
        float r[8][4];
#pragma unroll
        for (int u = 0; u < S; ++u) {
            const AxisW2 W0 = axis_dup(unit_axis<D, G>(B[0], lane, u, 0));
            const AxisW2 W1 = axis_dup(unit_axis<D, G>(B[1], lane, u, 1));
            const AxisW2 W2 = axis_dup(unit_axis<D, G>(B[2], lane, u, 2));
            const AxisW W3 = unit_axis<D, G>(B[3], lane, u, 3);
            const uint64_t w = f2_dup(W3.w[v3]), w1 = f2_dup(W3.d1[v3]), w2 = f2_dup(W3.d2[v3]);
            uint64_t qb[8];
            if constexpr (HESS) {
                const uint64_t sg = f2_fma(gg, w, f2_fma(gd[3], w1, f2_mul(gs[9], w2)));
                const uint64_t sd[3] = {f2_fma(gd[0], w, f2_mul(gs[3], w1)), f2_fma(gd[1], w, f2_mul(gs[6], w1)),
                                        f2_fma(gd[2], w, f2_mul(gs[8], w1))};
                const uint64_t sh[6] = {f2_mul(gs[0], w), f2_mul(gs[1], w), f2_mul(gs[2], w),
                                        f2_mul(gs[4], w), f2_mul(gs[5], w), f2_mul(gs[7], w)};
                unit_blend_t_hess_f2<3>(sg, sd, sh, W0, W1, W2, qb);
            } else {
                const uint64_t sg = f2_fma(gg, w, f2_fma(gd[3], w1, f2_mul(gs[0], w2)));
                const uint64_t sd[3] = {f2_mul(gd[0], w), f2_mul(gd[1], w), f2_mul(gd[2], w)};
                unit_blend_t_f2<3>(sg, sd, f2_mul(gs[0], w), W0, W1, W2, qb);
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) f2_unpack(qb[v], r[v][u * 2], r[v][u * 2 + 1]);
        }
        if (run_aggregate<D, G, 32>(active, c, reinterpret_cast<float(&)[32]>(r))) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const uint32_t g[D] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u),
                                       c[3] + static_cast<uint32_t>(v3)};
                const uint32_t id = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
                red_add_v4(row0 + static_cast<int64_t>(id) * p.grad.rs[0], r[v][0], r[v][1], r[v][2], r[v][3]);
            }
        }
    }
}

template <int D, int FC, int G, bool HESS>
cudaError_t launch_priv(const BwdParams& p, cudaStream_t s) {
    if (p.priv.n == 0) return cudaSuccess;
    if (p.priv.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(hermite_bwd_priv_kernel<D, FC, G, HESS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, p.priv.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(static_cast<unsigned>((p.c.n + p.priv.chunk - 1) / p.priv.chunk), static_cast<unsigned>(p.priv.n), G);
    hermite_bwd_priv_kernel<D, FC, G, HESS><<<grid, kPrivBlock, p.priv.smem_bytes, s>>>(p);
    return cudaGetLastError();
}

template <int D, int FC, int G, bool HESS>
cudaError_t launch_split(const BwdParams& p, cudaStream_t s) {
    cudaError_t e = launch_priv<D, FC, G, HESS>(p, s);
    if (e != cudaSuccess || p.c.nlvl == 0) return e;
    dim3 grid(static_cast<unsigned>((p.c.n * G + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    hermite_bwd_split_kernel<D, FC, G, HESS><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, int FC, bool VEC, bool HESS>
cudaError_t launch(const BwdParams& p, cudaStream_t s) {
    if (VEC && D == 2 && FC == 1) {  // 16-byte rows: one part per row
        cudaError_t e = launch_priv<2, 1, 1, HESS>(p, s);
        if (e != cudaSuccess) return e;
    }
    if (p.c.nlvl == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    hermite_bwd_kernel<D, FC, VEC, HESS><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, bool HESS>
cudaError_t pick(const BwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (fc == 2) return vec ? launch<D, 2, true, HESS>(p, s) : launch<D, 2, false, HESS>(p, s);
    return vec ? launch<D, 1, true, HESS>(p, s) : launch<D, 1, false, HESS>(p, s);
}

template <bool HESS>
cudaError_t dispatch(const BwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (p.c.d == 4) {
        if (p.c.nlvl == 0) return cudaSuccess;
        if (vec && fc == p.c.F && p.c.F == 2) {  // packed 128-byte rows: lane octets
            dim3 grid(static_cast<unsigned>((p.c.n * 8 + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
            hermite_bwd_oct4_kernel<HESS><<<grid, kBlock, 0, s>>>(p);
            return cudaGetLastError();
        }
        dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
        hermite_bwd4_kernel<HESS><<<grid, kBlock, 0, s>>>(p);
        return cudaGetLastError();
    }
    if (vec && fc == p.c.F) {
        // packed rows of 2^d * F floats: 32 bytes -> lane pairs, 64 bytes -> quads
        if (p.c.d == 2 && p.c.F == 2) return launch_split<2, 2, 2, HESS>(p, s);
        if (p.c.d == 3 && p.c.F == 1) return launch_split<3, 1, 2, HESS>(p, s);
        if (p.c.d == 3 && p.c.F == 2) return launch_split<3, 2, 4, HESS>(p, s);
    }
    return p.c.d == 2 ? pick<2, HESS>(p, fc, vec, s) : pick<3, HESS>(p, fc, vec, s);
}

}  // namespace

int launch_hermite_bwd(const BwdParams& p, int fc, bool vec, bool hess, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return hess ? dispatch<true>(p, fc, vec, s) : dispatch<false>(p, fc, vec, s);
}

}  // namespace hg
