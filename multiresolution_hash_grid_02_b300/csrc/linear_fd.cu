// INGP-FD: the d-linear encoding with central finite differences, forward
// and backward.
//
// "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
// 研究背景与动机 and 关键设计 2: the finite-difference baseline (INGP-FD)
// takes the Laplacian from 2d+1 d-linear encodes, at x and x +- eps e_i,
//   d gamma / dx_i ~ (gamma(x + eps e_i) - gamma(x - eps e_i)) / (2 eps),
//   lap gamma      ~ sum_i (gamma(x + eps e_i) - 2 gamma(x) + gamma(x - eps e_i)) / eps^2,
// with each shifted coordinate one fp32 add, located like any coordinate.
//
// Mapping: one thread per (point, level), grid.y = level, as the d-linear
// kernels.  The 2d+1 encodes share work: the centre cell's 2^d rows are read
// once, and a stencil point that stays in that cell (its shifted coordinate
// keeps the cell index) only re-weights them; a stencil point that crosses a
// cell face reads its own cell's rows.  The backward likewise sums the
// contributions of same-cell stencil points into the centre rows before the
// scatter, so those cost no extra REDs; small one-to-one levels accumulate in
// shared memory first (privatised, as the d-linear backward).
#include <cuda_runtime.h>

#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;
constexpr int kPrivBlock = 512;

// Cell and local coordinate of the shifted coordinate x +- eps (s = 0: +, 1: -).
__device__ __forceinline__ void locate_shifted(float x, float eps, int s, const Level& lv, uint32_t& c, float& t) {
    locate(s ? __fsub_rn(x, eps) : __fadd_rn(x, eps), lv, c, t);
}

// Corner v (bit k = side along axis k) of the face position u along axis i:
// u's bits are the other axes' sides, b the side along axis i.
__device__ __forceinline__ constexpr int face_corner(int u, int i, int b) {
    return ((u >> i) << (i + 1)) | (b << i) | (u & ((1 << i) - 1));
}

// d-linear weights of the 2^(D-1) face positions along axis i (the product
// of the other axes' weights).
template <int D>
__device__ __forceinline__ void face_weights(const float (&t)[D], int i, float (&wo)[1 << (D - 1)]) {
#pragma unroll
    for (int u = 0; u < (1 << (D - 1)); ++u) {
        const int v = face_corner(u, i, 0);
        float w = 1.f;
#pragma unroll
        for (int k = 0; k < D; ++k)
            if (k != i) w *= ((v >> k) & 1) ? t[k] : 1.f - t[k];
        wo[u] = w;
    }
}

// FC features of a table row (8-/4-byte pair loads on the VEC path).
template <int FC, typename TT, bool VEC>
__device__ __forceinline__ void load_feats(const TT* e, float (&val)[FC]) {
    if constexpr (VEC && sizeof(TT) == 4) {
        const float2 q = __ldg(reinterpret_cast<const float2*>(e));
        val[0] = q.x;
        val[FC - 1] = q.y;
    } else if constexpr (VEC) {
        const float2 q = __half22float2(__ldg(reinterpret_cast<const __half2*>(e)));
        val[0] = q.x;
        val[FC - 1] = q.y;
    } else {
#pragma unroll
        for (int f = 0; f < FC; ++f) val[f] = to_f32<TT>(e[f]);
    }
}

template <int D, int FC, typename TT, bool VEC>
__global__ void __launch_bounds__(kBlock) linear_fd_fwd_kernel(const __grid_constant__ FwdParams p) {
    constexpr int V = 1 << D;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const bool active = (p.c.level_mask >> l) & 1u;

    float x[D], t[D], ts[2 * D];
    uint32_t c[D], cs[2 * D];
#pragma unroll
    for (int i = 0; i < D; ++i) {
        x[i] = __ldg(p.coords + n * D + i);
        locate(x[i], lv, c[i], t[i]);
#pragma unroll
        for (int s = 0; s < 2; ++s) locate_shifted(x[i], p.eps, s, lv, cs[2 * i + s], ts[2 * i + s]);
    }
    uint32_t idx[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        uint32_t g[D];
#pragma unroll
        for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
        idx[v] = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
    }
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
    for (int f0 = 0; f0 < F; f0 += FC) {
        float cv[V][FC], g0[FC];
#pragma unroll
        for (int f = 0; f < FC; ++f) g0[f] = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int f = 0; f < FC; ++f) cv[v][f] = 0.f;
        if (active) {
#pragma unroll
            for (int v = 0; v < V; ++v) load_feats<FC, TT, VEC>(base + static_cast<int64_t>(idx[v]) * p.tab.rs[0] + f0, cv[v]);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float w = corner_weight<D>(t, v);
#pragma unroll
                for (int f = 0; f < FC; ++f) g0[f] = fmaf(w, cv[v][f], g0[f]);
            }
        }
        float dg[D][FC], lp[FC];
#pragma unroll
        for (int f = 0; f < FC; ++f) lp[f] = 0.f;
#pragma unroll
        for (int i = 0; i < D; ++i) {
            constexpr int H = V / 2;
            float wo[H];
            face_weights<D>(t, i, wo);
            float gs[2][FC];
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int j = 2 * i + s;
                // the shifted cell along axis i: dc = 0 (same cell), +-1 (a neighbour that shares a
                // face with the centre cell) or further; its low / high faces come from the centre's
                // rows where they coincide and are read otherwise
                const int dc = static_cast<int>(cs[j]) - static_cast<int>(c[i]);
                const bool own_lo = dc == 0 || dc == 1, own_hi = dc == 0 || dc == -1;
                float lo[H][FC], hi[H][FC];
#pragma unroll
                for (int u = 0; u < H; ++u)
#pragma unroll
                    for (int f = 0; f < FC; ++f) {
                        lo[u][f] = dc == 0 ? cv[face_corner(u, i, 0)][f] : cv[face_corner(u, i, 1)][f];
                        hi[u][f] = dc == 0 ? cv[face_corner(u, i, 1)][f] : cv[face_corner(u, i, 0)][f];
                    }
                if (active && !own_lo) {
#pragma unroll
                    for (int u = 0; u < H; ++u) {
                        uint32_t g[D];
#pragma unroll
                        for (int k = 0; k < D; ++k) g[k] = k == i ? cs[j] : c[k] + ((face_corner(u, i, 0) >> k) & 1u);
                        load_feats<FC, TT, VEC>(
                            base + static_cast<int64_t>(vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0])) *
                                       p.tab.rs[0] + f0,
                            lo[u]);
                    }
                }
                if (active && !own_hi) {
#pragma unroll
                    for (int u = 0; u < H; ++u) {
                        uint32_t g[D];
#pragma unroll
                        for (int k = 0; k < D; ++k)
                            g[k] = k == i ? cs[j] + 1u : c[k] + ((face_corner(u, i, 0) >> k) & 1u);
                        load_feats<FC, TT, VEC>(
                            base + static_cast<int64_t>(vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0])) *
                                       p.tab.rs[0] + f0,
                            hi[u]);
                    }
                }
#pragma unroll
                for (int f = 0; f < FC; ++f) {
                    float acc = 0.f;
#pragma unroll
                    for (int u = 0; u < H; ++u) acc = fmaf(wo[u], fmaf(ts[j], hi[u][f] - lo[u][f], lo[u][f]), acc);
                    gs[s][f] = active ? acc : 0.f;
                }
                if (p.stencil) {
#pragma unroll
                    for (int f = 0; f < FC; ++f) {
                        const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
                        __stcs(p.stencil + n * p.c.ssn + j * p.c.ssj + lf * p.c.ssf, gs[s][f]);
                    }
                }
            }
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                dg[i][f] = (gs[0][f] - gs[1][f]) * p.half_inv_eps;
                lp[f] = fmaf((gs[0][f] - g0[f]) + (gs[1][f] - g0[f]), p.inv_eps2, lp[f]);
            }
        }
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
            __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, g0[f]);
            if (p.dgamma) {
#pragma unroll
                for (int i = 0; i < D; ++i) __stcs(p.dgamma + n * p.c.dsn + i * p.c.dsj + lf * p.c.dsf, dg[i][f]);
            }
            if (p.lap) __stcs(p.lap + n * p.c.sn + lf * p.c.sf, lp[f]);
        }
    }
}

// The backward of one (point, level, feature chunk): the upstream weight of
// each stencil value in the outputs, the centre cell's corner contributions
// (with those of same-cell stencil points folded in) and the crossing stencil
// points' own corners, handed to add(vertex, values).
template <int D, int FC, typename Add>
__device__ __forceinline__ void fd_point_bwd(const BwdParams& p, int64_t n, int l, int f0, const float (&t)[D],
                                             const uint32_t (&c)[D], const float (&ts)[2 * D],
                                             const uint32_t (&cs)[2 * D], Add&& add) {
    constexpr int V = 1 << D;
    const int F = p.c.F;
    float gg[FC], gl[FC];
#pragma unroll
    for (int f = 0; f < FC; ++f) {
        const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
        gg[f] = p.g_gamma ? __ldg(p.g_gamma + n * p.c.sn + lf * p.c.sf) : 0.f;
        gl[f] = p.g_lap ? __ldg(p.g_lap + n * p.c.sn + lf * p.c.sf) : 0.f;
    }
    float acc[V][FC];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const float w = corner_weight<D>(t, v);
#pragma unroll
        for (int f = 0; f < FC; ++f) acc[v][f] = w * fmaf(-2.0f * D * p.inv_eps2, gl[f], gg[f]);
    }
#pragma unroll
    for (int i = 0; i < D; ++i) {
        constexpr int H = V / 2;
        float wo[H];
        face_weights<D>(t, i, wo);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int j = 2 * i + s;
            float u[FC];
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
                const float gd = p.g_dgamma ? __ldg(p.g_dgamma + n * p.c.dsn + i * p.c.dsj + lf * p.c.dsf) : 0.f;
                const float gs = p.g_stencil ? __ldg(p.g_stencil + n * p.c.ssn + j * p.c.ssj + lf * p.c.ssf) : 0.f;
                u[f] = fmaf(s ? -gd : gd, p.half_inv_eps, fmaf(gl[f], p.inv_eps2, gs));
            }
            // faces of the shifted cell that coincide with the centre cell's fold into its rows; the
            // others are scattered on their own
            const int dc = static_cast<int>(cs[j]) - static_cast<int>(c[i]);
            const bool own_lo = dc == 0 || dc == 1, own_hi = dc == 0 || dc == -1;
#pragma unroll
            for (int q = 0; q < H; ++q) {
                float vlo[FC], vhi[FC];
#pragma unroll
                for (int f = 0; f < FC; ++f) {
                    // (1 - t) is exact at t = 1, so a corner of weight zero receives exactly zero
                    vhi[f] = wo[q] * ts[j] * u[f];
                    vlo[f] = wo[q] * (1.f - ts[j]) * u[f];
                    const int c0 = face_corner(q, i, 0), c1 = face_corner(q, i, 1);
                    acc[c0][f] += (dc == 0 ? vlo[f] : 0.f) + (dc == -1 ? vhi[f] : 0.f);
                    acc[c1][f] += (dc == 0 ? vhi[f] : 0.f) + (dc == 1 ? vlo[f] : 0.f);
                }
                if (!own_lo) {
                    uint32_t g[D];
#pragma unroll
                    for (int k = 0; k < D; ++k) g[k] = k == i ? cs[j] : c[k] + ((face_corner(q, i, 0) >> k) & 1u);
                    add(g, vlo);
                }
                if (!own_hi) {
                    uint32_t g[D];
#pragma unroll
                    for (int k = 0; k < D; ++k) g[k] = k == i ? cs[j] + 1u : c[k] + ((face_corner(q, i, 0) >> k) & 1u);
                    add(g, vhi);
                }
            }
        }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
        uint32_t g[D];
#pragma unroll
        for (int k = 0; k < D; ++k) g[k] = c[k] + ((v >> k) & 1u);
        add(g, acc[v]);
    }
}

template <int D>
__device__ __forceinline__ void locate_stencil(const BwdParams& p, int64_t n, const Level& lv, float (&t)[D],
                                               uint32_t (&c)[D], float (&ts)[2 * D], uint32_t (&cs)[2 * D]) {
#pragma unroll
    for (int i = 0; i < D; ++i) {
        const float x = __ldg(p.coords + n * D + i);
        locate(x, lv, c[i], t[i]);
#pragma unroll
        for (int s = 0; s < 2; ++s) locate_shifted(x, p.eps, s, lv, cs[2 * i + s], ts[2 * i + s]);
    }
}

// Two blocks per SM (128 registers): 4.78 ms on the 3D INGP-FD workload
// (2^21 points) against 5.10 ms unbounded (252 registers) and 4.98 ms at three.
template <int D, int FC, bool VEC>
__global__ void __launch_bounds__(kBlock, 2) linear_fd_bwd_kernel(const __grid_constant__ BwdParams p) {
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const Level& lv = p.c.lv[l];
    float t[D], ts[2 * D];
    uint32_t c[D], cs[2 * D];
    locate_stencil<D>(p, n, lv, t, c, ts, cs);
    float* base = p.grad.ptr[0] + l * p.grad.ls[0];
    for (int f0 = 0; f0 < p.c.F; f0 += FC) {
        fd_point_bwd<D, FC>(p, n, l, f0, t, c, ts, cs, [&](const uint32_t (&g)[D], const float (&val)[FC]) {
            float* e = base + static_cast<int64_t>(vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0])) * p.grad.rs[0] + f0;
            if constexpr (VEC) {
                red_add_v2(e, val[0], val[FC - 1]);
            } else {
#pragma unroll
                for (int f = 0; f < FC; ++f) red_add_f32(e + f, val[f]);
            }
        });
    }
}

// Privatised backward for small one-to-one levels: a CTA accumulates a chunk
// of points into a shared-memory copy of the level's gradient rows (every
// stencil point of a one-to-one level stays inside the level's grid), then
// adds each row that received anything into the table.
template <int D, int FC>
__global__ void __launch_bounds__(kPrivBlock) linear_fd_bwd_priv_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ float sacc[];
    const int l = p.priv.lvl[blockIdx.y];
    const uint32_t rows = p.priv.rows[blockIdx.y];
    const int F = p.c.F;
    const uint32_t vals = rows * static_cast<uint32_t>(F);
    for (uint32_t i = threadIdx.x; i < vals; i += kPrivBlock) sacc[i] = 0.f;
    __syncthreads();
    const Level& lv = p.c.lv[l];
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * p.priv.chunk;
    const int64_t n1 = min(n0 + p.priv.chunk, p.c.n);
    for (int64_t n = n0 + threadIdx.x; n < n1; n += kPrivBlock) {
        float t[D], ts[2 * D];
        uint32_t c[D], cs[2 * D];
        locate_stencil<D>(p, n, lv, t, c, ts, cs);
        for (int f0 = 0; f0 < F; f0 += FC) {
            fd_point_bwd<D, FC>(p, n, l, f0, t, c, ts, cs, [&](const uint32_t (&g)[D], const float (&val)[FC]) {
                float* a = sacc + vertex_index<D>(g, lv, true, 0u) * F + f0;
#pragma unroll
                for (int f = 0; f < FC; ++f) atomicAdd(a + f, val[f]);
            });
        }
    }
    __syncthreads();
    float* base = p.grad.ptr[0] + l * p.grad.ls[0];
    for (uint32_t i = threadIdx.x; i < vals; i += kPrivBlock) {
        const float a = sacc[i];
        if (a != 0.f) red_add_f32(base + static_cast<int64_t>(i / F) * p.grad.rs[0] + i % F, a);
    }
}

template <int D, int FC, typename TT, bool VEC>
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    linear_fd_fwd_kernel<D, FC, TT, VEC><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, typename TT>
cudaError_t pick_fwd(const FwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (fc == 2) return vec ? launch_fwd<D, 2, TT, true>(p, s) : launch_fwd<D, 2, TT, false>(p, s);
    return launch_fwd<D, 1, TT, false>(p, s);
}

template <int D, int FC, bool VEC>
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t s) {
    if (p.priv.n > 0) {
        if (p.priv.smem_bytes > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(linear_fd_bwd_priv_kernel<D, FC>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, p.priv.smem_bytes);
            if (e != cudaSuccess) return e;
        }
        dim3 grid(static_cast<unsigned>((p.c.n + p.priv.chunk - 1) / p.priv.chunk), static_cast<unsigned>(p.priv.n));
        linear_fd_bwd_priv_kernel<D, FC><<<grid, kPrivBlock, p.priv.smem_bytes, s>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || p.c.nlvl == 0) return e;
    }
    if (p.c.nlvl == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    linear_fd_bwd_kernel<D, FC, VEC><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t pick_bwd(const BwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (fc == 2) return vec ? launch_bwd<D, 2, true>(p, s) : launch_bwd<D, 2, false>(p, s);
    return launch_bwd<D, 1, false>(p, s);
}

}  // namespace

int launch_linear_fd_fwd(const FwdParams& p, int fc, bool vec, int dtype, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.c.d == 2) return dtype == HG_F16 ? pick_fwd<2, __half>(p, fc, vec, s) : pick_fwd<2, float>(p, fc, vec, s);
    if (p.c.d == 4) return dtype == HG_F16 ? pick_fwd<4, __half>(p, fc, vec, s) : pick_fwd<4, float>(p, fc, vec, s);
    return dtype == HG_F16 ? pick_fwd<3, __half>(p, fc, vec, s) : pick_fwd<3, float>(p, fc, vec, s);
}

int launch_linear_fd_bwd(const BwdParams& p, int fc, bool vec, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.c.d == 4) return pick_bwd<4>(p, fc, vec, s);
    return p.c.d == 2 ? pick_bwd<2>(p, fc, vec, s) : pick_bwd<3>(p, fc, vec, s);
}

}  // namespace hg
