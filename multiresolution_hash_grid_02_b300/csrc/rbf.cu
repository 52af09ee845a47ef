// Gaussian-RBF multi-resolution grid (DInf-Grid), forward and backward.
//
// "DInf-Grid：一种基于可微特征网格的神经微分方程求解器", 可微的径向基函数插值 and
// 多分辨率特征网格: per level, f(x) = sum_{i in N(x)} w(x, x_i) F_i with the
// normalised Gaussian weight w = phi(|x - x_i|) / sum_j phi(|x - x_j|),
// phi(r) = exp(-(eps r)^2), over a ring neighbourhood of the point's cell
// (distances in the level's grid units; ring R = the box c_i - R + 1 ..
// c_i + R clipped to the grid).  The page computes this with autodiff in
// PyTorch and suggests a custom CUDA kernel for the weights and the
// neighbour aggregation.
//
// Design: exp(-eps^2 |y - g|^2) = prod_i exp(-eps^2 (y_i - g_i)^2) and the
// neighbourhood is a box, so the normalised weight is a product of 1D
// normalised weights, w_g = prod_i omega_i(g_i).  Each axis needs 2R
// exponentials (not (2R)^d), and gamma, its gradient and its Laplacian
// are separable contractions -- axis 0 innermost, with value, d/dx_0 and
// d2/dx_0^2 partial sums, as the Hermite blend -- of the 1D weights and
// their 1D quotient-rule derivatives (d/dx = N d/dy folded in).  One thread
// per (point, level); taps outside the grid get weight 0 and are not read.
// The backward is the transposed contraction, accumulated per CTA in a
// shared-memory tile of its points' neighbourhoods (the page samples
// stratified points, so a CTA's points are neighbours) before the scatter.
#include <cuda_runtime.h>

#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;

// The 2R taps of one axis: vertex g = first + k, its normalised 1D weight
// and that weight's first and second x-derivatives; `valid` bit k = inside.
template <int K>
struct RbfAxis {
    int32_t first;
    uint32_t valid;
    float w[K], d1[K], d2[K];
};

template <int K>
__device__ __forceinline__ RbfAxis<K> rbf_axis(uint32_t c, float t, const Level& lv, float eps2) {
    RbfAxis<K> a;
    a.first = static_cast<int32_t>(c) - K / 2 + 1;
    a.valid = 0u;
    float e[K], e1[K], e2[K], s = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int32_t g = a.first + k;
        const bool in = g >= 0 && g <= static_cast<int32_t>(lv.N);
        a.valid |= static_cast<uint32_t>(in) << k;
        const float r = t - static_cast<float>(k - K / 2 + 1);        // y - g, in grid units
        const float ek = in ? expf(-eps2 * r * r) : 0.f;
        e[k] = ek;
        e1[k] = -2.f * eps2 * r * ek;
        e2[k] = fmaf(4.f * eps2 * eps2, r * r, -2.f * eps2) * ek;
        s += e[k];
        s1 += e1[k];
        s2 += e2[k];
    }
    const float inv = 1.f / s;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float w = e[k] * inv;
        const float w1 = (e1[k] - w * s1) * inv;
        const float w2 = (e2[k] - 2.f * w1 * s1 - w * s2) * inv;
        a.w[k] = w;
        a.d1[k] = w1 * lv.fN;
        a.d2[k] = w2 * lv.fN2;
    }
    return a;
}

template <int D, int K>
__device__ __forceinline__ void rbf_axes(const float* coords, int64_t n, const Level& lv, float eps2,
                                         RbfAxis<K> (&A)[D]) {
#pragma unroll
    for (int i = 0; i < D; ++i) {
        uint32_t c;
        float t;
        locate(__ldg(coords + n * D + i), lv, c, t);
        A[i] = rbf_axis<K>(c, t, lv, eps2);
    }
}

template <int FC, typename TT>
__device__ __forceinline__ void load_fc(const TT* e, float (&v)[FC]) {
#pragma unroll
    for (int f = 0; f < FC; ++f) v[f] = to_f32<TT>(__ldg(e + f));
}

// Row of vertex (g0, g1[, g2]) -- only called for taps inside the grid.
template <int D>
__device__ __forceinline__ int64_t rbf_row(const Level& lv, uint32_t tmask, int32_t g0, int32_t g1, int32_t g2) {
    uint32_t g[D];
    g[0] = static_cast<uint32_t>(g0);
    g[1] = static_cast<uint32_t>(g1);
    if constexpr (D == 3) g[2] = static_cast<uint32_t>(g2);
    return vertex_index<D>(g, lv, lv.dense & 1u, tmask);
}

// Axis-0 contraction of one row of taps (fixed g1, g2): s, s1, s2 per feature.
template <int D, int K, int FC, typename TT>
__device__ __forceinline__ void rbf_line(const TT* base, int64_t rs, int f0, const Level& lv, uint32_t tmask,
                                         const RbfAxis<K>& a0, int32_t g1, int32_t g2, float (&s)[FC],
                                         float (&s1)[FC], float (&s2)[FC]) {
#pragma unroll
    for (int f = 0; f < FC; ++f) s[f] = s1[f] = s2[f] = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if ((a0.valid >> k) & 1u) {
            float v[FC];
            load_fc<FC, TT>(base + rbf_row<D>(lv, tmask, a0.first + k, g1, g2) * rs + f0, v);
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                s[f] = fmaf(a0.w[k], v[f], s[f]);
                s1[f] = fmaf(a0.d1[k], v[f], s1[f]);
                s2[f] = fmaf(a0.d2[k], v[f], s2[f]);
            }
        }
    }
}

template <int D, int R, int FC, typename TT>
__global__ void __launch_bounds__(kBlock) rbf_fwd_kernel(const __grid_constant__ FwdParams p) {
    constexpr int K = 2 * R;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const bool active = (p.c.level_mask >> l) & 1u;
    RbfAxis<K> A[D];
    rbf_axes<D, K>(p.coords, n, lv, p.eps * p.eps, A);
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
    const int64_t rs = p.tab.rs[0];
    const uint32_t tm = p.c.tmask[0];
    for (int f0 = 0; f0 < F; f0 += FC) {
        float g[FC], dg[3][FC], lp[FC];
#pragma unroll
        for (int f = 0; f < FC; ++f) g[f] = dg[0][f] = dg[1][f] = dg[2][f] = lp[f] = 0.f;
        if (active) {
            if constexpr (D == 2) {
#pragma unroll
                for (int k1 = 0; k1 < K; ++k1) {
                    if (!((A[1].valid >> k1) & 1u)) continue;
                    float s[FC], s1[FC], s2[FC];
                    rbf_line<2, K, FC, TT>(base, rs, f0, lv, tm, A[0], A[1].first + k1, 0, s, s1, s2);
#pragma unroll
                    for (int f = 0; f < FC; ++f) {
                        g[f] = fmaf(s[f], A[1].w[k1], g[f]);
                        dg[0][f] = fmaf(s1[f], A[1].w[k1], dg[0][f]);
                        dg[1][f] = fmaf(s[f], A[1].d1[k1], dg[1][f]);
                        lp[f] = fmaf(s2[f], A[1].w[k1], fmaf(s[f], A[1].d2[k1], lp[f]));
                    }
                }
            } else {
#pragma unroll 1
                for (int k2 = 0; k2 < K; ++k2) {
                    if (!((A[2].valid >> k2) & 1u)) continue;
                    float a[FC], b[FC], cc[FC], dl[FC];
#pragma unroll
                    for (int f = 0; f < FC; ++f) a[f] = b[f] = cc[f] = dl[f] = 0.f;
#pragma unroll
                    for (int k1 = 0; k1 < K; ++k1) {
                        if (!((A[1].valid >> k1) & 1u)) continue;
                        float s[FC], s1[FC], s2[FC];
                        rbf_line<3, K, FC, TT>(base, rs, f0, lv, tm, A[0], A[1].first + k1, A[2].first + k2, s, s1,
                                               s2);
#pragma unroll
                        for (int f = 0; f < FC; ++f) {
                            a[f] = fmaf(s[f], A[1].w[k1], a[f]);
                            b[f] = fmaf(s1[f], A[1].w[k1], b[f]);
                            cc[f] = fmaf(s[f], A[1].d1[k1], cc[f]);
                            dl[f] = fmaf(s2[f], A[1].w[k1], fmaf(s[f], A[1].d2[k1], dl[f]));
                        }
                    }
                    const float w2 = A[2].w[k2], d12 = A[2].d1[k2], d22 = A[2].d2[k2];
#pragma unroll
                    for (int f = 0; f < FC; ++f) {
                        g[f] = fmaf(a[f], w2, g[f]);
                        dg[0][f] = fmaf(b[f], w2, dg[0][f]);
                        dg[1][f] = fmaf(cc[f], w2, dg[1][f]);
                        dg[2][f] = fmaf(a[f], d12, dg[2][f]);
                        lp[f] = fmaf(dl[f], w2, fmaf(a[f], d22, lp[f]));
                    }
                }
            }
        }
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
            __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, g[f]);
            if (p.dgamma) {
#pragma unroll
                for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, dg[j][f]);
            }
            if (p.lap) __stcs(p.lap + n * p.c.sn + lf * p.c.sf, lp[f]);
        }
    }
}

// Transposed contraction of one (point, level, feature chunk): the
// coefficient gradient of every tap inside the grid, handed to
// add(g0, g1, g2, values) with the tap's vertex coordinates (g2 = 0 in 2D).
template <int D, int R, int FC, typename Add>
__device__ __forceinline__ void rbf_point_bwd(const BwdParams& p, int64_t n, int l, int f0, const RbfAxis<2 * R> (&A)[D],
                                              const Level& lv, Add&& add) {
    constexpr int K = 2 * R;
    const int F = p.c.F;
    float gg[FC], gd[3][FC], gl[FC];
#pragma unroll
    for (int f = 0; f < FC; ++f) {
        const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
        gg[f] = p.g_gamma ? __ldg(p.g_gamma + n * p.c.sn + lf * p.c.sf) : 0.f;
        gl[f] = p.g_lap ? __ldg(p.g_lap + n * p.c.sn + lf * p.c.sf) : 0.f;
#pragma unroll
        for (int j = 0; j < 3; ++j)
            gd[j][f] = (p.g_dgamma && j < D) ? __ldg(p.g_dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf) : 0.f;
    }
    // per (g1[, g2]): the adjoints s, s1, s2 of the axis-0 line sums, then each tap's gradient
    auto line = [&](int32_t g1, int32_t g2, const float (&s)[FC], const float (&s1)[FC], const float (&s2)[FC]) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if ((A[0].valid >> k) & 1u) {
                float v[FC];
#pragma unroll
                for (int f = 0; f < FC; ++f) v[f] = fmaf(s[f], A[0].w[k], fmaf(s1[f], A[0].d1[k], s2[f] * A[0].d2[k]));
                add(A[0].first + k, g1, g2, v);
            }
        }
    };
    if constexpr (D == 2) {
#pragma unroll
        for (int k1 = 0; k1 < K; ++k1) {
            if (!((A[1].valid >> k1) & 1u)) continue;
            float s[FC], s1[FC], s2[FC];
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                s[f] = fmaf(gg[f], A[1].w[k1], fmaf(gd[1][f], A[1].d1[k1], gl[f] * A[1].d2[k1]));
                s1[f] = gd[0][f] * A[1].w[k1];
                s2[f] = gl[f] * A[1].w[k1];
            }
            line(A[1].first + k1, 0, s, s1, s2);
        }
    } else {
#pragma unroll 1
        for (int k2 = 0; k2 < K; ++k2) {
            if (!((A[2].valid >> k2) & 1u)) continue;
            const float w2 = A[2].w[k2], d12 = A[2].d1[k2], d22 = A[2].d2[k2];
            float a[FC], b[FC], cc[FC], dl[FC];
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                a[f] = fmaf(gg[f], w2, fmaf(gd[2][f], d12, gl[f] * d22));
                b[f] = gd[0][f] * w2;
                cc[f] = gd[1][f] * w2;
                dl[f] = gl[f] * w2;
            }
#pragma unroll
            for (int k1 = 0; k1 < K; ++k1) {
                if (!((A[1].valid >> k1) & 1u)) continue;
                float s[FC], s1[FC], s2[FC];
#pragma unroll
                for (int f = 0; f < FC; ++f) {
                    s[f] = fmaf(a[f], A[1].w[k1], fmaf(cc[f], A[1].d1[k1], dl[f] * A[1].d2[k1]));
                    s1[f] = b[f] * A[1].w[k1];
                    s2[f] = dl[f] * A[1].w[k1];
                }
                line(A[1].first + k1, A[2].first + k2, s, s1, s2);
            }
        }
    }
}

constexpr int kTileBlock = 256;  // 8 warps: the lane interleave below relies on it
static_assert(kTileBlock == 8 * 32, "eight warps of 32 lanes");
constexpr int kTileFloats = 24 * 1024;  // 96 KB of dynamic shared memory: two CTAs per SM

// Tiled backward for coherent points (the page's structured sampling): a CTA
// takes kTileBlock consecutive points of one level, finds the bounding box
// of their tap neighbourhoods (a block reduction of their cells), and when
// the box's rows fit kTileFloats it accumulates every contribution in a
// shared-memory tile of that box and then adds each touched row into the
// table once -- consecutive stratified points share most of their taps, so
// this replaces tens of REDs on the same rows by one.  A CTA whose box does
// not fit (scattered points on a fine level) scatters directly.
template <int D, int R, int FC, bool VEC>
__global__ void __launch_bounds__(kTileBlock) rbf_bwd_tile_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ float tile[];
    __shared__ int32_t box_lo[3], box_hi[3];
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    // the CTA's points, interleaved over the lanes: lane j of warp w takes point w + 8 j, so the lanes of
    // one instruction sit in different cells and their shared-memory adds rarely collide (measured: 2D
    // workload 1.70 -> 0.82 ms, 3D 22.5 -> 13.3 ms against consecutive points per warp)
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kTileBlock + (threadIdx.x >> 5) + 8 * (threadIdx.x & 31);
    const bool have = n < p.c.n;
    const Level& lv = p.c.lv[l];
    const int F = p.c.F;
    RbfAxis<2 * R> A[D];
    if (have) rbf_axes<D, 2 * R>(p.coords, n, lv, p.eps * p.eps, A);
    // bounding box of the CTA's taps, clipped to the grid
    if (threadIdx.x < 3) {
        box_lo[threadIdx.x] = INT32_MAX;
        box_hi[threadIdx.x] = INT32_MIN;
    }
    __syncthreads();
    if (have) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            atomicMin(&box_lo[i], max(A[i].first, 0));
            atomicMax(&box_hi[i], min(A[i].first + 2 * R - 1, static_cast<int32_t>(lv.N)));
        }
    }
    __syncthreads();
    int32_t lo[3] = {0, 0, 0}, ext[3] = {1, 1, 1};
    int64_t vol = 1;
#pragma unroll
    for (int i = 0; i < D; ++i) {
        lo[i] = box_lo[i];
        ext[i] = box_hi[i] - box_lo[i] + 1;
        vol *= ext[i];
    }
    float* base = p.grad.ptr[0] + l * p.grad.ls[0];
    const uint32_t tm = p.c.tmask[0];
    if (vol * F > kTileFloats) {  // the same branch for the whole CTA: scatter directly
        if (!have) return;
        for (int f0 = 0; f0 < F; f0 += FC) {
            rbf_point_bwd<D, R, FC>(p, n, l, f0, A, lv, [&](int32_t g0, int32_t g1, int32_t g2, const float (&v)[FC]) {
                float* e = base + rbf_row<D>(lv, tm, g0, g1, g2) * p.grad.rs[0] + f0;
                if constexpr (VEC) {
                    red_add_v2(e, v[0], v[FC - 1]);
                } else {
#pragma unroll
                    for (int f = 0; f < FC; ++f) red_add_f32(e + f, v[f]);
                }
            });
        }
        return;
    }
    const int32_t vals = static_cast<int32_t>(vol) * F;
    for (int32_t i = threadIdx.x; i < vals; i += kTileBlock) tile[i] = 0.f;
    __syncthreads();
    if (have) {
        for (int f0 = 0; f0 < F; f0 += FC) {
            rbf_point_bwd<D, R, FC>(p, n, l, f0, A, lv, [&](int32_t g0, int32_t g1, int32_t g2, const float (&v)[FC]) {
                const int32_t r = (g0 - lo[0]) + ext[0] * ((g1 - lo[1]) + ext[1] * (D == 3 ? g2 - lo[2] : 0));
                float* a = tile + r * F + f0;
#pragma unroll
                for (int f = 0; f < FC; ++f) atomicAdd(a + f, v[f]);
            });
        }
    }
    __syncthreads();
    for (int32_t r = threadIdx.x; r < static_cast<int32_t>(vol); r += kTileBlock) {
        const int32_t g0 = lo[0] + r % ext[0];
        const int32_t g1 = lo[1] + (r / ext[0]) % ext[1];
        const int32_t g2 = D == 3 ? lo[2] + r / (ext[0] * ext[1]) : 0;
        float* e = base + rbf_row<D>(lv, tm, g0, g1, g2) * p.grad.rs[0];
        const float* a = tile + r * F;
        for (int f0 = 0; f0 < F; f0 += FC) {
            bool any = false;
#pragma unroll
            for (int f = 0; f < FC; ++f) any = any || a[f0 + f] != 0.f;
            if (!any) continue;
            if constexpr (VEC) {
                red_add_v2(e + f0, a[f0], a[f0 + FC - 1]);
            } else {
#pragma unroll
                for (int f = 0; f < FC; ++f) red_add_f32(e + f0 + f, a[f0 + f]);
            }
        }
    }
}

template <int D, int R, int FC, typename TT>
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    rbf_fwd_kernel<D, R, FC, TT><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, int R, typename TT>
cudaError_t pick_fwd(const FwdParams& p, int fc, cudaStream_t s) {
    return fc == 2 ? launch_fwd<D, R, 2, TT>(p, s) : launch_fwd<D, R, 1, TT>(p, s);
}

template <int D, int R, int FC, bool VEC>
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t s) {
    if (p.c.nlvl == 0) return cudaSuccess;
    constexpr int kSmem = kTileFloats * static_cast<int>(sizeof(float));
    cudaError_t e = cudaFuncSetAttribute(rbf_bwd_tile_kernel<D, R, FC, VEC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>((p.c.n + kTileBlock - 1) / kTileBlock), static_cast<unsigned>(p.c.nlvl));
    rbf_bwd_tile_kernel<D, R, FC, VEC><<<grid, kTileBlock, kSmem, s>>>(p);
    return cudaGetLastError();
}

template <int D, int R>
cudaError_t pick_bwd(const BwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (fc == 2) return vec ? launch_bwd<D, R, 2, true>(p, s) : launch_bwd<D, R, 2, false>(p, s);
    return launch_bwd<D, R, 1, false>(p, s);
}

template <int D, typename TT>
cudaError_t fwd_rings(const FwdParams& p, int fc, int rings, cudaStream_t s) {
    switch (rings) {
        case 1: return pick_fwd<D, 1, TT>(p, fc, s);
        case 2: return pick_fwd<D, 2, TT>(p, fc, s);
        case 3: return pick_fwd<D, 3, TT>(p, fc, s);
        default: return pick_fwd<D, 4, TT>(p, fc, s);
    }
}

template <int D>
cudaError_t bwd_rings(const BwdParams& p, int fc, bool vec, int rings, cudaStream_t s) {
    switch (rings) {
        case 1: return pick_bwd<D, 1>(p, fc, vec, s);
        case 2: return pick_bwd<D, 2>(p, fc, vec, s);
        case 3: return pick_bwd<D, 3>(p, fc, vec, s);
        default: return pick_bwd<D, 4>(p, fc, vec, s);
    }
}

}  // namespace

int launch_rbf_fwd(const FwdParams& p, int fc, int rings, int dtype, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.c.d == 2) return dtype == HG_F16 ? fwd_rings<2, __half>(p, fc, rings, s) : fwd_rings<2, float>(p, fc, rings, s);
    return dtype == HG_F16 ? fwd_rings<3, __half>(p, fc, rings, s) : fwd_rings<3, float>(p, fc, rings, s);
}

int launch_rbf_bwd(const BwdParams& p, int fc, bool vec, int rings, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return p.c.d == 2 ? bwd_rings<2>(p, fc, vec, rings, s) : bwd_rings<3>(p, fc, vec, rings, s);
}

}  // namespace hg
