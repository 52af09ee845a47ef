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
// For coherent points a CTA first stages the table rows of its taps'
// bounding box in shared memory (rbf_fwd_box_kernel).
// The backward is the transposed contraction, accumulated per CTA in a
// shared-memory tile of its points' neighbourhoods (the page samples
// stratified points, so a CTA's points are neighbours) before the scatter,
// one thread per run of same-cell points and tap row, with the points'
// separable factors summed in registers (rbf_bwd_cells_kernel).
#include <cuda_runtime.h>

#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;

// The 2R taps of one axis: vertex g = first + k (bit k of `valid` set when
// it lies inside the grid) and its normalised 1D weight w[k].  The weight's
// derivatives need no more per-tap state: with e_k = exp(-eps^2 r_k^2),
// r_k = y - g_k, the quotient rule gives dw_k/dy = -2 eps^2 w_k delta_k and
// d2w_k/dy2 = 4 eps^4 w_k (delta_k^2 - var), where delta_k = r_k - mu and
// mu, var are the weighted mean and variance of the offsets r_k.  So an
// axis holds 2R weights plus tau = delta_0 (delta_k = tau - k) and var,
// which keeps three axes of a point in registers.
template <int K>
struct RbfAxis {
    int32_t first;
    uint32_t valid;
    float tau, var;
    float w[K];
};

template <int K>
__device__ __forceinline__ RbfAxis<K> rbf_axis(uint32_t c, float t, const Level& lv, float eps2) {
    RbfAxis<K> a;
    a.first = static_cast<int32_t>(c) - K / 2 + 1;
    a.valid = 0u;
    float e[K], s = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int32_t g = a.first + k;
        const bool in = g >= 0 && g <= static_cast<int32_t>(lv.N);
        a.valid |= static_cast<uint32_t>(in) << k;
        const float r = t - static_cast<float>(k - K / 2 + 1);        // y - g, in grid units
        e[k] = in ? expf(-eps2 * r * r) : 0.f;
        s += e[k];
    }
    const float inv = 1.f / s;
    float mu = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        a.w[k] = e[k] * inv;
        mu = fmaf(a.w[k], t - static_cast<float>(k - K / 2 + 1), mu);
    }
    a.tau = (t - mu) + static_cast<float>(K / 2 - 1);
    float var = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float dl = a.tau - static_cast<float>(k);
        var = fmaf(a.w[k] * dl, dl, var);
    }
    a.var = var;
    return a;
}

// w[k] for a k only known at run time, by selects: indexing the array
// itself would move the point's axes to local memory.
template <int K>
__device__ __forceinline__ float rbf_weight(const RbfAxis<K>& a, int k) {
    float w = a.w[0];
#pragma unroll
    for (int j = 1; j < K; ++j) w = k == j ? a.w[j] : w;
    return w;
}

// delta_k and q_k = delta_k^2 - var of tap k of an axis.
template <int K>
__device__ __forceinline__ void rbf_moments(const RbfAxis<K>& a, int k, float& dl, float& q) {
    dl = a.tau - static_cast<float>(k);
    q = fmaf(dl, dl, -a.var);
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

// Axis-0 contraction of one row of taps (fixed g1, g2) per feature:
// s = sum w theta, sd = sum w delta theta, sq = sum w q theta.
template <int D, int K, int FC, typename TT>
__device__ __forceinline__ void rbf_line(const TT* base, int64_t rs, int f0, const Level& lv, uint32_t tmask,
                                         const RbfAxis<K>& a0, int32_t g1, int32_t g2, float (&s)[FC],
                                         float (&sd)[FC], float (&sq)[FC]) {
#pragma unroll
    for (int f = 0; f < FC; ++f) s[f] = sd[f] = sq[f] = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if ((a0.valid >> k) & 1u) {
            float v[FC], dl, q;
            load_fc<FC, TT>(base + rbf_row<D>(lv, tmask, a0.first + k, g1, g2) * rs + f0, v);
            rbf_moments(a0, k, dl, q);
            const float wd = a0.w[k] * dl, wq = a0.w[k] * q;
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                s[f] = fmaf(a0.w[k], v[f], s[f]);
                sd[f] = fmaf(wd, v[f], sd[f]);
                sq[f] = fmaf(wq, v[f], sq[f]);
            }
        }
    }
}

// gamma, d gamma / d x_i and lap gamma of one point and feature chunk from
// the axis-0 sums of each tap row: line(k1, k2, s, sd, sq) returns, for the
// row of taps (k1, k2) (k2 = 0 in 2D), s = sum w theta, sd = sum w delta
// theta and sq = sum w q theta over k0.  The outer axes fold in as the
// Hermite blend does: in offset units dg_i = sum W delta_i theta and
// lp = sum W (q_0 + q_1 [+ q_2]) theta with the tap weight W = w_0 w_1 [w_2];
// the gradient and Laplacian are -v dg and v^2 lp.
template <int D, int K, int FC, typename Line>
__device__ __forceinline__ void rbf_contract(const RbfAxis<K> (&A)[D], float v, float (&g)[FC], float (&dg)[3][FC],
                                             float (&lp)[FC], Line&& line) {
#pragma unroll
    for (int f = 0; f < FC; ++f) g[f] = dg[0][f] = dg[1][f] = dg[2][f] = lp[f] = 0.f;
    if constexpr (D == 2) {
#pragma unroll
        for (int k1 = 0; k1 < K; ++k1) {
            if (!((A[1].valid >> k1) & 1u)) continue;
            float s[FC], sd[FC], sq[FC], dl1, q1;
            line(k1, 0, s, sd, sq);
            rbf_moments(A[1], k1, dl1, q1);
            const float w1 = A[1].w[k1], wd1 = w1 * dl1;
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                g[f] = fmaf(w1, s[f], g[f]);
                dg[0][f] = fmaf(w1, sd[f], dg[0][f]);
                dg[1][f] = fmaf(wd1, s[f], dg[1][f]);
                lp[f] = fmaf(w1, fmaf(q1, s[f], sq[f]), lp[f]);
            }
        }
    } else {
#pragma unroll 1
        for (int k2 = 0; k2 < K; ++k2) {
            if (!((A[D - 1].valid >> k2) & 1u)) continue;
            float a[FC], b[FC], cc[FC], dl[FC];
#pragma unroll
            for (int f = 0; f < FC; ++f) a[f] = b[f] = cc[f] = dl[f] = 0.f;
#pragma unroll
            for (int k1 = 0; k1 < K; ++k1) {
                if (!((A[1].valid >> k1) & 1u)) continue;
                float s[FC], sd[FC], sq[FC], dl1, q1;
                line(k1, k2, s, sd, sq);
                rbf_moments(A[1], k1, dl1, q1);
                const float w1 = A[1].w[k1], wd1 = w1 * dl1;
#pragma unroll
                for (int f = 0; f < FC; ++f) {
                    a[f] = fmaf(w1, s[f], a[f]);
                    b[f] = fmaf(w1, sd[f], b[f]);
                    cc[f] = fmaf(wd1, s[f], cc[f]);
                    dl[f] = fmaf(w1, fmaf(q1, s[f], sq[f]), dl[f]);
                }
            }
            float dl2, q2;
            rbf_moments(A[D - 1], k2, dl2, q2);
            const float w2 = rbf_weight(A[D - 1], k2), wd2 = w2 * dl2;
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                g[f] = fmaf(w2, a[f], g[f]);
                dg[0][f] = fmaf(w2, b[f], dg[0][f]);
                dg[1][f] = fmaf(w2, cc[f], dg[1][f]);
                dg[2][f] = fmaf(wd2, a[f], dg[2][f]);
                lp[f] = fmaf(w2, fmaf(q2, a[f], dl[f]), lp[f]);
            }
        }
    }
#pragma unroll
    for (int f = 0; f < FC; ++f) {
        lp[f] *= v * v;
#pragma unroll
        for (int j = 0; j < 3; ++j) dg[j][f] *= -v;
    }
}

template <int D, int FC>
__device__ __forceinline__ void rbf_store(const FwdParams& p, int64_t n, int l, int f0, const float (&g)[FC],
                                          const float (&dg)[3][FC], const float (&lp)[FC]) {
#pragma unroll
    for (int f = 0; f < FC; ++f) {
        const int64_t lf = static_cast<int64_t>(l) * p.c.F + f0 + f;
        __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, g[f]);
        if (p.dgamma) {
#pragma unroll
            for (int j = 0; j < D; ++j) __stcs(p.dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf, dg[j][f]);
        }
        if (p.lap) __stcs(p.lap + n * p.c.sn + lf * p.c.sf, lp[f]);
    }
}

// One point, every feature chunk, taps gathered from the table (through L1).
template <int D, int K, int FC, typename TT>
__device__ __forceinline__ void rbf_fwd_gather(const FwdParams& p, int64_t n, int l, const Level& lv, bool active,
                                               const RbfAxis<K> (&A)[D]) {
    const float v = 2.f * p.eps * p.eps * lv.fN;  // d/dx = N d/dy on the weights' derivatives
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
    const int64_t rs = p.tab.rs[0];
    const uint32_t tm = p.c.tmask[0];
    for (int f0 = 0; f0 < p.c.F; f0 += FC) {
        float g[FC], dg[3][FC], lp[FC];
        if (active) {
            rbf_contract<D, K, FC>(A, v, g, dg, lp,
                                   [&](int k1, int k2, float (&s)[FC], float (&sd)[FC], float (&sq)[FC]) {
                                       int32_t g2 = 0;
                                       if constexpr (D == 3) g2 = A[D - 1].first + k2;
                                       rbf_line<D, K, FC, TT>(base, rs, f0, lv, tm, A[0], A[1].first + k1, g2, s,
                                                              sd, sq);
                                   });
        } else {
#pragma unroll
            for (int f = 0; f < FC; ++f) g[f] = dg[0][f] = dg[1][f] = dg[2][f] = lp[f] = 0.f;
        }
        rbf_store<D, FC>(p, n, l, f0, g, dg, lp);
    }
}

// Box-staged forward for coherent points: a CTA of kBlock consecutive points
// first copies the rows of its taps' bounding box -- not clipped to the
// grid; rows outside it are zeros, as their weights are -- into shared
// memory (fp32), then each point reads tap row (k1, k2) at a fixed offset
// from its own corner of the box: no hash, no bounds test and no L1 gather
// per tap, and the axis-0 weights and their moment products are computed
// once per point instead of once per tap row.  A CTA whose box does not
// fit (scattered points) gathers each tap row from the table through L1;
// that path is latency-bound and runs at this kernel's occupancy (a
// gather-only kernel measured 3.82 / 2.81 / 2.62 ms on the 3D workload at
// two / four / six blocks per SM, against 1.23 ms for the box path).
// CTAs per SM: the register budget against latency hiding, measured on the full-size workloads -- 3D
// (box of 61 x 7 x 6 rows) 1.35 / 1.23 / 1.22 ms at 2 / 3 / 4 (4 spills), 2D 0.244 / 0.262 / 0.289 ms.
constexpr int kBoxFloats = 6 * 1024;  // 24 KB: two stratified rows of 128 points on the 3D grid's finest level
template <int D>
constexpr int box_ctas() { return D == 2 ? 2 : 3; }

template <int D, int R, int FC, typename TT>
__global__ void __launch_bounds__(kBlock, box_ctas<D>()) rbf_fwd_box_kernel(const __grid_constant__ FwdParams p) {
    constexpr int K = 2 * R;
    extern __shared__ float4 box_smem4[];
    float* box = reinterpret_cast<float*>(box_smem4);
    __shared__ int32_t box_lo[3], box_hi[3];
    const int l = p.c.lvl[blockIdx.y];
    const int t = threadIdx.x;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kBlock;
    const int cnt = static_cast<int>(min(static_cast<int64_t>(kBlock), p.c.n - n0));
    const bool have = t < cnt;
    const int64_t n = n0 + (have ? t : cnt - 1);
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const bool active = (p.c.level_mask >> l) & 1u;
    RbfAxis<K> A[D];
    rbf_axes<D, K>(p.coords, n, lv, p.eps * p.eps, A);
    if (!active) {  // the same for the whole CTA
        if (have) rbf_fwd_gather<D, K, FC, TT>(p, n, l, lv, false, A);
        return;
    }
    if (t < 3) {
        box_lo[t] = t < D ? INT32_MAX : 0;
        box_hi[t] = t < D ? INT32_MIN : 0;
    }
    __syncthreads();
    if (have) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            atomicMin(&box_lo[i], A[i].first);
            atomicMax(&box_hi[i], A[i].first + K - 1);
        }
    }
    __syncthreads();
    int32_t lo[3], ext[3];
    int64_t vol = 1;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        lo[i] = box_lo[i];
        ext[i] = box_hi[i] - box_lo[i] + 1;
        vol *= ext[i];
    }
    if (vol * F > kBoxFloats) {  // the same for the whole CTA
        if (have) rbf_fwd_gather<D, K, FC, TT>(p, n, l, lv, true, A);
        return;
    }
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
    const int64_t rs = p.tab.rs[0];
    const uint32_t tm = p.c.tmask[0];
    const int32_t N = static_cast<int32_t>(lv.N);
    for (int32_t r = t; r < static_cast<int32_t>(vol); r += kBlock) {
        const int32_t g0 = lo[0] + r % ext[0];
        const int32_t g1 = lo[1] + (r / ext[0]) % ext[1];
        const int32_t g2 = lo[2] + r / (ext[0] * ext[1]);
        const bool in = g0 >= 0 && g0 <= N && g1 >= 0 && g1 <= N && (D == 2 || (g2 >= 0 && g2 <= N));
        float* dst = box + r * F;
        if (in) {
            const TT* src = base + rbf_row<D>(lv, tm, g0, g1, g2) * rs;
            for (int f = 0; f < F; ++f) dst[f] = to_f32<TT>(__ldg(src + f));
        } else {
            for (int f = 0; f < F; ++f) dst[f] = 0.f;
        }
    }
    __syncthreads();
    if (!have) return;
    float w0[K], wd0[K], wq0[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        float dl, q;
        rbf_moments(A[0], k, dl, q);
        w0[k] = A[0].w[k];
        wd0[k] = w0[k] * dl;
        wq0[k] = w0[k] * q;
    }
    int32_t o2 = 0;
    if constexpr (D == 3) o2 = A[D - 1].first - lo[2];
    const float* corner = box + (A[0].first - lo[0] + ext[0] * (A[1].first - lo[1] + ext[1] * o2)) * F;
    const int32_t s1 = ext[0] * F, s2 = ext[0] * ext[1] * F;  // floats between tap rows along axes 1 and 2
    const float v = 2.f * p.eps * p.eps * lv.fN;
    for (int f0 = 0; f0 < F; f0 += FC) {
        float g[FC], dg[3][FC], lp[FC];
        rbf_contract<D, K, FC>(A, v, g, dg, lp, [&](int k1, int k2, float (&s)[FC], float (&sd)[FC], float (&sq)[FC]) {
            const float* row = corner + k1 * s1 + k2 * s2 + f0;
#pragma unroll
            for (int f = 0; f < FC; ++f) s[f] = sd[f] = sq[f] = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float x[FC];
                if constexpr (FC == 2) {
                    const float2 y = *reinterpret_cast<const float2*>(row + k * F);
                    x[0] = y.x;
                    x[FC - 1] = y.y;
                } else {
                    x[0] = row[k * F];
                }
#pragma unroll
                for (int f = 0; f < FC; ++f) {
                    s[f] = fmaf(w0[k], x[f], s[f]);
                    sd[f] = fmaf(wd0[k], x[f], sd[f]);
                    sq[f] = fmaf(wq0[k], x[f], sq[f]);
                }
            }
        });
        rbf_store<D, FC>(p, n, l, f0, g, dg, lp);
    }
}

// Cell-run backward.  The points of a run (consecutive points in one cell)
// share their K^d taps, and with the moment form above the gradient of tap
// (k0, k1, k2) summed over the run's points is
//   sum_p  w0[k0] Sw[k1,k2] + (w0 delta0)[k0] Sd[k1,k2] + (w0 q0)[k0] Sq[k1,k2],
// where per point P = w1 w2, Sd = bd0 P, Sq = cl P and
//   Sw = a0 P + bd1 (w1 delta1) w2 + bd2 w1 (w2 delta2) + cl ((w1 q1) w2 + w1 (w2 q2))
// (a0 = g_gamma, bd_i = -v g_dgamma_i, cl = v^2 g_lap; in 2D w2 = 1 and
// delta2 = q2 = 0): the transposed contraction with axis 0 folded in last.  A CTA writes each point's
// factors to shared memory (axis 0's three weight vectors, the weights and
// moments of axes 1 and 2, the upstream coefficients), then one thread per
// (run, k1, k2) -- kCellRows rows k1 of one k2 -- sums the K x FC gradients
// of its taps over the run's points
// in registers and adds each into the CTA's tile once.  Per point this
// takes about a sixth of the instructions of a per-point scatter with the
// runs summed by warp shuffles (3D: 6.9 -> 2.6 ms; 2D: 0.49 -> 0.42 ms), and
// one shared-memory add per tap and run instead of per tap and point.  The
// tile covers the bounding box of the CTA's taps (clipped to the grid); each
// touched row is added to the table once.  When it does not fit (scattered
// points on a fine level), each run's taps are added to the table directly.
// Any point order is correct; a random one gives runs of one point.
constexpr int kCellBlock = 256;
constexpr int kCellTileFloats = 6 * 1024;  // 24 KB: the full-grid 3D box of two stratified rows of 128 points
constexpr int kCellCtas = 3;
// Tap rows k1 per thread: more rows share the point's shared-memory loads but leave fewer threads per
// run.  Measured on the full-size workloads at one / two / three rows: 3D 2.61 / 2.78 / 2.99 ms, 2D
// 0.42 / 0.46 / 0.47 ms.
constexpr int kCellRows = 1;

template <int D, int K, int FC>
struct CellRec {
    static constexpr int a0 = 0;                  // w0[K], (w0 delta0)[K], (w0 q0)[K]
    static constexpr int a1 = 3 * K;              // w1[K], tau1, var1
    static constexpr int a2 = a1 + K + 2;         // 3D: w2[K], tau2, var2
    static constexpr int coef = a1 + (D - 1) * (K + 2);  // a0[FC], bd0[FC], bd1[FC], bd2[FC], cl[FC]
    static constexpr int key = coef + 5 * FC;     // the cell: first tap of each axis (int32)
    static constexpr int size = (key + 3 + 3) & ~3;  // floats; a multiple of 4 keeps records 16-byte aligned
    static_assert((3 * K) % 4 == 0 || (3 * K) % 4 == 2, "axis-0 block: float4s and at most one float2");
    static_assert(a1 % 2 == 0 && a2 % 2 == 0 && coef % 2 == 0, "float2 fields");
};

template <int D, int K, int FC>
constexpr int cell_smem_bytes() {
    return (kCellBlock * CellRec<D, K, FC>::size + kCellTileFloats) * static_cast<int>(sizeof(float));
}

// v[0 .. M) from 16-byte-aligned shared memory, in float4 loads (and one float2).
template <int M>
__device__ __forceinline__ void lds_floats(const float* s, float (&v)[M]) {
#pragma unroll
    for (int i = 0; i + 4 <= M; i += 4) {
        const float4 x = *reinterpret_cast<const float4*>(s + i);
        v[i] = x.x;
        v[i + 1] = x.y;
        v[i + 2] = x.z;
        v[i + 3] = x.w;
    }
    if constexpr (M % 4 == 2) {
        const float2 x = *reinterpret_cast<const float2*>(s + M - 2);
        v[M - 2] = x.x;
        v[M - 1] = x.y;
    }
}

template <int D, int R, int FC, bool VEC>
__global__ void __launch_bounds__(kCellBlock, kCellCtas) rbf_bwd_cells_kernel(const __grid_constant__ BwdParams p) {
    constexpr int K = 2 * R;
    using Rec = CellRec<D, K, FC>;
    constexpr int J = K % kCellRows == 0 ? kCellRows : 1;  // tap rows of a thread: k1, k1 + K/J, ...
    constexpr int kItems = (K / J) * (D == 3 ? K : 1);       // threads per run
    constexpr int kSlots = kCellBlock / kItems;              // runs in progress at once
    static_assert(kSlots >= 1, "a run's threads fit the block");
    extern __shared__ float4 cell_smem4[];
    float* rec = reinterpret_cast<float*>(cell_smem4);  // [kCellBlock][Rec::size]
    float* tile = rec + kCellBlock * Rec::size;         // [kCellTileFloats]
    __shared__ int32_t box_lo[3], box_hi[3];
    __shared__ int32_t run_start[kCellBlock + 1];
    __shared__ int32_t warp_runs[kCellBlock / 32];
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kCellBlock;
    const int cnt = static_cast<int>(min(static_cast<int64_t>(kCellBlock), p.c.n - n0));
    const bool have = t < cnt;
    const int64_t n = n0 + (have ? t : cnt - 1);
    const Level& lv = p.c.lv[l];
    const int F = p.c.F;
    const int32_t N = static_cast<int32_t>(lv.N);
    const float v = 2.f * p.eps * p.eps * lv.fN;
    float* my = rec + t * Rec::size;
    int32_t* my_key = reinterpret_cast<int32_t*>(my + Rec::key);
    {
        RbfAxis<K> A[D];
        rbf_axes<D, K>(p.coords, n, lv, p.eps * p.eps, A);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float dl, q;
            rbf_moments(A[0], k, dl, q);
            my[Rec::a0 + k] = A[0].w[k];
            my[Rec::a0 + K + k] = A[0].w[k] * dl;
            my[Rec::a0 + 2 * K + k] = A[0].w[k] * q;
            my[Rec::a1 + k] = A[1].w[k];
            if constexpr (D == 3) my[Rec::a2 + k] = A[D - 1].w[k];
        }
        my[Rec::a1 + K] = A[1].tau;
        my[Rec::a1 + K + 1] = A[1].var;
        if constexpr (D == 3) {
            my[Rec::a2 + K] = A[D - 1].tau;
            my[Rec::a2 + K + 1] = A[D - 1].var;
        }
        my_key[0] = A[0].first;
        my_key[1] = A[1].first;
        my_key[2] = D == 3 ? A[D - 1].first : 0;
        if (t < 3) {  // an absent axis 2 spans the single index 0
            box_lo[t] = t < D ? INT32_MAX : 0;
            box_hi[t] = t < D ? INT32_MIN : 0;
        }
    }
    __syncthreads();
    // bounding box of the CTA's taps (clipped to the grid), and the runs: a point starts one when its cell
    // differs from the previous point's
    bool lead = false;
    if (have) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            atomicMin(&box_lo[i], max(my_key[i], 0));
            atomicMax(&box_hi[i], min(my_key[i] + K - 1, N));
        }
        lead = t == 0;
        if (!lead) {
            const int32_t* prev = reinterpret_cast<const int32_t*>(my - Rec::size + Rec::key);
            lead = prev[0] != my_key[0] || prev[1] != my_key[1] || prev[2] != my_key[2];
        }
    }
    const uint32_t ball = __ballot_sync(0xffffffffu, lead);
    if (lane == 0) warp_runs[warp] = __popc(ball);
    __syncthreads();
    int before = 0, runs = 0;
#pragma unroll
    for (int w = 0; w < kCellBlock / 32; ++w) {
        const int c = warp_runs[w];
        before += w < warp ? c : 0;
        runs += c;
    }
    if (lead) run_start[before + __popc(ball & ((1u << lane) - 1u))] = t;
    if (t == 0) run_start[runs] = cnt;
    int32_t lo[3], ext[3];
    int64_t vol = 1;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        lo[i] = box_lo[i];
        ext[i] = box_hi[i] - box_lo[i] + 1;
        vol *= ext[i];
    }
    const bool tiled = vol * F <= kCellTileFloats;  // the same for the whole CTA
    if (tiled)
        for (int32_t i = t; i < static_cast<int32_t>(vol) * F; i += kCellBlock) tile[i] = 0.f;
    float* gbase = p.grad.ptr[0] + l * p.grad.ls[0];
    const int64_t rs = p.grad.rs[0];
    const uint32_t tm = p.c.tmask[0];
    const int slot = t / kItems, item = t - slot * kItems;
    const int k1 = item % (K / J), k2 = item / (K / J);
    for (int f0 = 0; f0 < F; f0 += FC) {
        // the point's upstream coefficients for this feature chunk (zero past the end)
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
            float c[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
            if (have) {
                if (p.g_gamma) c[0] = __ldg(p.g_gamma + n * p.c.sn + lf * p.c.sf);
                if (p.g_dgamma) {
#pragma unroll
                    for (int j = 0; j < D; ++j) c[1 + j] = -v * __ldg(p.g_dgamma + n * p.c.dsn + j * p.c.dsj + lf * p.c.dsf);
                }
                if (p.g_lap) c[4] = v * v * __ldg(p.g_lap + n * p.c.sn + lf * p.c.sf);
            }
#pragma unroll
            for (int j = 0; j < 5; ++j) my[Rec::coef + j * FC + f] = c[j];
        }
        __syncthreads();
        if (slot < kSlots) {
            for (int r = slot; r < runs; r += kSlots) {
                const int pa = run_start[r], pb = run_start[r + 1];
                const int32_t* key = reinterpret_cast<const int32_t*>(rec + pa * Rec::size + Rec::key);
                const int32_t g0 = key[0], g2 = key[2] + k2;
                bool in1[J], any = false;
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int32_t g1 = key[1] + k1 + j * (K / J);
                    in1[j] = g1 >= 0 && g1 <= N;
                    any = any || in1[j];
                }
                if (!any || g2 < 0 || g2 > N) continue;  // outside the grid: weight 0, no row
                float acc[J][K][FC];
#pragma unroll
                for (int j = 0; j < J; ++j)
#pragma unroll
                    for (int k = 0; k < K; ++k)
#pragma unroll
                        for (int f = 0; f < FC; ++f) acc[j][k][f] = 0.f;
#pragma unroll 1
                for (int q = pa; q < pb; ++q) {
                    const float* pr = rec + q * Rec::size;
                    float a0[3 * K];
                    lds_floats<3 * K>(pr + Rec::a0, a0);
                    const float2 m1 = *reinterpret_cast<const float2*>(pr + Rec::a1 + K);
                    float w2 = 1.f, wd2 = 0.f, wq2 = 0.f;
                    if constexpr (D == 3) {
                        w2 = pr[Rec::a2 + k2];
                        const float2 m2 = *reinterpret_cast<const float2*>(pr + Rec::a2 + K);
                        const float dl2 = m2.x - static_cast<float>(k2), q2 = fmaf(dl2, dl2, -m2.y);
                        wd2 = w2 * dl2;
                        wq2 = w2 * q2;
                    }
                    float c[5][FC];
                    if constexpr (FC == 2) {
#pragma unroll
                        for (int i = 0; i < 5; ++i) {
                            const float2 x = *reinterpret_cast<const float2*>(pr + Rec::coef + 2 * i);
                            c[i][0] = x.x;
                            c[i][FC - 1] = x.y;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 5; ++i) c[i][0] = pr[Rec::coef + i];
                    }
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const int kk = k1 + j * (K / J);
                        const float w1 = pr[Rec::a1 + kk];
                        const float dl1 = m1.x - static_cast<float>(kk), q1 = fmaf(dl1, dl1, -m1.y);
                        float P = w1, t1 = w1 * dl1, t2 = 0.f, t3 = w1 * q1;
                        if constexpr (D == 3) {
                            P = w1 * w2;
                            t1 = (w1 * dl1) * w2;
                            t2 = w1 * wd2;
                            t3 = fmaf(w1 * q1, w2, w1 * wq2);
                        }
#pragma unroll
                        for (int f = 0; f < FC; ++f) {
                            float sw = fmaf(c[2][f], t1, c[0][f] * P);
                            if constexpr (D == 3) sw = fmaf(c[3][f], t2, sw);
                            sw = fmaf(c[4][f], t3, sw);
                            const float sd = c[1][f] * P, sq = c[4][f] * P;
#pragma unroll
                            for (int k = 0; k < K; ++k)
                                acc[j][k][f] =
                                    fmaf(a0[k], sw, fmaf(a0[K + k], sd, fmaf(a0[2 * K + k], sq, acc[j][k][f])));
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    if (!in1[j]) continue;
                    const int32_t g1 = key[1] + k1 + j * (K / J);
#pragma unroll
                    for (int k = 0; k < K; ++k) {
                        const int32_t gk = g0 + k;
                        if (gk < 0 || gk > N) continue;
                        if (tiled) {
                            const int32_t e = (gk - lo[0]) + ext[0] * ((g1 - lo[1]) + ext[1] * (g2 - lo[2]));
#pragma unroll
                            for (int f = 0; f < FC; ++f) atomicAdd(tile + e * F + f0 + f, acc[j][k][f]);
                        } else {
                            float* e = gbase + rbf_row<D>(lv, tm, gk, g1, g2) * rs + f0;
                            if constexpr (VEC) {
                                red_add_v2(e, acc[j][k][0], acc[j][k][FC - 1]);
                            } else {
#pragma unroll
                                for (int f = 0; f < FC; ++f) red_add_f32(e + f, acc[j][k][f]);
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
    if (!tiled) return;
    for (int32_t r = t; r < static_cast<int32_t>(vol); r += kCellBlock) {
        const int32_t g0 = lo[0] + r % ext[0];
        const int32_t g1 = lo[1] + (r / ext[0]) % ext[1];
        const int32_t g2 = lo[2] + r / (ext[0] * ext[1]);
        float* e = gbase + rbf_row<D>(lv, tm, g0, g1, g2) * rs;
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
    constexpr int kSmem = kBoxFloats * static_cast<int>(sizeof(float));
    cudaError_t e = cudaFuncSetAttribute(rbf_fwd_box_kernel<D, R, FC, TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmem);
    if (e != cudaSuccess) return e;
    rbf_fwd_box_kernel<D, R, FC, TT><<<grid, kBlock, kSmem, s>>>(p);
    return cudaGetLastError();
}

template <int D, int R, typename TT>
cudaError_t pick_fwd(const FwdParams& p, int fc, cudaStream_t s) {
    return fc == 2 ? launch_fwd<D, R, 2, TT>(p, s) : launch_fwd<D, R, 1, TT>(p, s);
}

template <int D, int R, int FC, bool VEC>
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t s) {
    if (p.c.nlvl == 0) return cudaSuccess;
    constexpr int kSmem = cell_smem_bytes<D, 2 * R, FC>();
    cudaError_t e = cudaFuncSetAttribute(rbf_bwd_cells_kernel<D, R, FC, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>((p.c.n + kCellBlock - 1) / kCellBlock), static_cast<unsigned>(p.c.nlvl));
    rbf_bwd_cells_kernel<D, R, FC, VEC><<<grid, kCellBlock, kSmem, s>>>(p);
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
