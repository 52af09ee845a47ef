// d-linear (Instant-NGP) encoding, forward and backward, and the
// vertex-index kernel.
//
// "SIGGRAPH 2022｜InstantNGP 与多分辨率哈希编码", 流程与原理 steps 1-3: the
// cell's 2^d corners are looked up (one-to-one at coarse levels, hashed at
// fine ones) and their F-dimensional features blended with d-linear weights
// prod_i (v_i ? t_i : 1 - t_i).  The backward scatters g_gamma * w_v.
#include <cuda_runtime.h>

#include "hg_device.cuh"

namespace hg {
namespace {

constexpr int kBlock = 256;

// VEC: FC == 2 and the row's pair is 8-byte (f32) / 4-byte (f16) aligned.
template <int D, int FC, typename TT, bool VEC>
__global__ void __launch_bounds__(kBlock) linear_fwd_kernel(const __grid_constant__ FwdParams p) {
    constexpr int V = 1 << D;
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];
    const bool active = (p.c.level_mask >> l) & 1u;

    uint32_t c[D];
    float t[D];
#pragma unroll
    for (int i = 0; i < D; ++i) locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
    uint32_t idx[V];
    float w[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        uint32_t g[D];
#pragma unroll
        for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
        idx[v] = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
        w[v] = corner_weight<D>(t, v);
    }
    const TT* base = static_cast<const TT*>(p.tab.ptr[0]) + l * p.tab.ls[0];
    for (int f0 = 0; f0 < F; f0 += FC) {
        float acc[FC];
#pragma unroll
        for (int f = 0; f < FC; ++f) acc[f] = 0.f;
        if (active) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const TT* e = base + static_cast<int64_t>(idx[v]) * p.tab.rs[0] + f0;
                float val[FC];
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
#pragma unroll
                for (int f = 0; f < FC; ++f) acc[f] = fmaf(w[v], val[f], acc[f]);
            }
        }
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
            __stcs(p.gamma + n * p.c.sn + lf * p.c.sf, acc[f]);
        }
    }
}

template <int D, int FC, bool VEC>
__global__ void __launch_bounds__(kBlock) linear_bwd_kernel(const __grid_constant__ BwdParams p) {
    constexpr int V = 1 << D;
    const int l = p.c.lvl[blockIdx.y];
    if (!((p.c.level_mask >> l) & 1u)) return;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int F = p.c.F;
    const Level& lv = p.c.lv[l];

    uint32_t c[D];
    float t[D];
#pragma unroll
    for (int i = 0; i < D; ++i) locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
    float* base = p.grad.ptr[0] + l * p.grad.ls[0];
    for (int f0 = 0; f0 < F; f0 += FC) {
        float up[FC];
#pragma unroll
        for (int f = 0; f < FC; ++f) {
            const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
            up[f] = __ldcs(p.g_gamma + n * p.c.sn + lf * p.c.sf);
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
            uint32_t g[D];
#pragma unroll
            for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
            const uint32_t id = vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0]);
            const float w = corner_weight<D>(t, v);
            float* e = base + static_cast<int64_t>(id) * p.grad.rs[0] + f0;
            if constexpr (VEC) {
                red_add_v2(e, w * up[0], w * up[FC - 1]);
            } else {
#pragma unroll
                for (int f = 0; f < FC; ++f) red_add_f32(e + f, w * up[f]);
            }
        }
    }
}

constexpr int kPrivBlock = 512;

// Privatised d-linear backward for small one-to-one levels (see the Hermite
// version): a CTA accumulates a chunk of points into a shared-memory copy of
// the level's gradient rows, then adds each row that received anything into
// the table.
template <int D, int FC>
__global__ void __launch_bounds__(kPrivBlock) linear_bwd_priv_kernel(const __grid_constant__ BwdParams p) {
    constexpr int V = 1 << D;
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
        uint32_t c[D];
        float t[D];
#pragma unroll
        for (int i = 0; i < D; ++i) locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
        for (int f0 = 0; f0 < F; f0 += FC) {
            float up[FC];
#pragma unroll
            for (int f = 0; f < FC; ++f) {
                const int64_t lf = static_cast<int64_t>(l) * F + f0 + f;
                up[f] = __ldg(p.g_gamma + n * p.c.sn + lf * p.c.sf);
            }
#pragma unroll
            for (int v = 0; v < V; ++v) {
                uint32_t g[D];
#pragma unroll
                for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
                const float w = corner_weight<D>(t, v);
                float* a = sacc + vertex_index<D>(g, lv, true, 0u) * F + f0;
#pragma unroll
                for (int f = 0; f < FC; ++f) atomicAdd(a + f, w * up[f]);
            }
        }
    }
    __syncthreads();
    float* base = p.grad.ptr[0] + l * p.grad.ls[0];
    for (uint32_t i = threadIdx.x; i < vals; i += kPrivBlock) {
        const float a = sacc[i];
        if (a != 0.f) red_add_f32(base + static_cast<int64_t>(i / F) * p.grad.rs[0] + i % F, a);
    }
}

template <int D, int FC>
cudaError_t launch_priv(const BwdParams& p, cudaStream_t s) {
    if (p.priv.n == 0) return cudaSuccess;
    if (p.priv.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(linear_bwd_priv_kernel<D, FC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             p.priv.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(static_cast<unsigned>((p.c.n + p.priv.chunk - 1) / p.priv.chunk), static_cast<unsigned>(p.priv.n));
    linear_bwd_priv_kernel<D, FC><<<grid, kPrivBlock, p.priv.smem_bytes, s>>>(p);
    return cudaGetLastError();
}

__global__ void __launch_bounds__(kBlock) indices_kernel(const __grid_constant__ IdxParams p) {
    const int l = p.c.lvl[blockIdx.y];
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (n >= p.c.n) return;
    const int d = p.c.d;
    const Level& lv = p.c.lv[l];
    const int V = 1 << d;
    uint32_t c[4];
    float t[4];
    for (int i = 0; i < d; ++i) locate(p.coords[n * d + i], lv, c[i], t[i]);
    uint32_t* out = p.idx + (n * p.c.L + l) * static_cast<int64_t>((d + 1) * V);
    for (int k = 0; k <= d; ++k) {
        for (int v = 0; v < V; ++v) {
            uint32_t id;
            if (d == 2) {
                const uint32_t g[2] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u)};
                id = vertex_index<2>(g, lv, (lv.dense >> k) & 1u, p.c.tmask[k]);
            } else if (d == 3) {
                const uint32_t g[3] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u)};
                id = vertex_index<3>(g, lv, (lv.dense >> k) & 1u, p.c.tmask[k]);
            } else {
                const uint32_t g[4] = {c[0] + (v & 1u), c[1] + ((v >> 1) & 1u), c[2] + ((v >> 2) & 1u),
                                       c[3] + ((v >> 3) & 1u)};
                id = vertex_index<4>(g, lv, (lv.dense >> k) & 1u, p.c.tmask[k]);
            }
            out[k * V + v] = id;
        }
    }
}

template <int D, int FC, typename TT, bool VEC>
cudaError_t launch_fwd(const FwdParams& p, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    linear_fwd_kernel<D, FC, TT, VEC><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, typename TT>
cudaError_t pick_fwd(const FwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (fc == 2) return vec ? launch_fwd<D, 2, TT, true>(p, s) : launch_fwd<D, 2, TT, false>(p, s);
    return launch_fwd<D, 1, TT, false>(p, s);
}

template <int D, int FC, bool VEC>
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t s) {
    cudaError_t e = launch_priv<D, FC>(p, s);
    if (e != cudaSuccess || p.c.nlvl == 0) return e;
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    linear_bwd_kernel<D, FC, VEC><<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t pick_bwd(const BwdParams& p, int fc, bool vec, cudaStream_t s) {
    if (fc == 2) return vec ? launch_bwd<D, 2, true>(p, s) : launch_bwd<D, 2, false>(p, s);
    return launch_bwd<D, 1, false>(p, s);
}

}  // namespace

int launch_linear_fwd(const FwdParams& p, int fc, bool vec, int dtype, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.c.d == 2) return dtype == HG_F16 ? pick_fwd<2, __half>(p, fc, vec, s) : pick_fwd<2, float>(p, fc, vec, s);
    if (p.c.d == 4) return dtype == HG_F16 ? pick_fwd<4, __half>(p, fc, vec, s) : pick_fwd<4, float>(p, fc, vec, s);
    return dtype == HG_F16 ? pick_fwd<3, __half>(p, fc, vec, s) : pick_fwd<3, float>(p, fc, vec, s);
}

int launch_linear_bwd(const BwdParams& p, int fc, bool vec, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.c.d == 4) return pick_bwd<4>(p, fc, vec, s);
    return p.c.d == 2 ? pick_bwd<2>(p, fc, vec, s) : pick_bwd<3>(p, fc, vec, s);
}

int launch_indices(const IdxParams& p, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    dim3 grid(static_cast<unsigned>((p.c.n + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    indices_kernel<<<grid, kBlock, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace hg
