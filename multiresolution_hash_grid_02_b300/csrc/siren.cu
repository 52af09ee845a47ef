// SIREN chain-rule consumer of the multiresolution encoding: forward and backward.
//
// "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs", 整体框架
// and 关键设计 2: the encoding's outputs gamma, grad gamma and lap gamma feed a
// SIREN, u = W2 sin(omega z) + b2 with z = W1 gamma + b1, and the chain rule
// with sigma'' = -omega^2 sigma gives, in one pass,
//   d u / d x_i = W2 [omega cos(omega z) * y_i],          y_i = W1 d gamma / d x_i,
//   lap u       = W2 [omega cos(omega z) * s - omega^2 sin(omega z) * sum_i y_i^2],  s = W1 lap gamma.
// The backward is the vector-Jacobian product to the encoder outputs (what
// the encoding's backward takes) and to the weights.
//
// Design: FP32 FMA on the CUDA cores.  The first layer contracts the d + 2
// input rows of a point (K = L F features each) with W1: small K, and with
// omega = 30 magnifying the rounding of z thirtyfold, too precision-sensitive
// for tf32 or bf16 tensor cores.  A CTA of 256 threads takes a tile of `pts`
// points staged in shared memory; tp = H / 16 threads share a point, each
// owning 16 hidden units, so every weight read from shared memory feeds d + 2
// FMAs (the backward: 512 threads of 8 units).  CTAs are persistent (one wave): the weights are staged once per CTA
// and the weight gradients are added to global memory once per CTA.
#include <cuda_runtime.h>

#include "hermite_blend.cuh"
#include "hg_device.cuh"
#include "hg_params.h"
#include "siren_tc.cuh"

namespace hg {
namespace {

constexpr int kThreads = 256;
constexpr int kUnits = 16;  // hidden units per thread
constexpr int kMaxO = 4;

// Shared-memory layout of a CTA, in floats; every region starts on 16 bytes.
struct SirenSmem {
    int w1t, b1, w2, b2, x, w1, g, gw2, gb1, gb2, total;
};

__host__ __device__ inline int take(int& at, int n) {
    const int here = at;
    at += (n + 3) & ~3;
    return here;
}

__host__ __device__ inline SirenSmem siren_layout(const SirenParams& p, bool bwd) {
    const int R = p.d + 2;
    SirenSmem m;
    int at = 0;
    m.w1t = take(at, p.K * p.H);             // W1 transposed, [K][H]: the forward contraction
    m.b1 = take(at, p.H);
    m.w2 = take(at, p.O * p.H);
    m.b2 = take(at, p.O);
    m.x = take(at, p.nbuf * R * p.pts * (p.K + 4));  // inputs [nbuf][R][pts][K + 4] (padding: no bank conflicts)
    if (bwd) {
        m.w1 = take(at, p.H * p.K);          // W1 as given, [H][K]: the input gradients
        // pre-activation gradients [R][pts][H + 4]; after the last tile the CTA's W1 gradient [H][K]
        m.g = take(at, max(R * p.pts * (p.H + 4), p.H * p.K));
        m.gw2 = take(at, p.O * p.H);
        m.gb1 = take(at, p.H);
        m.gb2 = take(at, p.O);
    } else {
        m.w1 = m.g = m.gw2 = m.gb1 = m.gb2 = -1;
    }
    m.total = at;
    return m;
}

// Weights into shared memory (W1 transposed for the forward contraction).
__device__ void stage_weights(const SirenParams& p, const SirenSmem& L, float* sm, bool bwd, int nt = kThreads) {
    for (int i = threadIdx.x; i < p.H * p.K; i += nt) {
        const float w = __ldg(p.W1 + i);
        sm[L.w1t + (i % p.K) * p.H + i / p.K] = w;
        if (bwd) sm[L.w1 + i] = w;
    }
    for (int i = threadIdx.x; i < p.H; i += nt) sm[L.b1 + i] = __ldg(p.b1 + i);
    for (int i = threadIdx.x; i < p.O * p.H; i += nt) sm[L.w2 + i] = __ldg(p.W2 + i);
    for (int i = threadIdx.x; i < p.O; i += nt) sm[L.b2 + i] = p.b2 ? __ldg(p.b2 + i) : 0.f;
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool valid) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 4 : 0) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Issue the asynchronous copy of a tile's input rows into X, [R][pts][K + 4];
// points past n and NULL rows are zero-filled.  A thread takes four
// consecutive features of one point (lanes: consecutive points, so the reads
// are coalesced).
__device__ void issue_tile(const SirenParams& p, float* X, int64_t n0, int R, int nt = kThreads) {
    const int P = p.pts, K4 = p.K / 4;
    const int total = R * K4 * P;
    for (int i = threadIdx.x; i < total; i += nt) {
        const int pp = i & (P - 1), rk = i / P;  // P is a power of two
        const int k = 4 * (rk % K4), r = rk / K4;
        const int64_t n = n0 + pp;
        const float* src = p.in[r];
        const bool ok = src && n < p.n;
        const float* e = ok ? src + k * p.n + n : p.W1;  // nothing is read when !ok (zero fill)
        float* d = X + (r * P + pp) * (p.K + 4) + k;
#pragma unroll
        for (int c = 0; c < 4; ++c) cp_async4(d + c, ok ? e + c * p.n : e, ok);
    }
}

// Hidden unit of a thread's slot jj: thread q of a point owns j = 4 q + 4 tp t + e
// (jj = 4 t + e), so the four weight vectors a thread loads for one feature lie
// in different banks from those of the point's other threads.
__device__ __forceinline__ int unit_of(int q, int tp, int jj) { return 4 * q + 4 * tp * (jj >> 2) + (jj & 3); }

__device__ __forceinline__ float lane4(const float4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// First layer for the thread's point (row pl of the tile) and its units:
// acc[r][jj] = sum_k W1[unit_of(q, tp, jj)][k] X[r][pl][k], k ascending.  The
// contraction runs on f32x2 pairs of units (two round-to-nearest FMAs per
// instruction, the same sums), which halves the issued FMA instructions.
template <int R, int U = kUnits>
__device__ __forceinline__ void first_layer(const float* W1T, const float* X, int K, int H, int P, int pl, int q,
                                            int tp, float (&acc)[R][U]) {
    uint64_t a2[R][U / 2];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < U / 2; ++e) a2[r][e] = 0;
    const int ld = K + 4;
    const float* xp = X + pl * ld;
    for (int k = 0; k < K; k += 4) {
        float4 xr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) xr[r] = *reinterpret_cast<const float4*>(xp + r * P * ld + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float* wrow = W1T + (k + kk) * H + 4 * q;
            uint64_t w[U / 2];
#pragma unroll
            for (int v = 0; v < U / 4; ++v) {
                const float4 wq = *reinterpret_cast<const float4*>(wrow + 4 * tp * v);
                w[2 * v] = f2_pack(wq.x, wq.y);
                w[2 * v + 1] = f2_pack(wq.z, wq.w);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint64_t xv = f2_dup(lane4(xr[r], kk));
#pragma unroll
                for (int e = 0; e < U / 2; ++e) a2[r][e] = f2_fma(w[e], xv, a2[r][e]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < U / 2; ++e) f2_unpack(a2[r][e], acc[r][2 * e], acc[r][2 * e + 1]);
}

// The forward of one staged tile X ([R][pts][K + 4]) for the thread's point
// (row pl) and units: the first layer, then u, grad u and lap u reduced over
// the point's tp threads; the point's first thread stores them.
template <int D>
__device__ __forceinline__ void siren_tile_fwd(const SirenParams& p, const float* W1T, const float* b1,
                                               const float* W2, const float* b2, const float* X, int64_t n0, int pl,
                                               int q) {
    constexpr int R = D + 2;
    const int tp = p.tp, P = p.pts, H = p.H, O = p.O;
    const float om = p.omega, om2 = om * om;
    float acc[R][kUnits];
    first_layer<R>(W1T, X, p.K, H, P, pl, q, tp, acc);
    float pu[kMaxO], pdu[D][kMaxO], plap[kMaxO];
#pragma unroll
    for (int o = 0; o < kMaxO; ++o) {
        pu[o] = plap[o] = 0.f;
#pragma unroll
        for (int i = 0; i < D; ++i) pdu[i][o] = 0.f;
    }
#pragma unroll
    for (int jj = 0; jj < kUnits; ++jj) {
        const int j = unit_of(q, tp, jj);
        float a, c;
        sincosf(om * (acc[0][jj] + b1[j]), &a, &c);
        float y2 = 0.f;
#pragma unroll
        for (int i = 0; i < D; ++i) y2 = fmaf(acc[1 + i][jj], acc[1 + i][jj], y2);
        const float oc = om * c;
        const float tl = fmaf(oc, acc[R - 1][jj], -om2 * a * y2);  // omega c s - omega^2 a sum y^2
#pragma unroll
        for (int o = 0; o < kMaxO; ++o) {
            if (o < O) {
                const float w2 = W2[o * H + j];
                pu[o] = fmaf(w2, a, pu[o]);
#pragma unroll
                for (int i = 0; i < D; ++i) pdu[i][o] = fmaf(w2, oc * acc[1 + i][jj], pdu[i][o]);
                plap[o] = fmaf(w2, tl, plap[o]);
            }
        }
    }
    // sum over the tp threads of the point (consecutive lanes)
    for (int m = 1; m < tp; m <<= 1) {
#pragma unroll
        for (int o = 0; o < kMaxO; ++o) {
            pu[o] += __shfl_xor_sync(0xffffffffu, pu[o], m);
            plap[o] += __shfl_xor_sync(0xffffffffu, plap[o], m);
#pragma unroll
            for (int i = 0; i < D; ++i) pdu[i][o] += __shfl_xor_sync(0xffffffffu, pdu[i][o], m);
        }
    }
    const int64_t n = n0 + pl;
    if (q == 0 && n < p.n) {
#pragma unroll
        for (int o = 0; o < kMaxO; ++o) {
            if (o < O) {
                if (p.u) __stcs(p.u + o * p.n + n, pu[o] + b2[o]);
                if (p.du) {
#pragma unroll
                    for (int i = 0; i < D; ++i) __stcs(p.du + (static_cast<int64_t>(i) * O + o) * p.n + n, pdu[i][o]);
                }
                if (p.lapu) __stcs(p.lapu + o * p.n + n, plap[o]);
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) siren_fwd_kernel(const __grid_constant__ SirenParams p) {
    constexpr int R = D + 2;
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    const SirenSmem L = siren_layout(p, false);
    stage_weights(p, L, sm, false);
    const int tp = p.tp, P = p.pts;
    float* Xb[2] = {sm + L.x, sm + L.x + (p.nbuf - 1) * R * P * (p.K + 4)};
    const int pl = threadIdx.x / tp, q = threadIdx.x % tp;
    const int64_t tiles = (p.n + P - 1) / P;
    int cur = 0;
    if (static_cast<int64_t>(blockIdx.x) < tiles) issue_tile(p, Xb[0], static_cast<int64_t>(blockIdx.x) * P, R);
    cp_async_commit();
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t tn = t + gridDim.x;
        if (p.nbuf == 2) {  // the next tile's copy flies while this one computes
            if (tn < tiles) issue_tile(p, Xb[cur ^ 1], tn * P, R);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // this tile (and the weights) visible to every thread
        siren_tile_fwd<D>(p, sm + L.w1t, sm + L.b1, sm + L.w2, sm + L.b2, Xb[cur], t * P, pl, q);
        __syncthreads();  // this tile's buffer read by every thread
        if (p.nbuf == 1 && tn < tiles) {
            issue_tile(p, Xb[0], tn * P, R);
            cp_async_commit();
        }
        cur ^= p.nbuf - 1;
    }
    cp_async_wait<0>();
}

// Fused encoder + SIREN forward ("Hermite-NGP", 整体框架: the encoding feeds
// the network directly).  Instead of reading gamma, grad gamma and lap gamma
// back from global memory, each tile's inputs are computed in place: the
// CTA's threads encode (point, level) items of the tile -- the 2^d corner
// rows of a packed F = 2 table read whole, the one-thread separable blend --
// and write each level's two features into the shared-memory tile at
// columns 2 l, 2 l + 1 (inactive levels and points past n as zeros), then
// the tile's SIREN forward runs as in siren_fwd_kernel.  The encoder outputs
// never leave the chip; with all levels' tables resident in L2 (the 2D PINN
// grid: ~60 MB) the gathers stay on chip too.  One input buffer; the CTAs on
// an SM (two) overlap one another's encode and contraction.
template <int D, typename TT>
__global__ void __launch_bounds__(kThreads, 2) encode_siren_fwd_kernel(const __grid_constant__ SirenParams p,
                                                                      const __grid_constant__ FwdParams e) {
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    const SirenSmem L = siren_layout(p, false);
    stage_weights(p, L, sm, false);
    const int tp = p.tp, P = p.pts, ld = p.K + 4, levels = e.c.L;
    float* X = sm + L.x;
    const int pl = threadIdx.x / tp, q = threadIdx.x % tp;
    const int64_t tiles = (p.n + P - 1) / P;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t n0 = t * P;
        for (int i = threadIdx.x; i < P * levels; i += kThreads) {
            const int pp = i & (P - 1), l = i / P;  // P is a power of two
            const int64_t n = n0 + pp;
            float g[2] = {0.f, 0.f}, dg[2][3] = {{0.f, 0.f, 0.f}, {0.f, 0.f, 0.f}}, lp[2] = {0.f, 0.f};
            if (n < e.c.n && ((e.c.level_mask >> l) & 1u)) encode_item_f2<D, TT>(e, n, l, g, dg, lp);
            float* x = X + pp * ld + 2 * l;
            *reinterpret_cast<float2*>(x) = make_float2(g[0], g[1]);
#pragma unroll
            for (int j = 0; j < D; ++j)
                *reinterpret_cast<float2*>(x + (1 + j) * P * ld) = make_float2(dg[0][j], dg[1][j]);
            *reinterpret_cast<float2*>(x + (D + 1) * P * ld) = make_float2(lp[0], lp[1]);
        }
        __syncthreads();  // the tile (and the weights) visible to every thread
        siren_tile_fwd<D>(p, sm + L.w1t, sm + L.b1, sm + L.w2, sm + L.b2, X, n0, pl, q);
        __syncthreads();  // every thread done with the tile before the next encode
    }
}

// ---------------------------------------------------------------------------
// Tensor-core forward (tcgen05, split tf32; see siren_tc.cuh).  A CTA of 512
// threads takes tiles of 128 points: the tile's inputs (the encoder's
// feature-major outputs) are split into tf32 hi/lo parts in shared memory;
// one thread issues, for every input row r, the three products of
// Z_r = X_r W1^T (K / 8 MMAs of 128 x H x 8 each) into TMEM columns
// [r H, (r+1) H); then each thread reads its point's row of Z (TMEM lane =
// point; the four warps of a lane quadrant take one quarter of the hidden
// units each) and forms u, grad u and lap u as the CUDA-core forward does.
// One CTA per SM (the split operands take ~180 KB for d = 3, K = 32); the
// staging loads are issued in batches so several are in flight per thread.
// Measured (2^21 points, K = 32, H = 64): 3D 1.45 ms against 1.62 ms on the
// CUDA cores; 2D 0.74 against 0.69 ms (fewer rows per point, so the
// staging, not the contraction, dominates) -- hence d >= 3 only.  Staging
// the raw tile with 4-byte cp.async copies during the previous epilogue was
// slower (1.76 ms), and so was encoding in place for the fused forward with
// one CTA per SM (7.6 against 3.3 ms: the gathers cannot be hidden).
// ---------------------------------------------------------------------------
constexpr int kTcPts = 128;
constexpr int kTcThreads = 512;
constexpr int kTcGroups = kTcThreads / kTcPts;  // warps per TMEM lane quadrant: unit groups
constexpr int kTcSpin = 1 << 20;  // polls of the completion barrier before giving up

struct TcLayout {
    int w, x, b1, w2, b2, red, total;  // byte offsets in dynamic shared memory
};

__host__ __device__ inline int tc_take(int& at, int bytes, int align) {
    at = (at + align - 1) / align * align;
    const int here = at;
    at += bytes;
    return here;
}

__host__ __device__ inline TcLayout tc_layout(const SirenParams& p) {
    const int R = p.d + 2;
    TcLayout t;
    int at = 0;
    t.w = tc_take(at, 2 * p.H * p.K * 4, 1024);           // W1 hi, lo: [H][K] core layout each
    t.x = tc_take(at, 2 * R * kTcPts * p.K * 4, 1024);     // X_r hi, lo: [128][K] core layout each
    t.b1 = tc_take(at, p.H * 4, 16);
    t.w2 = tc_take(at, p.O * p.H * 4, 16);
    t.b2 = tc_take(at, kMaxO * 4, 16);
    t.red = tc_take(at, (kTcGroups - 1) * kTcPts * kMaxO * (p.d + 2) * 4, 16);  // other groups' partial outputs
    t.total = at;
    return t;
}

__host__ __device__ inline uint32_t tc_cols(const SirenParams& p) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>((p.d + 2) * p.H)) c <<= 1;
    return c;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) siren_fwd_tc_kernel(const __grid_constant__ SirenParams p) {
    constexpr int R = D + 2;
    extern __shared__ __align__(1024) unsigned char tsm[];
    __shared__ __align__(8) uint64_t mbar;
    __shared__ uint32_t tslot;
    const TcLayout Lt = tc_layout(p);
    const int K = p.K, H = p.H, O = p.O;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* sw = tsm + Lt.w;
    unsigned char* sx = tsm + Lt.x;
    float* b1s = reinterpret_cast<float*>(tsm + Lt.b1);
    float* w2s = reinterpret_cast<float*>(tsm + Lt.w2);
    float* b2s = reinterpret_cast<float*>(tsm + Lt.b2);
    float* red = reinterpret_cast<float*>(tsm + Lt.red);
    const int wbytes = H * K * 4, xbytes = kTcPts * K * 4;
    for (int i = tid; i < H * K; i += kTcThreads) {
        float hi, lo;
        tc::split_tf32(__ldg(p.W1 + i), hi, lo);
        const uint32_t o = tc::kmajor_off(i / K, i % K, K);
        *reinterpret_cast<float*>(sw + o) = hi;
        *reinterpret_cast<float*>(sw + wbytes + o) = lo;
    }
    for (int i = tid; i < H; i += kTcThreads) b1s[i] = __ldg(p.b1 + i);
    for (int i = tid; i < O * H; i += kTcThreads) w2s[i] = __ldg(p.W2 + i);
    for (int i = tid; i < kMaxO; i += kTcThreads) b2s[i] = (p.b2 && i < O) ? __ldg(p.b2 + i) : 0.f;
    if (tid == 0) tc::mbar_init(&mbar, 1);
    const uint32_t cols = tc_cols(p);
    if (warp == 0) tc::tmem_alloc(&tslot, cols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = tslot;
    const uint32_t idesc = tc::idesc_tf32(H);
    const uint32_t lbo = 128, sbo = static_cast<uint32_t>(K / 4) * 128;
    const float om = p.omega, om2 = om * om;
    const int64_t tiles = (p.n + kTcPts - 1) / kTcPts;
    uint32_t phase = 0;
    int64_t failed = -1;  // the tile whose products did not complete in time
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t n0 = t * kTcPts;
        // (1) the tile's inputs, split, into the operand layout (points past n: zeros); the loads of
        // B items are issued together, so several are in flight per thread
        {
            constexpr int B = 4;
            const int K4 = K / 4, total = R * K4 * kTcPts;
            for (int i0 = tid; i0 < total; i0 += B * kTcThreads) {
                float v[B][4];
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const int i = i0 + b * kTcThreads;
                    const int m = i & (kTcPts - 1), rc = i / kTcPts;
                    const int c = rc % K4, r = rc / K4;
                    const int64_t n = n0 + m;
                    const float* src = i < total ? p.in[r] : nullptr;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        v[b][q] = (src && n < p.n) ? __ldg(src + static_cast<int64_t>(4 * c + q) * p.n + n) : 0.f;
                }
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const int i = i0 + b * kTcThreads;
                    if (i >= total) break;
                    const int m = i & (kTcPts - 1), rc = i / kTcPts;
                    const int c = rc % K4, r = rc / K4;
                    float4 hi, lo;
                    tc::split_tf32(v[b][0], hi.x, lo.x);
                    tc::split_tf32(v[b][1], hi.y, lo.y);
                    tc::split_tf32(v[b][2], hi.z, lo.z);
                    tc::split_tf32(v[b][3], hi.w, lo.w);
                    const uint32_t o = tc::kmajor_off(m, 4 * c, K);
                    *reinterpret_cast<float4*>(sx + (2 * r) * xbytes + o) = hi;
                    *reinterpret_cast<float4*>(sx + (2 * r + 1) * xbytes + o) = lo;
                }
            }
        }
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // (2) Z_r = X_r W1^T for every row: hi*hi, hi*lo, lo*hi
        if (tid == 0) {
            for (int r = 0; r < R; ++r) {
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t xa = tc::smem_u32(sx + (2 * r + (pass == 2 ? 1 : 0)) * xbytes);
                    const uint32_t wb = tc::smem_u32(sw + (pass == 1 ? wbytes : 0));
                    for (int s = 0; s < K / 8; ++s)
                        tc::mma_tf32(tmem + static_cast<uint32_t>(r * H), tc::desc(xa + s * 256, lbo, sbo),
                                     tc::desc(wb + s * 256, lbo, sbo), idesc, pass > 0 || s > 0);
                }
            }
            tc::commit(&mbar);
        }
        const bool done = tc::mbar_wait(&mbar, phase, kTcSpin);
        phase ^= 1u;
        if (__syncthreads_or(!done)) {
            failed = t;
            break;
        }
        tc::fence_after();
        // (3) epilogue: the thread's point is TMEM lane 32 (warp % 4) + lane; its group's quarter of the units
        const int quad = warp & 3, grp = warp >> 2, m = quad * 32 + lane;
        const uint32_t lbase = tmem + ((static_cast<uint32_t>(quad) * 32u) << 16);
        float pu[kMaxO], pdu[D][kMaxO], plap[kMaxO];
#pragma unroll
        for (int o = 0; o < kMaxO; ++o) {
            pu[o] = plap[o] = 0.f;
#pragma unroll
            for (int i = 0; i < D; ++i) pdu[i][o] = 0.f;
        }
        const int hq = H / kTcGroups;
        for (int j0 = grp * hq; j0 < (grp + 1) * hq; j0 += 16) {
            uint32_t zr[R][16];
#pragma unroll
            for (int r = 0; r < R; ++r) tc::tmem_ld16_async(lbase + static_cast<uint32_t>(r * H + j0), zr[r]);
            tc::tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int j = j0 + jj;
                float a, c;
                sincosf(om * (__uint_as_float(zr[0][jj]) + b1s[j]), &a, &c);
                float y2 = 0.f;
#pragma unroll
                for (int i = 0; i < D; ++i) y2 = fmaf(__uint_as_float(zr[1 + i][jj]), __uint_as_float(zr[1 + i][jj]), y2);
                const float oc = om * c;
                const float tl = fmaf(oc, __uint_as_float(zr[R - 1][jj]), -om2 * a * y2);
#pragma unroll
                for (int o = 0; o < kMaxO; ++o) {
                    if (o < O) {
                        const float w2 = w2s[o * H + j];
                        pu[o] = fmaf(w2, a, pu[o]);
#pragma unroll
                        for (int i = 0; i < D; ++i) pdu[i][o] = fmaf(w2, oc * __uint_as_float(zr[1 + i][jj]), pdu[i][o]);
                        plap[o] = fmaf(w2, tl, plap[o]);
                    }
                }
            }
        }
        // the other groups' partial sums to group 0, which stores the point's outputs (groups in order)
        if (grp > 0) {
            float* rp = red + ((grp - 1) * kTcPts + m) * (kMaxO * R);
#pragma unroll
            for (int o = 0; o < kMaxO; ++o) {
                rp[o * R] = pu[o];
                rp[o * R + 1] = plap[o];
#pragma unroll
                for (int i = 0; i < D; ++i) rp[o * R + 2 + i] = pdu[i][o];
            }
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        const int64_t n = n0 + m;
        if (grp == 0 && n < p.n) {
#pragma unroll
            for (int g = 0; g < kTcGroups - 1; ++g) {
                const float* rp = red + (g * kTcPts + m) * (kMaxO * R);
#pragma unroll
                for (int o = 0; o < kMaxO; ++o) {
                    pu[o] += rp[o * R];
                    plap[o] += rp[o * R + 1];
#pragma unroll
                    for (int i = 0; i < D; ++i) pdu[i][o] += rp[o * R + 2 + i];
                }
            }
#pragma unroll
            for (int o = 0; o < kMaxO; ++o) {
                if (o < O) {
                    if (p.u) __stcs(p.u + o * p.n + n, pu[o] + b2s[o]);
                    if (p.du) {
#pragma unroll
                        for (int i = 0; i < D; ++i) __stcs(p.du + (static_cast<int64_t>(i) * O + o) * p.n + n, pdu[i][o]);
                    }
                    if (p.lapu) __stcs(p.lapu + o * p.n + n, plap[o]);
                }
            }
        }
        __syncthreads();  // the reduction buffer and the operands are free for the next tile
    }
    if (failed >= 0) {
        // the products did not complete in time: mark the tile's outputs invalid (NaN), give the tensor
        // core a bounded while longer to finish before the accumulator memory is released
        (void)tc::mbar_wait(&mbar, phase ^ 1u, kTcSpin);
        if (tid < kTcPts) {
            const int64_t n = failed * kTcPts + tid;
            if (n < p.n && p.u) p.u[n] = __int_as_float(0x7fc00000);
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_free(tmem, cols);
}

// Backward.  Per tile: (1) recompute the first layer, form the pre-activation
// gradients g_z = d/dz, g_y_i = d/dy_i, g_s = d/ds of the thread's units into
// shared memory ([R][pts][H + 4]; rows z, y_1 .. y_d, s), and sum the
// output-layer and bias gradients over the warp's points; (2) input gradients
// g_in[r][k] = sum_j W1[j][k] G[r][j] per point, four features per thread at
// a time; (3) first-layer weight gradient gW1[j][k] += sum_{r, point}
// G[r][j] X[r][k]: each 4 x 4 block of it is owned by `groups` threads, each
// summing a share of the tile's R * pts rows into registers that persist
// across the CTA's tiles, and the blocks are summed in shared memory and
// added to global memory once per CTA.
// 512 threads, 8 hidden units each (tp = H / 8): 16 warps per SM at one CTA
// per SM (the tiles' shared memory allows one) against 8 with 256 threads of
// 16 units, whose 231 registers also allowed no more.
constexpr int kBwdThreads = 512;
constexpr int kBwdUnits = 8;

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) siren_bwd_kernel(const __grid_constant__ SirenParams p) {
    constexpr int R = D + 2, U = kBwdUnits, NT = kBwdThreads;
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    const SirenSmem L = siren_layout(p, true);
    stage_weights(p, L, sm, true, NT);
    for (int i = threadIdx.x; i < p.O * p.H; i += NT) sm[L.gw2 + i] = 0.f;
    for (int i = threadIdx.x; i < p.H; i += NT) sm[L.gb1 + i] = 0.f;
    for (int i = threadIdx.x; i < p.O; i += NT) sm[L.gb2 + i] = 0.f;
    const float* W1T = sm + L.w1t;
    const float* W1 = sm + L.w1;
    const float* b1 = sm + L.b1;
    const float* W2 = sm + L.w2;
    float* G = sm + L.g;
    float* gW2s = sm + L.gw2;
    float* gb1s = sm + L.gb1;
    float* gb2s = sm + L.gb2;
    const int tp = p.tp, P = p.pts, H = p.H, K = p.K, O = p.O;
    float* Xb[2] = {sm + L.x, sm + L.x + (p.nbuf - 1) * R * P * (K + 4)};
    const int pl = threadIdx.x / tp, q = threadIdx.x % tp;
    const int lane = threadIdx.x & 31;
    const float om = p.omega, om2 = om * om;
    const int gld = H + 4, xld = K + 4;
    bool want_in = false;
#pragma unroll
    for (int r = 0; r < R; ++r) want_in = want_in || p.g_in[r];
    // first-layer weight-gradient ownership: block b (4 units x 4 features), group grp of `groups`
    const int nb = (H / 4) * (K / 4), groups = NT / nb;  // nb <= 512 (H <= 128, K <= 64)
    const int grp = threadIdx.x / nb, b = threadIdx.x % nb;
    const bool owner = p.gW1 && grp < groups;
    const int bj = 4 * (b / (K / 4)), bk = 4 * (b % (K / 4));
    const int rows = R * P, share = (rows + groups - 1) / groups;
    const int m0 = grp * share, m1 = min(rows, m0 + share);
    uint64_t a3[4][2] = {};  // the block's sums, f32x2 pairs over k
    const int64_t tiles = (p.n + P - 1) / P;
    int cur = 0;
    if (static_cast<int64_t>(blockIdx.x) < tiles) issue_tile(p, Xb[0], static_cast<int64_t>(blockIdx.x) * P, R, NT);
    cp_async_commit();
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t tn = t + gridDim.x;
        if (p.nbuf == 2) {  // the next tile's copy flies while this one computes
            if (tn < tiles) issue_tile(p, Xb[cur ^ 1], tn * P, R, NT);
            cp_async_commit();
        }
        const float* X = Xb[cur];
        const int64_t n0 = t * P;
        const int64_t n = n0 + pl;
        const bool have = n < p.n;
        float gu[kMaxO], gdu[D][kMaxO], glu[kMaxO];
#pragma unroll
        for (int o = 0; o < kMaxO; ++o) {
            const bool ok = have && o < O;
            gu[o] = (ok && p.g_u) ? __ldg(p.g_u + o * p.n + n) : 0.f;
            glu[o] = (ok && p.g_lapu) ? __ldg(p.g_lapu + o * p.n + n) : 0.f;
#pragma unroll
            for (int i = 0; i < D; ++i)
                gdu[i][o] = (ok && p.g_du) ? __ldg(p.g_du + (static_cast<int64_t>(i) * O + o) * p.n + n) : 0.f;
        }
        if (p.nbuf == 2)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        __syncthreads();  // this tile (and the weights) visible to every thread
        // (1) pre-activation gradients
        {
            float acc[R][U];
            first_layer<R, U>(W1T, X, K, H, P, pl, q, tp, acc);
            float* Gp = G + pl * gld;
#pragma unroll
            for (int jj = 0; jj < U; ++jj) {
                const int j = unit_of(q, tp, jj);
                float a, c;
                sincosf(om * (acc[0][jj] + b1[j]), &a, &c);
                const float oc = om * c, oa = om * a;
                float y2 = 0.f;
#pragma unroll
                for (int i = 0; i < D; ++i) y2 = fmaf(acc[1 + i][jj], acc[1 + i][jj], y2);
                const float s = acc[R - 1][jj];
                // adjoints of a, omega c y_i and the Laplacian's bracket through W2
                float Uo = 0.f, Pl = 0.f, Dv[D];
#pragma unroll
                for (int i = 0; i < D; ++i) Dv[i] = 0.f;
#pragma unroll
                for (int o = 0; o < kMaxO; ++o) {
                    if (o < O) {
                        const float w2 = W2[o * H + j];
                        Uo = fmaf(w2, gu[o], Uo);
                        Pl = fmaf(w2, glu[o], Pl);
#pragma unroll
                        for (int i = 0; i < D; ++i) Dv[i] = fmaf(w2, gdu[i][o], Dv[i]);
                    }
                }
                const float ga = fmaf(-om2 * Pl, y2, Uo);  // d/da
                float gc = Pl * s;                          // d/dc, over omega
#pragma unroll
                for (int i = 0; i < D; ++i) gc = fmaf(Dv[i], acc[1 + i][jj], gc);
                gc *= om;
                Gp[j] = fmaf(oc, ga, -oa * gc);  // d/dz: a = sin(omega z), c = cos(omega z)
#pragma unroll
                for (int i = 0; i < D; ++i)
                    Gp[(1 + i) * P * gld + j] = fmaf(oc, Dv[i], -2.f * om2 * a * Pl * acc[1 + i][jj]);
                Gp[(R - 1) * P * gld + j] = oc * Pl;
                // output-layer and bias gradients of unit j, summed over the warp's points
                if (p.gb1) {
                    float v = Gp[j];
                    for (int m = tp; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                    if (lane < tp) atomicAdd(gb1s + j, v);
                }
                if (p.gW2) {
                    const float tl = fmaf(oc, s, -om2 * a * y2);
#pragma unroll
                    for (int o = 0; o < kMaxO; ++o) {
                        if (o < O) {
                            float v = fmaf(glu[o], tl, gu[o] * a);
#pragma unroll
                            for (int i = 0; i < D; ++i) v = fmaf(gdu[i][o], oc * acc[1 + i][jj], v);
                            for (int m = tp; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                            if (lane < tp) atomicAdd(gW2s + o * H + j, v);
                        }
                    }
                }
            }
            if (p.gb2) {
#pragma unroll
                for (int o = 0; o < kMaxO; ++o) {
                    if (o < O) {
                        float v = q == 0 ? gu[o] : 0.f;
                        for (int m = 1; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
                        if (lane == 0) atomicAdd(gb2s + o, v);
                    }
                }
            }
        }
        __syncthreads();
        // (2) input gradients of the thread's point, 4 features at a time
        if (want_in) {
            for (int kc = 4 * q; kc < K; kc += 4 * tp) {
                uint64_t a2[R][2];  // f32x2 pairs of features
#pragma unroll
                for (int r = 0; r < R; ++r) a2[r][0] = a2[r][1] = 0;
                for (int j = 0; j < H; j += 4) {
                    float4 g4[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) g4[r] = *reinterpret_cast<const float4*>(G + (r * P + pl) * gld + j);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float4 wa = *reinterpret_cast<const float4*>(W1 + (j + jj) * K + kc);
                        const uint64_t w0 = f2_pack(wa.x, wa.y), w1 = f2_pack(wa.z, wa.w);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint64_t gv = f2_dup(lane4(g4[r], jj));
                            a2[r][0] = f2_fma(gv, w0, a2[r][0]);
                            a2[r][1] = f2_fma(gv, w1, a2[r][1]);
                        }
                    }
                }
                if (have) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        if (p.g_in[r]) {
                            float v[4];
                            f2_unpack(a2[r][0], v[0], v[1]);
                            f2_unpack(a2[r][1], v[2], v[3]);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) __stcs(p.g_in[r] + (kc + kk) * p.n + n, v[kk]);
                        }
                    }
                }
            }
        }
        // (3) first-layer weight gradient: this thread's block over its share of the tile's rows
        if (owner) {
            for (int m = m0; m < m1; ++m) {
                const float4 g4 = *reinterpret_cast<const float4*>(G + m * gld + bj);
                const float4 x4 = *reinterpret_cast<const float4*>(X + m * xld + bk);
                const uint64_t x01 = f2_pack(x4.x, x4.y), x23 = f2_pack(x4.z, x4.w);
#pragma unroll
                for (int aa = 0; aa < 4; ++aa) {
                    const uint64_t gv = f2_dup(lane4(g4, aa));
                    a3[aa][0] = f2_fma(gv, x01, a3[aa][0]);
                    a3[aa][1] = f2_fma(gv, x23, a3[aa][1]);
                }
            }
        }
        __syncthreads();  // this tile's X and G read by every thread
        if (p.nbuf == 1 && tn < tiles) {
            issue_tile(p, Xb[0], tn * P, R, NT);
            cp_async_commit();
        }
        cur ^= p.nbuf - 1;
    }
    cp_async_wait<0>();
    __syncthreads();
    // the CTA's weight gradients, added once; the groups' blocks are summed in the (now free) G region
    if (p.gW1) {
        float* gW1s = G;  // [H][K]
        for (int e = threadIdx.x; e < H * K; e += NT) gW1s[e] = 0.f;
        __syncthreads();
        if (owner) {
#pragma unroll
            for (int aa = 0; aa < 4; ++aa) {
                float v[4];
                f2_unpack(a3[aa][0], v[0], v[1]);
                f2_unpack(a3[aa][1], v[2], v[3]);
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) atomicAdd(gW1s + (bj + aa) * K + bk + bb, v[bb]);
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < H * K; e += NT) atomicAdd(p.gW1 + e, gW1s[e]);
    }
    if (p.gW2)
        for (int e = threadIdx.x; e < O * H; e += NT) atomicAdd(p.gW2 + e, gW2s[e]);
    if (p.gb1)
        for (int e = threadIdx.x; e < H; e += NT) atomicAdd(p.gb1 + e, gb1s[e]);
    if (p.gb2)
        for (int e = threadIdx.x; e < O; e += NT) atomicAdd(p.gb2 + e, gb2s[e]);
}

template <int D>
cudaError_t set_smem(bool bwd, size_t bytes) {
    return bwd ? cudaFuncSetAttribute(siren_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(bytes))
               : cudaFuncSetAttribute(siren_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(bytes));
}

template <int D>
cudaError_t occupancy(bool bwd, size_t bytes, int* blocks) {
    cudaError_t e = set_smem<D>(bwd, bytes);
    if (e != cudaSuccess) return e;
    return bwd ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, siren_bwd_kernel<D>, kBwdThreads, bytes)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, siren_fwd_kernel<D>, kThreads, bytes);
}

template <int D>
cudaError_t launch(const SirenParams& p, bool bwd, int ctas, cudaStream_t s) {
    const size_t bytes = siren_smem_bytes(p, bwd);
    cudaError_t e = set_smem<D>(bwd, bytes);
    if (e != cudaSuccess) return e;
    if (bwd)
        siren_bwd_kernel<D><<<ctas, kBwdThreads, bytes, s>>>(p);
    else
        siren_fwd_kernel<D><<<ctas, kThreads, bytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t dispatch(const SirenParams& p, bool bwd, int ctas, cudaStream_t s) {
    switch (p.d) {
        case 1: return launch<1>(p, bwd, ctas, s);
        case 2: return launch<2>(p, bwd, ctas, s);
        case 3: return launch<3>(p, bwd, ctas, s);
        default: return launch<4>(p, bwd, ctas, s);
    }
}

}  // namespace

void siren_bwd_tiles(SirenParams& p) {
    p.tp = p.H / kBwdUnits;
    p.pts = kBwdThreads / p.tp;
}

size_t siren_smem_bytes(const SirenParams& p, bool bwd) {
    return static_cast<size_t>(siren_layout(p, bwd).total) * sizeof(float);
}

int siren_ctas_per_sm(const SirenParams& p, bool bwd, int* ctas) {
    const size_t bytes = siren_smem_bytes(p, bwd);
    switch (p.d) {
        case 1: return occupancy<1>(bwd, bytes, ctas);
        case 2: return occupancy<2>(bwd, bytes, ctas);
        case 3: return occupancy<3>(bwd, bytes, ctas);
        default: return occupancy<4>(bwd, bytes, ctas);
    }
}

int launch_siren_fwd(const SirenParams& p, int ctas, void* stream) {
    return dispatch(p, false, ctas, static_cast<cudaStream_t>(stream));
}

int launch_siren_bwd(const SirenParams& p, int ctas, void* stream) {
    return dispatch(p, true, ctas, static_cast<cudaStream_t>(stream));
}

namespace {
template <int D, typename TT>
cudaError_t fused_attr(size_t bytes, int* per_sm, const SirenParams& p, const FwdParams& e, int ctas,
                       cudaStream_t s, bool launch) {
    cudaError_t err = cudaFuncSetAttribute(encode_siren_fwd_kernel<D, TT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(bytes));
    if (err != cudaSuccess) return err;
    if (!launch)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, encode_siren_fwd_kernel<D, TT>, kThreads, bytes);
    encode_siren_fwd_kernel<D, TT><<<ctas, kThreads, bytes, s>>>(p, e);
    return cudaGetLastError();
}

cudaError_t fused_dispatch(const SirenParams& p, const FwdParams& e, int dtype, int* per_sm, int ctas, cudaStream_t s,
                           bool launch) {
    const size_t bytes = siren_smem_bytes(p, false);
    if (p.d == 2)
        return dtype == HG_F16 ? fused_attr<2, __half>(bytes, per_sm, p, e, ctas, s, launch)
                               : fused_attr<2, float>(bytes, per_sm, p, e, ctas, s, launch);
    return dtype == HG_F16 ? fused_attr<3, __half>(bytes, per_sm, p, e, ctas, s, launch)
                           : fused_attr<3, float>(bytes, per_sm, p, e, ctas, s, launch);
}
}  // namespace

bool siren_tc_usable(const SirenParams& p, int smem_max) {
    return p.d >= 3 && p.H >= 16 * kTcGroups && (p.d + 2) * p.H <= 512 && p.K % 8 == 0 && p.O <= kMaxO &&
           tc_layout(p).total + 1024 <= smem_max;
}

namespace {
template <int D>
cudaError_t tc_launch(const SirenParams& p, cudaStream_t s) {
    const int bytes = tc_layout(p).total;
    cudaError_t err = cudaFuncSetAttribute(siren_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    const int64_t tiles = (p.n + kTcPts - 1) / kTcPts;
    const int ctas = static_cast<int>(tiles < sms ? tiles : sms);  // one CTA per SM (shared memory)
    siren_fwd_tc_kernel<D><<<ctas, kTcThreads, bytes, s>>>(p);
    return cudaGetLastError();
}
}  // namespace

int launch_siren_fwd_tc(const SirenParams& p, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return p.d == 3 ? tc_launch<3>(p, s) : tc_launch<4>(p, s);
}

int encode_siren_ctas_per_sm(const SirenParams& p, int dtype, int* ctas) {
    return fused_dispatch(p, FwdParams{}, dtype, ctas, 0, nullptr, false);
}

int launch_encode_siren_fwd(const SirenParams& p, const FwdParams& e, int dtype, int ctas, void* stream) {
    return fused_dispatch(p, e, dtype, nullptr, ctas, static_cast<cudaStream_t>(stream), true);
}

}  // namespace hg
