// Device helpers of the hash-grid kernels: cell location, vertex indexing,
// the cubic Hermite bases and the order-bucket slot tables.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "hg_params.h"

namespace hg {

// Spatial-hash multipliers, one per axis (the first is 1).
constexpr uint32_t kPrime1 = 2654435761u;
constexpr uint32_t kPrime2 = 805459861u;
constexpr uint32_t kPrime3 = 3674653429u;

// Clamp x to [0,1] (fmaxf maps NaN to 0), pos = fl32(x * N), cell index
// c = min(floor(pos), N-1) and local coordinate t = pos - c (exact in fp32).
__device__ __forceinline__ void locate(float x, const Level& lv, uint32_t& c, float& t) {
    x = fminf(fmaxf(x, 0.0f), 1.0f);
    const float pos = __fmul_rn(x, lv.fN);
    const uint32_t ci = min(static_cast<uint32_t>(pos), lv.N - 1u);
    c = ci;
    t = __fsub_rn(pos, static_cast<float>(ci));
}

// Index of vertex g in a table of mask+1 entries: one-to-one (axis 0
// fastest) when the level's grid fits, else XOR of g_i * prime_i mod T.
template <int D>
__device__ __forceinline__ uint32_t vertex_index(const uint32_t (&g)[D], const Level& lv, bool dense,
                                                 uint32_t tmask) {
    if (dense) {
        uint32_t i = g[0] + g[1] * lv.side;
        if constexpr (D >= 3) i += g[2] * lv.side2;
        if constexpr (D == 4) i += g[3] * lv.side3;
        return i;
    }
    uint32_t h = g[0] ^ (g[1] * kPrime1);
    if constexpr (D >= 3) h ^= g[2] * kPrime2;
    if constexpr (D == 4) h ^= g[3] * kPrime3;
    return h & tmask;
}

// Per-axis cubic Hermite weights of the two cell corners (v = 0 low side,
// v = 1 high side) for the value basis (a = 0) and the slope basis (a = 1),
// with the level's scale factors folded in:
//   w [v][a] = basis            * dx^a
//   d1[v][a] = d(basis)/dt * N  * dx^a     (d/dx)
//   d2[v][a] = d2(basis)/dt2*N^2* dx^a     (d2/dx2)
// (dx * N = 1 is used exactly for the slope basis.)
struct Basis1 {
    float w[2][2], d1[2][2], d2[2][2];
};

__device__ __forceinline__ Basis1 hermite_basis(float t, const Level& lv) {
    const float u = 1.0f - t;
    const float tu = t * u;
    Basis1 b;
    // value bases: (1-t)^2 (1+2t) and t^2 (3-2t)
    b.w[0][0] = u * u * fmaf(2.0f, t, 1.0f);
    b.w[1][0] = t * t * fmaf(-2.0f, t, 3.0f);
    b.d1[0][0] = -6.0f * tu * lv.fN;
    b.d1[1][0] = 6.0f * tu * lv.fN;
    b.d2[0][0] = fmaf(12.0f, t, -6.0f) * lv.fN2;
    b.d2[1][0] = fmaf(-12.0f, t, 6.0f) * lv.fN2;
    // slope bases: t (1-t)^2 and -t^2 (1-t)
    b.w[0][1] = tu * u * lv.dx;
    b.w[1][1] = -tu * t * lv.dx;
    b.d1[0][1] = u * fmaf(-3.0f, t, 1.0f);
    b.d1[1][1] = t * fmaf(3.0f, t, -2.0f);
    b.d2[0][1] = fmaf(6.0f, t, -4.0f) * lv.fN;
    b.d2[1][1] = fmaf(6.0f, t, -2.0f) * lv.fN;
    return b;
}

// 4D slot order (order-major, lexicographic axis lists inside an order):
// f, fx, fy, fz, fw, fxy, fxz, fxw, fyz, fyw, fzw, fxyz, fxyw, fxzw, fyzw, fxyzw.
// kSlotAlpha4[slot] = alpha mask; kAlphaSlot4[alpha] = slot; kOrderOff4[k] = first slot of order k.
__host__ __device__ constexpr int slot_alpha4(int s) {
    constexpr int t[16] = {0, 1, 2, 4, 8, 3, 5, 9, 6, 10, 12, 7, 11, 13, 14, 15};
    return t[s];
}
__host__ __device__ constexpr int alpha_slot4(int a) {
    constexpr int t[16] = {0, 1, 2, 5, 3, 6, 8, 11, 4, 7, 9, 12, 10, 13, 14, 15};
    return t[a];
}
__host__ __device__ constexpr int order_off4(int k) {
    constexpr int t[5] = {0, 1, 5, 11, 15};
    return t[k];
}

// alpha (bit i = d/dx_i) -> position of its slot in the packed vertex row
// (order-major, lexicographic inside an order): 2D f,fx,fy,fxy;
// 3D f,fx,fy,fz,fxy,fxz,fyz,fxyz; 4D as above.
template <int D>
__device__ __forceinline__ constexpr int packed_slot(int alpha) {
    if (D == 2) return alpha;
    if (D == 4) return alpha_slot4(alpha);
    // 3D: masks 0,1,2,4,3,5,6,7 occupy slots 0..7
    return alpha == 3 ? 4 : (alpha == 4 ? 3 : alpha);
}

// alpha -> its order k and its position inside bucket k.
__device__ __forceinline__ constexpr int alpha_order(int alpha) {
    return (alpha & 1) + ((alpha >> 1) & 1) + ((alpha >> 2) & 1) + ((alpha >> 3) & 1);
}
template <int D>
__device__ __forceinline__ constexpr int bucket_slot(int alpha) {
    if (D == 4) return alpha_slot4(alpha) - order_off4(alpha_order(alpha));
    // k=1: x,y,z -> 0,1,2; k=2: xy,xz,yz -> 0,1,2; k=0 and k=3 -> 0
    if (alpha_order(alpha) == 1) return alpha == 1 ? 0 : (alpha == 2 ? 1 : 2);
    if (alpha_order(alpha) == 2) return alpha == 3 ? 0 : (alpha == 5 ? 1 : 2);
    return 0;
}

template <typename TT>
__device__ __forceinline__ float to_f32(TT v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

// Read-only loads of ROW_BYTES contiguous bytes (ROW_BYTES in {8,16,32,64},
// address aligned to min(32, ROW_BYTES)) into registers.
template <int ROW_BYTES>
struct RowRegs {
    static constexpr int kWords = ROW_BYTES / 4;
    uint32_t w[kWords];
};

__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t (&r)[8]);

template <int ROW_BYTES>
__device__ __forceinline__ void load_row(const void* p, RowRegs<ROW_BYTES>& r) {
    if constexpr (ROW_BYTES >= 32) {
        // one 256-bit load per 32 bytes: a single L1 wavefront per sector pair
#pragma unroll
        for (int i = 0; i < ROW_BYTES / 32; ++i) {
            uint32_t q[8];
            ld_nc_v8(static_cast<const char*>(p) + 32 * i, q);
#pragma unroll
            for (int j = 0; j < 8; ++j) r.w[8 * i + j] = q[j];
        }
    } else if constexpr (ROW_BYTES == 16) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int i = 0; i < ROW_BYTES / 16; ++i) {
            const uint4 v = __ldg(q + i);
            r.w[4 * i + 0] = v.x;
            r.w[4 * i + 1] = v.y;
            r.w[4 * i + 2] = v.z;
            r.w[4 * i + 3] = v.w;
        }
    } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
        r.w[0] = v.x;
        r.w[1] = v.y;
    }
}

template <typename TT, int ROW_BYTES>
__device__ __forceinline__ float row_elem(const RowRegs<ROW_BYTES>& r, int i) {
    if constexpr (sizeof(TT) == 4) {
        return __uint_as_float(r.w[i]);
    } else {
        const uint32_t word = r.w[i >> 1];
        const unsigned short bits = static_cast<unsigned short>((i & 1) ? (word >> 16) : (word & 0xffffu));
        return __half2float(__ushort_as_half(bits));
    }
}

// Fire-and-forget float atomics in global memory (RED; no return value).
__device__ __forceinline__ void red_add_f32(float* a, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_v2(float* a, float x, float y) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void red_add_v4(float* a, float x, float y, float z, float w) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(a), "f"(x), "f"(y), "f"(z), "f"(w)
                 : "memory");
}

}  // namespace hg

namespace hg {

// Multi-index alpha held by packed slot s (inverse of packed_slot).
template <int D>
__host__ __device__ constexpr int slot_alpha(int s) {
    return D == 2 ? s : (D == 4 ? slot_alpha4(s) : (s == 3 ? 4 : (s == 4 ? 3 : s)));
}

// Lane-split rows: G lanes share one (point, level); lane g owns the S = 2^D/G
// consecutive packed slots g*S .. g*S+S-1 of every corner row.  Bit i of the
// multi-index of unit u is the same in every lane when !split_bit_varies.
template <int D, int G>
__host__ __device__ constexpr bool split_bit_varies(int u, int i) {
    constexpr int S = (1 << D) / G;
    const int b0 = (slot_alpha<D>(u) >> i) & 1;
    for (int g = 1; g < G; ++g)
        if (((slot_alpha<D>(g * S + u) >> i) & 1) != b0) return true;
    return false;
}

// One axis' weights of the two corners for one basis order.
struct AxisW {
    float w[2], d1[2], d2[2];
};

__device__ __forceinline__ AxisW axis_pick(const Basis1& b, bool slope) {
    AxisW r;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        r.w[v] = slope ? b.w[v][1] : b.w[v][0];
        r.d1[v] = slope ? b.d1[v][1] : b.d1[v][0];
        r.d2[v] = slope ? b.d2[v][1] : b.d2[v][0];
    }
    return r;
}

// Weights of axis i for unit u of a G-lane split (compile-time when the bit
// does not vary across lanes).
template <int D, int G>
__device__ __forceinline__ AxisW unit_axis(const Basis1& b, int lane, int u, int i) {
    constexpr int S = (1 << D) / G;
    if (split_bit_varies<D, G>(u, i)) return axis_pick(b, (slot_alpha<D>(lane * S + u) >> i) & 1);
    return axis_pick(b, (slot_alpha<D>(u) >> i) & 1);
}

// 256-bit read-only load (sm_100+): 32 bytes, 32-byte aligned.
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t (&r)[8]) {
    float f[8];
    asm("ld.global.nc.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]), "=f"(f[4]), "=f"(f[5]), "=f"(f[6]), "=f"(f[7])
        : "l"(p));
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(f[i]);
}

}  // namespace hg

namespace hg {

// ---------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ f32x2 arithmetic): one 64-bit register holds the
// same quantity for features 0 (low half) and 1 (high half).  Each f32x2
// instruction is exactly two round-to-nearest fp32 operations.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ uint64_t f2_dup(float x) { return f2_pack(x, x); }
__device__ __forceinline__ void f2_unpack(uint64_t r, float& x, float& y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// One axis' weights broadcast to both halves of a pair.
struct AxisW2 {
    uint64_t w[2], d1[2], d2[2];
};

__device__ __forceinline__ AxisW2 axis_dup(const AxisW& a) {
    AxisW2 r;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        r.w[v] = f2_dup(a.w[v]);
        r.d1[v] = f2_dup(a.d1[v]);
        r.d2[v] = f2_dup(a.d2[v]);
    }
    return r;
}

// 256-bit read-only load as four 64-bit words (32-byte aligned).
__device__ __forceinline__ void ld_nc_v4b64(const void* p, uint64_t (&r)[4]) {
    asm("ld.global.nc.v4.b64 {%0,%1,%2,%3}, [%4];" : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]) : "l"(p));
}

// L2 eviction priorities for read-only loads (createpolicy + L2::cache_hint).
// Every level's pass re-reads the points' coordinates while its own stream
// (a level's upstream gradients or outputs, its table) passes through the
// L2: loaded evict-last, the coordinates stay resident from one pass to the
// next instead of coming back from DRAM once per level; the upstream
// gradients, read once, are loaded evict-first.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float ldg_hint(const float* p, uint64_t pol) {
    float v;
    asm("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
    return v;
}

}  // namespace hg

namespace hg {

// Warp-level aggregation of scatter contributions for spatially coherent
// points.  Items occupy G consecutive lanes each (lane = item * G + part);
// consecutive items of the warp whose cells are equal form a run.  The values
// x[] of every lane are summed over its run (same part) into the run's first
// item, whose lanes return true and issue the reductions; the other lanes
// return false.  When no run is longer than one item (random points), the
// exchange is skipped for the whole warp.  `active` is the warp's lanes that
// hold an item -- the low lanes (items beyond n sit at the end); every lane in
// it must call this function.
template <int D, int G, int NV>
__device__ __forceinline__ bool run_aggregate(unsigned active, const uint32_t (&c)[D], float (&x)[NV]) {
    const int wl = threadIdx.x & 31;
    bool same = wl >= G;
#pragma unroll
    for (int i = 0; i < D; ++i) {
        const uint32_t prev = __shfl_up_sync(active, c[i], G);
        same = same && prev == c[i];
    }
    const bool head = !same;
    const unsigned heads = __ballot_sync(active, head);
    if (heads == active) return true;
    // my run ends before the first head in a later item (or the last active lane)
    const int last_of_item = wl | (G - 1);
    const unsigned later = last_of_item >= 31 ? 0u : heads & ~((2u << last_of_item) - 1u);
    const int end = later ? __ffs(later) - 1 : 32 - __clz(active);
#pragma unroll
    for (int off = G; off < 32; off <<= 1) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const float y = __shfl_down_sync(active, x[k], off);
            if (wl + off < end) x[k] += y;
        }
    }
    return head;
}

}  // namespace hg

namespace hg {

// Lanes of the calling warp that hold one of the n items when items are
// numbered first_item + lane / G from lane 0 of the warp.
template <int G>
__device__ __forceinline__ unsigned item_lanes(int64_t first_item, int64_t n) {
    const int64_t left = (n - first_item) * G;
    return left >= 32 ? 0xffffffffu : (left <= 0 ? 0u : ((1u << left) - 1u));
}

}  // namespace hg

namespace hg {

// d-linear weight of corner v (bit i = high side along axis i) at local coordinates t.
template <int D>
__device__ __forceinline__ float corner_weight(const float (&t)[D], int v) {
    float w = 1.f;
#pragma unroll
    for (int i = 0; i < D; ++i) w *= ((v >> i) & 1) ? t[i] : 1.f - t[i];
    return w;
}

}  // namespace hg
