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
        if (D == 3) i += g[D - 1] * lv.side2;
        return i;
    }
    uint32_t h = g[0] ^ (g[1] * kPrime1);
    if (D == 3) h ^= g[D - 1] * kPrime2;
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

// alpha (bit i = d/dx_i) -> position of its slot in the packed vertex row
// (order-major, lexicographic inside an order): 2D f,fx,fy,fxy;
// 3D f,fx,fy,fz,fxy,fxz,fyz,fxyz.
template <int D>
__device__ __forceinline__ constexpr int packed_slot(int alpha) {
    if (D == 2) return alpha;
    // 3D: masks 0,1,2,4,3,5,6,7 occupy slots 0..7
    return alpha == 3 ? 4 : (alpha == 4 ? 3 : alpha);
}

// alpha -> its order k and its position inside bucket k.
__device__ __forceinline__ constexpr int alpha_order(int alpha) {
    return (alpha & 1) + ((alpha >> 1) & 1) + ((alpha >> 2) & 1);
}
template <int D>
__device__ __forceinline__ constexpr int bucket_slot(int alpha) {
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
// address aligned to min(16, ROW_BYTES)) into registers.
template <int ROW_BYTES>
struct RowRegs {
    static constexpr int kWords = ROW_BYTES / 4;
    uint32_t w[kWords];
};

template <int ROW_BYTES>
__device__ __forceinline__ void load_row(const void* p, RowRegs<ROW_BYTES>& r) {
    if constexpr (ROW_BYTES >= 16) {
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
