// Hardware probes for the roofline of the encoding kernels (declared in
// include/hg_probe.h): random whole-row gathers from, and random 16-byte
// vector REDs into, a buffer small enough to stay in L2, with the same
// lanes-per-row split the encoding kernels use.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hg_probe.h"
#include "hg_device.cuh"

namespace {

constexpr int kBlock = 256;

// A 32-bit integer mix (two multiply-xorshift rounds) used to pick rows.
__device__ __forceinline__ uint32_t mix(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// ROW bytes per row, LPR lanes per row; each lane reads CH = ROW/LPR bytes.
template <int ROW, int LPR>
__global__ void __launch_bounds__(kBlock) gather_kernel(const char* __restrict__ buf, uint32_t row_mask,
                                                        int rows_per_group, uint32_t seed, float* sink,
                                                        int64_t n_threads) {
    constexpr int CH = ROW / LPR;
    constexpr int W = CH / 4;  // 32-bit words per lane per row
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (tid >= n_threads) return;
    const uint32_t grp = static_cast<uint32_t>(tid / LPR), lane = static_cast<uint32_t>(tid % LPR);
    uint32_t acc = 0;
    for (int r = 0; r < rows_per_group; r += 8) {
        uint32_t v[8][W];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t row = mix(grp * 0x9e3779b9u + (r + j) * 0x85ebca6bu + seed) & row_mask;
            const char* p = buf + static_cast<size_t>(row) * ROW + lane * CH;
            if constexpr (CH % 32 == 0) {
#pragma unroll
                for (int h = 0; h < CH / 32; ++h) {
                    uint32_t q[8];
                    hg::ld_nc_v8(p + 32 * h, q);
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[j][8 * h + i] = q[i];
                }
            } else if constexpr (CH % 16 == 0) {
#pragma unroll
                for (int h = 0; h < CH / 16; ++h) {
                    const uint4 q = __ldg(reinterpret_cast<const uint4*>(p + 16 * h));
                    v[j][4 * h + 0] = q.x;
                    v[j][4 * h + 1] = q.y;
                    v[j][4 * h + 2] = q.z;
                    v[j][4 * h + 3] = q.w;
                }
            } else {
                const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));  // 8-byte rows
                v[j][0] = q.x;
                v[j][1] = q.y;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int i = 0; i < W; ++i) acc ^= v[j][i];
    }
    sink[tid] = __uint_as_float(acc & 0x007fffffu);
}

template <int ROW, int LPR>
__global__ void __launch_bounds__(kBlock) red_kernel(float* buf, uint32_t row_mask, int rows_per_group, uint32_t seed,
                                                     int64_t n_threads) {
    constexpr int CH = ROW / LPR;  // bytes per lane: 8 or a multiple of 16
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (tid >= n_threads) return;
    const uint32_t grp = static_cast<uint32_t>(tid / LPR), lane = static_cast<uint32_t>(tid % LPR);
    for (int r = 0; r < rows_per_group; ++r) {
        const uint32_t row = mix(grp * 0x9e3779b9u + r * 0x85ebca6bu + seed) & row_mask;
        float* p = buf + static_cast<size_t>(row) * (ROW / 4) + lane * (CH / 4);
        if constexpr (CH == 8) {
            hg::red_add_v2(p, 1.f, 1.f);
        } else {
#pragma unroll
            for (int h = 0; h < CH / 16; ++h) hg::red_add_v4(p + 4 * h, 1.f, 1.f, 1.f, 1.f);
        }
    }
}

// Replay of an encoding launch's row stream: one item per (point, level)
// shared by `lanes` consecutive threads, every corner row of the point's
// cell (the library's own cell location and index function, order-0 table
// geometry = the packed row), each lane moving its CH-byte chunk of the row
// with one vector load (gather) or one vector RED of 1.0s; no arithmetic.
template <int D, int CH, bool RED>
__global__ void __launch_bounds__(kBlock) replay_kernel(const __grid_constant__ hg::ReplayParams p) {
    const int l = p.c.lvl[blockIdx.y];
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t n = tid / p.lanes;
    const int lane = static_cast<int>(tid % p.lanes);
    if (n >= p.c.n || !((p.c.level_mask >> l) & 1u)) return;
    const hg::Level& lv = p.c.lv[l];
    uint32_t c[D];
    float t[D];
#pragma unroll
    for (int i = 0; i < D; ++i) hg::locate(__ldg(p.coords + n * D + i), lv, c[i], t[i]);
    char* lbase = p.base + l * p.level_bytes + lane * CH;
    uint32_t acc = 0;
#pragma unroll
    for (int v = 0; v < (1 << D); ++v) {
        uint32_t g[D];
#pragma unroll
        for (int i = 0; i < D; ++i) g[i] = c[i] + ((v >> i) & 1u);
        char* a = lbase + static_cast<int64_t>(hg::vertex_index<D>(g, lv, lv.dense & 1u, p.c.tmask[0])) * p.row_bytes;
        if constexpr (RED) {
            float* f = reinterpret_cast<float*>(a);
            if constexpr (CH == 16) hg::red_add_v4(f, 1.f, 1.f, 1.f, 1.f);
            else if constexpr (CH == 8) hg::red_add_v2(f, 1.f, 1.f);
            else hg::red_add_f32(f, 1.f);
        } else if constexpr (CH == 32) {
            uint32_t q[8];
            hg::ld_nc_v8(a, q);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc ^= q[i];
        } else if constexpr (CH == 16) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(a));
            acc ^= q.x ^ q.y ^ q.z ^ q.w;
        } else if constexpr (CH == 8) {
            const uint2 q = __ldg(reinterpret_cast<const uint2*>(a));
            acc ^= q.x ^ q.y;
        } else {
            acc ^= __ldg(reinterpret_cast<const uint32_t*>(a));
        }
    }
    if constexpr (!RED) p.sink[tid] = __uint_as_float(acc & 0x007fffffu);
}

template <int D, bool RED>
cudaError_t launch_replay_d(const hg::ReplayParams& p, int ch, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((p.c.n * p.lanes + kBlock - 1) / kBlock), static_cast<unsigned>(p.c.nlvl));
    switch (ch) {
        case 32: if constexpr (!RED) { replay_kernel<D, 32, RED><<<grid, kBlock, 0, s>>>(p); break; } else return cudaErrorInvalidValue;
        case 16: replay_kernel<D, 16, RED><<<grid, kBlock, 0, s>>>(p); break;
        case 8: replay_kernel<D, 8, RED><<<grid, kBlock, 0, s>>>(p); break;
        case 4: replay_kernel<D, 4, RED><<<grid, kBlock, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int ROW, int LPR>
cudaError_t launch_gather(const void* buf, uint32_t mask, int rpg, uint32_t seed, float* sink, int64_t nt,
                          cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>((nt + kBlock - 1) / kBlock);
    gather_kernel<ROW, LPR><<<blocks, kBlock, 0, s>>>(static_cast<const char*>(buf), mask, rpg, seed, sink, nt);
    return cudaGetLastError();
}

template <int ROW, int LPR>
cudaError_t launch_red(float* buf, uint32_t mask, int rpg, uint32_t seed, int64_t nt, cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>((nt + kBlock - 1) / kBlock);
    red_kernel<ROW, LPR><<<blocks, kBlock, 0, s>>>(buf, mask, rpg, seed, nt);
    return cudaGetLastError();
}

}  // namespace

namespace hg {
int launch_replay(const ReplayParams& p, bool red, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int ch = p.row_bytes / p.lanes;
    if (p.c.nlvl == 0 || p.c.n == 0) return cudaSuccess;
    switch (p.c.d) {
        case 2: return red ? launch_replay_d<2, true>(p, ch, s) : launch_replay_d<2, false>(p, ch, s);
        case 3: return red ? launch_replay_d<3, true>(p, ch, s) : launch_replay_d<3, false>(p, ch, s);
        default: return red ? launch_replay_d<4, true>(p, ch, s) : launch_replay_d<4, false>(p, ch, s);
    }
}
}  // namespace hg

extern "C" {

hg_status hg_probe_l2_gather(const void* buf, int32_t log2_rows, int32_t row_bytes, int32_t lanes_per_row,
                             int64_t n_threads, int32_t rows_per_group, uint32_t seed, float* sink, hg_stream stream) {
    if (!buf || !sink || !aligned(buf, 32) || !aligned(sink, 4)) return HG_ERR_INVALID_ARG;
    if (log2_rows < 4 || log2_rows > 30 || rows_per_group < 8 || rows_per_group % 8) return HG_ERR_INVALID_ARG;
    if (lanes_per_row != 1 && lanes_per_row != 2 && lanes_per_row != 4) return HG_ERR_INVALID_ARG;
    if (n_threads < lanes_per_row || n_threads % lanes_per_row || n_threads > int64_t(INT32_MAX)) return HG_ERR_INVALID_ARG;
    const uint32_t mask = (1u << log2_rows) - 1u;
    cudaError_t e;
    if (row_bytes == 8 && lanes_per_row == 1) e = launch_gather<8, 1>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 16 && lanes_per_row == 1) e = launch_gather<16, 1>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 32 && lanes_per_row == 1) e = launch_gather<32, 1>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 32 && lanes_per_row == 2) e = launch_gather<32, 2>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 64 && lanes_per_row == 1) e = launch_gather<64, 1>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 64 && lanes_per_row == 2) e = launch_gather<64, 2>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 64 && lanes_per_row == 4) e = launch_gather<64, 4>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else if (row_bytes == 128 && lanes_per_row == 4) e = launch_gather<128, 4>(buf, mask, rows_per_group, seed, sink, n_threads, stream);
    else return HG_ERR_INVALID_ARG;
    return e == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}

hg_status hg_probe_l2_red(float* buf, int32_t log2_rows, int32_t row_bytes, int32_t lanes_per_row, int64_t n_threads,
                          int32_t rows_per_group, uint32_t seed, hg_stream stream) {
    if (!buf || !aligned(buf, 16) || log2_rows < 4 || log2_rows > 30 || rows_per_group < 1) return HG_ERR_INVALID_ARG;
    if (lanes_per_row != 1 && lanes_per_row != 2 && lanes_per_row != 4 && lanes_per_row != 8) return HG_ERR_INVALID_ARG;
    if (n_threads < lanes_per_row || n_threads % lanes_per_row || n_threads > int64_t(INT32_MAX)) return HG_ERR_INVALID_ARG;
    const uint32_t mask = (1u << log2_rows) - 1u;
    cudaError_t e;
    if (row_bytes == 8 && lanes_per_row == 1) e = launch_red<8, 1>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 16 && lanes_per_row == 1) e = launch_red<16, 1>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 32 && lanes_per_row == 1) e = launch_red<32, 1>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 32 && lanes_per_row == 2) e = launch_red<32, 2>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 64 && lanes_per_row == 1) e = launch_red<64, 1>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 64 && lanes_per_row == 2) e = launch_red<64, 2>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 64 && lanes_per_row == 4) e = launch_red<64, 4>(buf, mask, rows_per_group, seed, n_threads, stream);
    else if (row_bytes == 128 && lanes_per_row == 8) e = launch_red<128, 8>(buf, mask, rows_per_group, seed, n_threads, stream);
    else return HG_ERR_INVALID_ARG;
    return e == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}

}  // extern "C"
