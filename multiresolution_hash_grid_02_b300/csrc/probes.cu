// Hardware probes for the roofline of the encoding kernels (declared in
// include/hg_probe.h): random 16-byte-vector row gathers from, and random
// 16-byte vector REDs into, a buffer small enough to stay in L2.
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

template <int ROW>
__global__ void __launch_bounds__(kBlock) gather_kernel(const uint4* __restrict__ buf, uint32_t row_mask,
                                                        int rows_per_thread, uint32_t seed, float* sink,
                                                        int64_t n_threads) {
    constexpr int Q = ROW / 16;
    const uint32_t tid = blockIdx.x * kBlock + threadIdx.x;
    if (tid >= n_threads) return;
    uint32_t acc = 0;
    for (int r = 0; r < rows_per_thread; r += 8) {
        uint4 v[8][Q];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t row = mix(tid * 0x9e3779b9u + (r + j) * 0x85ebca6bu + seed) & row_mask;
#pragma unroll
            for (int q = 0; q < Q; ++q) v[j][q] = __ldg(buf + static_cast<size_t>(row) * Q + q);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int q = 0; q < Q; ++q) acc ^= v[j][q].x ^ v[j][q].y ^ v[j][q].z ^ v[j][q].w;
    }
    sink[tid] = __uint_as_float(acc & 0x007fffffu);
}

__global__ void __launch_bounds__(kBlock) red_kernel(float* buf, uint32_t slot_mask, int ops_per_thread,
                                                     uint32_t seed, int64_t n_threads) {
    const uint32_t tid = blockIdx.x * kBlock + threadIdx.x;
    if (tid >= n_threads) return;
    for (int r = 0; r < ops_per_thread; ++r) {
        const uint32_t slot = mix(tid * 0x9e3779b9u + r * 0x85ebca6bu + seed) & slot_mask;
        hg::red_add_v4(buf + static_cast<size_t>(slot) * 4, 1.f, 1.f, 1.f, 1.f);
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

hg_status hg_probe_l2_gather(const void* buf, int32_t log2_rows, int32_t row_bytes, int64_t n_threads,
                             int32_t rows_per_thread, uint32_t seed, float* sink, hg_stream stream) {
    if (!buf || !sink || !aligned16(buf) || (reinterpret_cast<uintptr_t>(sink) & 3u)) return HG_ERR_INVALID_ARG;
    if ((row_bytes != 32 && row_bytes != 64) || log2_rows < 4 || log2_rows > 30) return HG_ERR_INVALID_ARG;
    if (rows_per_thread < 8 || rows_per_thread % 8 || n_threads < 1) return HG_ERR_INVALID_ARG;
    const int64_t blocks = (n_threads + kBlock - 1) / kBlock;
    if (blocks > INT32_MAX / kBlock) return HG_ERR_INVALID_ARG;
    const uint32_t mask = (1u << log2_rows) - 1u;
    const uint4* b = static_cast<const uint4*>(buf);
    if (row_bytes == 32)
        gather_kernel<32><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(b, mask, rows_per_thread, seed, sink,
                                                                               n_threads);
    else
        gather_kernel<64><<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(b, mask, rows_per_thread, seed, sink,
                                                                               n_threads);
    return cudaGetLastError() == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}

hg_status hg_probe_l2_red(float* buf, int32_t log2_slots, int64_t n_threads, int32_t ops_per_thread, uint32_t seed,
                          hg_stream stream) {
    if (!buf || !aligned16(buf) || log2_slots < 4 || log2_slots > 30 || ops_per_thread < 1 || n_threads < 1)
        return HG_ERR_INVALID_ARG;
    const int64_t blocks = (n_threads + kBlock - 1) / kBlock;
    if (blocks > INT32_MAX / kBlock) return HG_ERR_INVALID_ARG;
    red_kernel<<<static_cast<unsigned>(blocks), kBlock, 0, stream>>>(buf, (1u << log2_slots) - 1u, ops_per_thread,
                                                                    seed, n_threads);
    return cudaGetLastError() == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}

}  // extern "C"
