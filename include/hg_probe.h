/*
 * hg_probe.h -- hardware probes shipped in libhg.so for the roofline of the
 * encoding kernels.  The pages define no counterpart: these measure the chip,
 * not the method.  The encoding's gather and scatter are served from L2
 * (each level's table stays resident while that level is processed), so the
 * ceilings that matter are the rates of random 16-byte-vector reads from an
 * L2-resident buffer and of random 16-byte vector reductions (RED) into one.
 *
 * Conventions as in hg.h: device pointers owned by the caller, asynchronous
 * on `stream`, synchronous argument checking, hg_status results.
 */
#ifndef HG_PROBE_H
#define HG_PROBE_H

#include "hg.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Random-row gather: groups of `lanes_per_row` consecutive lanes (1, 2 or 4)
 * read whole rows of row_bytes (8, 16, 32, 64 or 128) bytes, each lane its
 * row_bytes/lanes_per_row-byte chunk (256-bit loads for 32-byte chunks,
 * 128-bit loads for 16-byte multiples, one 64-bit load for 8-byte rows), so
 * that one warp instruction covers whole rows.
 * Each group reads `rows_per_group` rows chosen by an integer hash among the
 * 2^log2_rows rows of `buf` (device, 32-byte aligned, 2^log2_rows * row_bytes
 * bytes); every lane writes one float to `sink` (device float [n_threads]).
 * Bytes moved = n_threads / lanes_per_row * rows_per_group * row_bytes.
 * Supported (row_bytes, lanes_per_row): (8, 1), (16, 1), (32, 1), (32, 2),
 * (64, 1), (64, 2), (64, 4), (128, 4).
 * Errors: HG_ERR_INVALID_ARG for NULL / misaligned pointers, an unsupported
 * (row_bytes, lanes_per_row) pair, log2_rows
 * outside 4..30, rows_per_group not a positive multiple of 8, n_threads not a
 * positive multiple of lanes_per_row; HG_ERR_CUDA on launch failure. */
hg_status hg_probe_l2_gather(const void* buf, int32_t log2_rows, int32_t row_bytes, int32_t lanes_per_row,
                             int64_t n_threads, int32_t rows_per_group, uint32_t seed, float* sink, hg_stream stream);

/* Random vector reduction: groups of `lanes_per_row` lanes (1, 2, 4 or 8) add
 * 1.0 to every float of whole rows of row_bytes (8, 16, 32, 64 or 128) bytes,
 * each lane issuing red.global.add.v4.f32 (16 bytes of payload; v2 for 8-byte
 * rows) on its
 * row_bytes/lanes_per_row-byte chunk, at rows chosen by an integer hash among
 * the 2^log2_rows rows of `buf` (device float, 16-byte aligned).  Payload
 * bytes = n_threads / lanes_per_row * rows_per_group * row_bytes.  Errors: as
 * above; supported (row_bytes, lanes_per_row): (8, 1), (16, 1), (32, 1), (32, 2),
 * (64, 1), (64, 2), (64, 4), (128, 8); rows_per_group >= 1. */
hg_status hg_probe_l2_red(float* buf, int32_t log2_rows, int32_t row_bytes, int32_t lanes_per_row, int64_t n_threads,
                          int32_t rows_per_group, uint32_t seed, hg_stream stream);

/* Replay of an encoding launch's memory stream -- the roofline probe of the
 * encoding kernels.  For every point and active level of `desc`, the rows of
 * the 2^d corners of the point's cell, located and indexed exactly as the
 * encoding does it (hg.h: clamp, pos = fl32(x * N_l), one-to-one or hashed
 * index in the order-0 table geometry, T = 2^log2_T[0] rows per level), each
 * row split over `lanes_per_row` consecutive threads that move
 * row_bytes / lanes_per_row bytes apiece with one vector access; no
 * arithmetic, no outputs.  Its rate is the ceiling of the kernels' own row
 * stream: the same addresses, the same lane split, only the memory work.
 *   coords: device float32 [n][d]
 *   hg_probe_replay_gather: reads rows of `table` (device; row r of level l
 *     at table + l * level_stride_bytes + r * row_bytes; the caller provides
 *     L * level_stride_bytes bytes); every thread writes one float to `sink`
 *     (device float [n * lanes_per_row]).  Chunks of 4, 8, 16 or 32 bytes.
 *   hg_probe_replay_red: adds 1.0 to every float of each chunk of `grad`
 *     (device float32, same geometry) with one RED per chunk.  Chunks of 4,
 *     8 or 16 bytes.
 * Errors: HG_ERR_INVALID_ARG for a bad descriptor (as hg_encode_fwd), n out
 * of range, NULL or chunk-misaligned pointers or strides, an unsupported
 * chunk, row_bytes not a multiple of lanes_per_row, level_stride_bytes below
 * T * row_bytes when L > 1; HG_ERR_CUDA on launch failure. */
hg_status hg_probe_replay_gather(const hg_grid_desc* desc, int64_t n, const float* coords, const void* table,
                                 int64_t level_stride_bytes, int32_t row_bytes, int32_t lanes_per_row, float* sink,
                                 hg_stream stream);
hg_status hg_probe_replay_red(const hg_grid_desc* desc, int64_t n, const float* coords, float* grad,
                              int64_t level_stride_bytes, int32_t row_bytes, int32_t lanes_per_row, hg_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* HG_PROBE_H */
