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
 * read whole rows of row_bytes (32, 64 or 128) bytes, each lane its
 * row_bytes/lanes_per_row-byte chunk (256-bit loads for 32-byte chunks,
 * 128-bit loads otherwise), so that one warp instruction covers whole rows.
 * Each group reads `rows_per_group` rows chosen by an integer hash among the
 * 2^log2_rows rows of `buf` (device, 32-byte aligned, 2^log2_rows * row_bytes
 * bytes); every lane writes one float to `sink` (device float [n_threads]).
 * Bytes moved = n_threads / lanes_per_row * rows_per_group * row_bytes.
 * Supported (row_bytes, lanes_per_row): (32, 1), (32, 2), (64, 1), (64, 2),
 * (64, 4), (128, 4).
 * Errors: HG_ERR_INVALID_ARG for NULL / misaligned pointers, an unsupported
 * (row_bytes, lanes_per_row) pair, log2_rows
 * outside 4..30, rows_per_group not a positive multiple of 8, n_threads not a
 * positive multiple of lanes_per_row; HG_ERR_CUDA on launch failure. */
hg_status hg_probe_l2_gather(const void* buf, int32_t log2_rows, int32_t row_bytes, int32_t lanes_per_row,
                             int64_t n_threads, int32_t rows_per_group, uint32_t seed, float* sink, hg_stream stream);

/* Random vector reduction: groups of `lanes_per_row` lanes (1, 2, 4 or 8) add
 * 1.0 to every float of whole rows of row_bytes (16, 32, 64 or 128) bytes, each
 * lane issuing red.global.add.v4.f32 (16 bytes of payload) on its
 * row_bytes/lanes_per_row-byte chunk, at rows chosen by an integer hash among
 * the 2^log2_rows rows of `buf` (device float, 16-byte aligned).  Payload
 * bytes = n_threads / lanes_per_row * rows_per_group * row_bytes.  Errors: as
 * above; supported (row_bytes, lanes_per_row): (16, 1), (32, 1), (32, 2),
 * (64, 1), (64, 2), (64, 4), (128, 8); rows_per_group >= 1. */
hg_status hg_probe_l2_red(float* buf, int32_t log2_rows, int32_t row_bytes, int32_t lanes_per_row, int64_t n_threads,
                          int32_t rows_per_group, uint32_t seed, hg_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* HG_PROBE_H */
