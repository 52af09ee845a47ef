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

/* Random-row gather: n_threads threads each read `rows_per_thread` rows of
 * row_bytes (32 or 64) bytes, chosen by an integer hash among the
 * 2^log2_rows rows of `buf` (device, 16-byte aligned, 2^log2_rows * row_bytes
 * bytes), with 16-byte vector loads, and write one float each to `sink`
 * (device float [n_threads]).  Bytes moved = n_threads * rows_per_thread *
 * row_bytes.  Errors: HG_ERR_INVALID_ARG for NULL / misaligned pointers,
 * row_bytes not 32 or 64, log2_rows outside 4..30, rows_per_thread not a
 * positive multiple of 8, n_threads < 1; HG_ERR_CUDA on launch failure. */
hg_status hg_probe_l2_gather(const void* buf, int32_t log2_rows, int32_t row_bytes, int64_t n_threads,
                             int32_t rows_per_thread, uint32_t seed, float* sink, hg_stream stream);

/* Random vector reduction: n_threads threads each issue `ops_per_thread`
 * red.global.add.v4.f32 (16 bytes of payload) at 16-byte slots chosen by an
 * integer hash among the 2^log2_slots slots of `buf` (device float,
 * 4 * 2^log2_slots floats, 16-byte aligned), adding 1.0 to each lane.
 * Payload bytes = n_threads * ops_per_thread * 16.  Errors: as above
 * (log2_slots in 4..30, ops_per_thread >= 1). */
hg_status hg_probe_l2_red(float* buf, int32_t log2_slots, int64_t n_threads, int32_t ops_per_thread, uint32_t seed,
                          hg_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* HG_PROBE_H */
