/*
 * mxfp8_testing.h -- testing and benchmarking hooks of the GB300 MXFP8
 * library.  NOT part of the layer's interface (include/mxfp8.h): each hook
 * changes process-wide state that every later call on any thread sees, so a
 * product caller never needs them.  The tests use them to force each
 * schedule, to turn a wait into an error on purpose, and to read back which
 * schedule ran.
 */
#ifndef MXFP8_GB300_TESTING_H
#define MXFP8_GB300_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Testing hook: pin the GEMM schedule, process-wide.
 * tokens_per_tile: 0 (automatic) or 16, 32, 64, 128, 256 (256 needs split_k -1),
 * or 144, 160, 176, 192: two 128-row weight tiles per CTA tile (dense,
 * persistent);
 * split_k: 0 automatic, -1 persistent tiles, 1..8 one tile per cluster of
 * split_k CTAs (K split among them, tokens_per_tile <= 128);
 * fuse_quant: -1 automatic, 0 never, 1 whenever the schedule allows
 * (one-tile schedules of mxfp8_linear) -- the GEMM then quantizes x itself. */
void mxfp8_set_schedule(int tokens_per_tile, int split_k, int fuse_quant);

/* Testing hook for failure detection: limit, in nanoseconds, of every
 * pipeline wait of later GEMM launches (0 restores the default, 4 s).  A wait
 * that runs out sets the device error word read by mxfp8_device_error(); the
 * kernel then unwinds (in-flight copies and MMAs drained, TMEM freed) and
 * returns, so the context stays usable.  Process-wide. */
void mxfp8_set_wait_limit_ns(uint64_t ns);

/* Testing hook: MMA pipelines per CTA for later launches (0 = automatic, 1,
 * 2, or 4; more than one only for tiles of <= 64 tokens, 4 only for 16).
 * Each pipeline has its own producer and MMA-issuing thread, owns every
 * pipes-th K block of a tile and accumulates in its own TMEM columns; the
 * epilogue sums them in pipeline order.  Process-wide. */
void mxfp8_set_pipes(int pipes);

/* Testing hook: the schedule of the calling thread's last GEMM launch, as
 * out5[0..4] = {tokens per tile + 1000 * (pipelines - 1), split (-1 =
 * persistent), fused quantization (0/1), grid size, stages per pipeline}. */
void mxfp8_last_schedule(int* out5);

/* 1 when this library is the debug build (MXFP8_DEBUG: every computed store
 * index is checked against its buffer; see mxfp8_device_error), else 0. */
int mxfp8_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_GB300_TESTING_H */
