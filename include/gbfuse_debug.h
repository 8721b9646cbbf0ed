/*
 * gbfuse_debug.h -- test, tuning and profiling hooks of the fused GEMM +
 * epilogue library (libgbfuse.so).  Not part of the product boundary in
 * gbfuse.h: a caller of the library needs none of these.  They exist so that
 * the tests can exercise the failure path and every kernel variant, and so
 * that the benchmark can attribute time; each one changes only how later
 * launches are scheduled or instrumented, never what they compute beyond the
 * order of rounding.  The settings are process-wide and not synchronised with
 * launches already enqueued.
 */
#ifndef GBFUSE_DEBUG_H
#define GBFUSE_DEBUG_H

#include "gbfuse.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Test hook: when `on` is non-zero, the next launches of the fused GEMM
 * kernels withhold one accumulator-ready signal so that the epilogue's
 * bounded wait runs out; the kernel then records GBF_ERR_TIMEOUT and exits
 * cleanly.  Off by default. */
GBF_API gbf_status_t gbf_debug_inject_timeout(int on);

/* Profiling hook: with a zeroed device buffer of `bytes` registered, each CTA
 * of later launches (if the buffer has room for 32 counters per CTA) adds,
 * per wait site i of its pipeline, the cycles spent waiting to counter 2i and
 * the number of waits to counter 2i+1, and its total cycles to counter 31
 * (unsigned 64-bit, CTA b at offset 32*b, b = linear block index).  NULL
 * turns it off (the default).  The caller owns and clears the buffer. */
GBF_API gbf_status_t gbf_debug_set_profile(void *counters, size_t bytes);

/* Tuning hook: the split-K cluster size of the swapped small-M and W4A16
 * kernels (1..8) for later launches, or 0 (default) for the automatic choice
 * (about two CTAs per SM).  Changes the partition of the work, not its
 * result beyond the order of the fp32 partial sums. */
GBF_API gbf_status_t gbf_debug_force_splits(int splits);

/* Tuning hook: for the dense product (and the gate/up GEMM) at M above the
 * swapped kernel's range, run the persistent kernel (1), its split-K form
 * over two CTAs per tile (5), the CTA-pair kernel (4), the CTA-pair kernel
 * with one MMA stream (6) or its split-K form over two pairs per tile (7) for
 * later launches instead of the automatic choice (0, the default); 5, 6 and 7
 * apply to the single product only (the gate/up GEMM then takes the
 * automatic choice; 7 also needs K >= 128).  Other values return GBF_ERR_INVALID_ARG.
 * Changes which kernel computes the result, not the result beyond the order
 * of rounding. */
GBF_API gbf_status_t gbf_debug_force_path(int path);

#ifdef __cplusplus
}
#endif

#endif /* GBFUSE_DEBUG_H */
