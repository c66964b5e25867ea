/*
 * libdspark_bench -- measurement kernels used by bench.py to state the ceilings the
 * draft-step kernels run against.  They compute nothing of the method and have no
 * counterpart in the source pages; they exist so that a bandwidth fraction is taken
 * against numbers measured on the same GPU in the same run.
 *
 * Conventions as in dspark.h: device pointers owned by the caller, work enqueued on
 * `stream` (a cudaStream_t), no allocation, no synchronization.  Return 0 on success,
 * else the cudaError_t of the failed launch (and nothing was enqueued).
 */
#ifndef DSPARK_BENCH_H
#define DSPARK_BENCH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Reads `bytes` bytes of `buf` (16-byte aligned; bytes a multiple of 16) `passes` times
 * with 16-byte loads that are cached in L2 but not in L1, and folds every loaded word into
 * one value written to *sink (device, 8 bytes) only if it equals an unlikely constant, so the
 * loads cannot be removed.  `grid` x `block` threads stride over the buffer; with a buffer
 * smaller than L2 and passes > 1, every pass after the first is served by L2, so
 * bytes * passes / time is the L2-to-SM read bandwidth.  grid, block > 0, block <= 1024,
 * passes >= 1. */
int dspark_bench_read(const void *buf, size_t bytes, int passes, unsigned long long *sink,
                      int grid, int block, void *stream);

/* Launches one empty kernel (1 CTA, 32 threads): two events around it measure the floor
 * that event timing puts under any single launch. */
int dspark_bench_empty(void *stream);

/* The same empty kernel on `ctas` CTAs that each request `smem_bytes` of dynamic shared
 * memory (up to 227 KB): the floor for a launch shaped like the draft-step kernels, which use
 * 90-220 KB per CTA.  ctas >= 1. */
int dspark_bench_empty_smem(int ctas, int smem_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_BENCH_H */
