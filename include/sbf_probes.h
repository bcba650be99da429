/* sbf_probes.h -- micro-benchmarks of the hardware ceilings that the Super
 * Bloom filter kernels are measured against (libsbf_probes.so).
 *
 * Not part of the filter's API: the benchmark calls these to measure, on the
 * GPU it runs on, the rate of the access pattern and of the instruction mix
 * that bound the insert and the query ("cuSBF: A Minimizer-Aware Bloom Filter
 * for Genomic Sequence Data on Modern GPUs", Sec. V-F and Fig. 7: the kernels
 * are limited by on-chip integer work while the filter fits in L2, and by
 * scattered shard accesses beyond it).
 *
 * Conventions: device pointers are caller-owned device memory; `stream` is a
 * cudaStream_t (NULL = legacy default stream); every call only enqueues one
 * kernel and returns (time it with events on `stream`).  Returns 0, or -1 for
 * invalid arguments (nothing launched), or -2 when the launch failed.
 * Random rows come from a counter-based generator (the SplitMix64 output
 * function applied to seed + i), so no index array is read. */
#ifndef SBF_PROBES_H
#define SBF_PROBES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Streaming-multiprocessor count of the current device (cudaGetDeviceProperties). */
int sbf_probe_sm_count(int *sms);

/* Integer instruction throughput.  kind: 0 = the mix that dominates the
 * filter kernels' ALU pipe (LOP3, funnel shift, compare, select, min: five
 * instructions per step), 1 = LOP3 only, 2 = funnel shift only, 3 = integer
 * multiply-add only (the FMA pipe), 4 = 64-bit unsigned minimum (min.u64;
 * three per step, counted as one operation each).  Each of blocks x threads threads runs
 * `iters` rounds of 32 steps over eight independent chains.  *ops receives the
 * instructions one launch executes (threads x iters x 32 x instructions per
 * step).  sink: device uint32[blocks * threads], written once per thread. */
int sbf_probe_alu(int kind, int iters, int blocks, int threads, uint32_t *sink, void *stream, double *ops);

/* Random 32-byte row read-modify-writes: n_updates rows chosen uniformly
 * among n_rows (a power of two) rows of buf (device uint64[4 * n_rows]).
 * mode 0: one thread per row, four 64-bit OR reductions (red.global.or.b64),
 * as the insert's run flush; mode 1: four consecutive lanes per row, one
 * reduction each (one 32-byte request per row); mode 2: a plain 32-byte load
 * and store per row (not atomic: a data point, not a filter update); mode 3:
 * each thread queues its row and four words in its warp's shared memory, then
 * the warp issues them as in mode 1 (threads a multiple of 32). */
int sbf_probe_rmw(int mode, uint64_t *buf, uint64_t n_rows, int64_t n_updates, uint64_t seed, int blocks,
                  int threads, void *stream);

/* Random 32-byte row reads (n_reads rows of buf, uniformly among n_rows, a
 * power of two), eight in flight per thread.  mode 0: ld.global.nc.v4.u64;
 * 1, 2, 3: the same with an L2 prefetch-size hint of 64, 128, 256 bytes;
 * 4: two 16-byte cp.async.cg copies into shared memory (the query's shard
 * staging); 5: the same with a 64-byte prefetch-size hint; 6: one 32-byte
 * bulk copy (cp.async.bulk) per row into shared memory, completed on a
 * per-thread mbarrier (bounded wait; a thread that gives up writes ~0 to its
 * sink word and stops).  threads <= 256.
 * sink: device uint64[blocks * threads], written once per thread. */
int sbf_probe_read(int mode, const uint64_t *buf, uint64_t n_rows, int64_t n_reads, uint64_t seed, int blocks,
                   int threads, uint64_t *sink, void *stream);

#ifdef __cplusplus
}
#endif

#endif
