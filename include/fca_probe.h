/*
 * fca_probe.h - micro-benchmarks that measure the bounds of the enumeration
 * kernels' roofline on the current GPU: the issue rate of 32-bit logical
 * operations (the closure and canonical tests are AND/ANDNOT/OR on words) and
 * the read bandwidth of an L2-resident buffer (the bitmap tier streams
 * extents and columns that fit in L2). The pages give no such numbers; these
 * probes exist so the measured kernels can be put against measured peaks.
 * Plain C ABI; all pointers are host pointers; calls are synchronous.
 */
#ifndef FCA_PROBE_H
#define FCA_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Issue rate of lop3.b32 with many independent chains per thread, on every SM.
 *   ops_per_s  receives LOP3 instructions per second (one per thread per op)
 *   ms         receives the kernel time (CUDA events)
 * Returns 0, or a CUDA error code.
 */
int fca_probe_lop3(double *ops_per_s, double *ms);

/*
 * Read bandwidth of a device buffer of `bytes` bytes (uint4 loads that skip
 * L1, all SMs, the buffer read 8 times per launch), best of `reps` launches
 * after one warm-up launch. With bytes well below the L2 size this is the L2
 * read bandwidth.
 *   gbps       receives bytes read per second / 1e9
 * Returns 0, or a CUDA error code (the buffer is allocated and freed inside).
 */
int fca_probe_read_bw(uint64_t bytes, int reps, double *gbps);

#ifdef __cplusplus
}
#endif

#endif /* FCA_PROBE_H */
