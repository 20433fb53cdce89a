/*
 * hoc_workload.h -- measurement and workload kernels that run beside the
 * collectives (they are not collectives themselves).
 *
 * HOCCL section 2.1 defines the contention rate I_x (Eq. 1): the share of SMs
 * that communication of class x occupies while compute kernels are active,
 * and Fig. 2b shows compute slowing down as it grows.  The probe below is the
 * compute kernel whose slowdown measures that contention on one GPU.  The XOR
 * transform stands in for a pipeline stage's compute on its activations
 * (section 2.1, PP overlaps activation transfers with compute) with an exact,
 * invertible result.
 */
#ifndef HOC_WORKLOAD_H
#define HOC_WORKLOAD_H

#include <stddef.h>
#include <stdint.h>

#include "hoc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Compute-bound probe: `ctas` CTAs of `threads` threads on `stream`; each
 * thread runs independent FMA chains for `iters` iterations and touches no
 * memory except `sink` (device, >= 12 bytes, may be NULL): the first CTA
 * writes the SM cycles and nanoseconds it ran to sink[0] and sink[1] (floats),
 * and sink[2] is written only in the unreachable case that a result equals a
 * sentinel.  `flags`, a combination of:
 *   HOC_PROBE_WHOLE_SM: threads must be 1024; 48 chains per thread (about 64
 *                  registers, the SM's whole register file for one CTA) and
 *                  nearly all shared memory reserved, so each CTA holds a whole
 *                  SM the way a GEMM tile does and any SM a collective kernel
 *                  occupies is lost to the probe.  Without it: 8 chains per
 *                  thread, small CTAs that can share an SM with other
 *                  kernels' CTAs.
 *   HOC_PROBE_PDL: launched with programmatic dependent launch allowed; the
 *                  kernel waits (griddepcontrol.wait) for the kernel before it
 *                  on the stream to finish before any FMA work, so only the
 *                  launch overlaps it -- the way back-to-back layer kernels
 *                  are launched to hide their launch latency.
 * ctas >= 1, 32 <= threads <= 1024 (a multiple of 32), iters >= 0; other
 * flag bits give HOC_ERR_INVALID_ARG. */
#define HOC_PROBE_WHOLE_SM 1
#define HOC_PROBE_PDL 2
hocResult_t hoc_probe_launch(void* stream, int ctas, int threads, int iters, int flags, float* sink);

/* out[i] = in[i] XOR key for `n` 16-bit words (device pointers; in == out is
 * allowed, other overlaps are not). */
hocResult_t hoc_xor16_launch(void* stream, const uint16_t* in, uint16_t* out, size_t n, uint16_t key);

/* Number of SMs of `device` (a query, no kernel). */
hocResult_t hoc_device_sm_count(int device, int* sms);

#ifdef __cplusplus
}
#endif

#endif /* HOC_WORKLOAD_H */
