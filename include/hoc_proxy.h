/*
 * hoc_proxy.h -- stream-memory-operation handshake with a host proxy.
 *
 * HOCCL section 3.2 (Fig. 4, Listing 1): the caller's GPU stream writes a start
 * flag in host memory and waits until the CPU proxy acknowledges it by writing
 * 0; the proxy then runs the communication and, when it has finished, writes a
 * finish value into an end flag that the stream waits for before resetting it.
 * The stream manager thereby orders host-driven communication between the
 * kernels before and after it without any SM and without blocking the
 * caller's thread.
 *
 * Here the proxy serves the one case where host-issued moves must wait for
 * GPU-side progress: an all-to-all(v) whose per-pair counts are computed on
 * the device (for example by an expert-routing kernel).  The counts travel to
 * the proxy through the handshake; the proxy plans the exchange (shift stages
 * and flow-size-aware chunk interleave, as hoc_alltoall) and issues it on copy
 * engines.  A watchdog in the proxy always writes the finish value, so no
 * stream waits forever: if the moves do not complete within the deadline, or
 * the counts are invalid, the stream is released and hoc_proxy_status() /
 * hoc_wait() report the error.  The flags live in mapped pinned host memory
 * and the stream operations are cuStreamWriteValue32 / cuStreamWaitValue32.
 *
 * Hardware queues: a stream held at a wait blocks the hardware work queue it
 * was mapped to, and with it every other stream mapped to that queue (CUDA
 * maps streams onto CUDA_DEVICE_MAX_CONNECTIONS queues in creation order, so
 * with many streams alive some always share one).  Before acknowledging a
 * task, while the caller's stream is held at the start flag, the proxy records
 * a probe event on each of its own candidate streams and issues the moves only
 * on streams whose probe completed.  If too few clear within 0.5 s (up to 64
 * candidates) the task is released with HOC_ERR_UNSUPPORTED and nothing moves.
 */
#ifndef HOC_PROXY_H
#define HOC_PROXY_H

#include <stddef.h>
#include <stdint.h>

#include "hoc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* All-to-all(v) with device-resident counts.  d_sendcounts: device array of
 * k*k uint64 element counts (row = source), valid when the work before this
 * call on `stream` has finished; with transpose != 0 the matrix is read
 * transposed (row = destination), so the counts of a dispatch serve the
 * inverse exchange (the combine) unchanged.  recv_capacity: host array of k element
 * capacities of the receive buffers (the counts are unknown at call time);
 * if a receiver's total exceeds its capacity nothing is moved and the error is
 * reported.  Displacements are prefix sums in rank order.  Returns as soon as
 * the handshake is queued on `stream`; later work on `stream` sees the moved
 * data.  The first call starts the proxy thread and allocates its pinned host
 * flags.  Not allowed while `stream` is being captured into a graph. */
hocResult_t hoc_alltoall_device_counts(hocComm_t comm, const void* const* send, void* const* recv,
                                       const uint64_t* d_sendcounts, int transpose, const size_t* recv_capacity,
                                       hocDataType_t dtype, void* stream);

/* Proxy bookkeeping: tasks completed, tasks released by the watchdog or an
 * error, and the first error code seen (then cleared). */
hocResult_t hoc_proxy_status(hocComm_t comm, uint64_t* completed, uint64_t* released_on_error,
                             hocResult_t* first_error);

/* Stream probing (see "Hardware queues" above): the proxy's candidate streams
 * so far, and how many probes it found still pending when it picked streams
 * (each is a candidate skipped because its queue was held or busy). */
hocResult_t hoc_proxy_queue_stats(hocComm_t comm, uint64_t* candidates, uint64_t* probes_not_clear);

#ifdef __cplusplus
}
#endif

#endif /* HOC_PROXY_H */
