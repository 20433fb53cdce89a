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
 * engines, in chunks of at least total bytes / 48 so that issuing the copies,
 * which starts only when the stream reaches the flag, takes no longer than
 * moving them.  A watchdog in the proxy always writes the finish value, so no
 * stream waits forever: if the moves do not complete within the deadline, or
 * the counts are invalid, the stream is released and hoc_proxy_status() /
 * hoc_wait() report the error.  The flags live in mapped pinned host memory
 * and the stream operations are cuStreamWriteValue32 / cuStreamWaitValue32.
 *
 * Held-stream window: from the start flag to the end flag the caller's
 * stream is held, and the moves must run meanwhile.  Three things stall them
 * until the stream is released: a proxy copy stream that shares the held
 * stream's hardware work queue (CUDA maps streams onto
 * CUDA_DEVICE_MAX_CONNECTIONS queues, 8 by default; the wait blocks its whole
 * queue -- on GB300 about 3 in 10 fresh processes hit it at 8 queues, none in
 * 8 at 32, all at 1: run with CUDA_DEVICE_MAX_CONNECTIONS=32, set before the
 * process starts CUDA); launching a kernel for the first time under lazy
 * module loading (CUDA_MODULE_LOADING=LAZY, the default; the load can wait for
 * the whole context, the held stream included); and a pageable host copy
 * queued behind the held stream.  The library loads all of its own kernels
 * before the proxy starts; load other kernels that run during the window
 * beforehand (one warm-up launch, or CUDA_MODULE_LOADING=EAGER) and keep
 * blocking host copies off the held stream.  Should a stall happen
 * anyway, the proxy's watchdog -- a host thread that makes no CUDA call --
 * releases the stream after 10 s and the call reports HOC_ERR_TIMEOUT with the
 * reason; no stream is left waiting and no thread deadlocks.
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
 * inverse exchange (the combine) unchanged.  send_capacity / recv_capacity:
 * host arrays of k element capacities of the send and receive buffers (the
 * counts are unknown at call time); if a sender's row total exceeds its send
 * capacity, or a receiver's column total its receive capacity, nothing is
 * moved and the error (HOC_ERR_INVALID_ARG) is reported by hoc_wait.  The
 * totals are compared without overflow.  Displacements are prefix sums in
 * rank order.  Returns as soon as the handshake is queued on `stream`; later
 * work on `stream` sees the moved data.  The first call starts the proxy
 * thread and allocates its pinned host flags.  Not allowed while `stream` is
 * being captured into a graph.  If the stream operations cannot all be
 * queued, the call returns HOC_ERR_CUDA and moves nothing; the proxy lets the
 * stream pass whatever flags it did queue. */
hocResult_t hoc_alltoall_device_counts(hocComm_t comm, const void* const* send, void* const* recv,
                                       const uint64_t* d_sendcounts, int transpose, const size_t* send_capacity,
                                       const size_t* recv_capacity, hocDataType_t dtype, void* stream);

/* Proxy bookkeeping: tasks completed, tasks released by the watchdog or an
 * error, and the first error code seen (then cleared). */
hocResult_t hoc_proxy_status(hocComm_t comm, uint64_t* completed, uint64_t* released_on_error,
                             hocResult_t* first_error);

#ifdef __cplusplus
}
#endif

#endif /* HOC_PROXY_H */
