/*
 * hoc.h -- zero-SM collective schedules over k simulated ranks on one GPU.
 *
 * Operations follow "HOCCL: Offloading Collective Communication from GPU Cores
 * to Accelerate Distributed Training":
 *   - the stream manager (section 3.2, Fig. 4) orders each collective against
 *     the kernels before and after it on the caller's stream;
 *   - the point-to-point executor (section 3.3) moves every chunk as one
 *     direct copy into the receiver's buffer, on copy engines (zero SMs) or,
 *     for comparison, on a TMA bulk-copy kernel (SM-driven);
 *   - the collective scheduler (section 3.4, Fig. 6) splits flows into chunks,
 *     orders all-to-all flows into contention-free shift stages (Eq. 6-8) and
 *     interleaves chunks in proportion to flow size on each copy queue.
 * Reductions (AllReduce, ReduceScatter) are outside the paper's zero-SM scope
 * (section 5, Limitations); here their arithmetic runs in a k-way reduce
 * kernel that folds each block in ring order (see hoc_allreduce).
 *
 * Conventions for every call:
 *   - Rank buffers are device pointers on the communicator's device, one per
 *     simulated rank, owned by the caller.  Pointer arrays are host arrays
 *     read during the call and not retained.
 *   - Counts are in elements of `dtype`; a count of 0 is a successful no-op.
 *     No rank buffer a call names may span more than 2^40 bytes, and no rank
 *     buffer may be cut into more than 2^24 chunks of `chunk_bytes`; past
 *     either limit the call returns HOC_ERR_INVALID_ARG and issues nothing.
 *   - Work is ordered after all prior work on `stream` and later work on
 *     `stream` sees the results.  Calls never block the host (except the
 *     first call of a new shape in graph mode, which builds a CUDA graph).
 *     `stream` is a cudaStream_t; NULL is the legacy default stream.
 *   - Errors are return codes; nothing is thrown across the ABI.  Errors of
 *     asynchronous work show up in a later call or in hoc_wait().
 *   - Buffers of different ranks must not overlap, except the in-place forms
 *     stated per call.  Any alignment is accepted; 16-byte-aligned buffers
 *     take the vector / bulk-copy paths, others the scalar paths.
 */
#ifndef HOC_H
#define HOC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HOC_MAX_RANKS 16

typedef enum {
  HOC_SUCCESS = 0,
  HOC_ERR_INVALID_ARG = 1,     /* bad rank count, pointer, size, dtype, op, alias */
  HOC_ERR_CUDA = 2,            /* a CUDA call failed; hoc_last_error_detail() says which */
  HOC_ERR_OOM = 3,             /* host or device allocation failed */
  HOC_ERR_NOT_INITIALIZED = 4, /* NULL communicator */
  HOC_ERR_UNSUPPORTED = 5,     /* valid request this build does not implement */
  HOC_ERR_TIMEOUT = 6,         /* a bounded wait (host or device) gave up */
  HOC_ERR_NO_DEVICE = 7        /* no usable CUDA device */
} hocResult_t;

typedef enum { HOC_INT32 = 0, HOC_FLOAT32 = 1, HOC_BFLOAT16 = 2, HOC_UINT8 = 3 } hocDataType_t;
typedef enum { HOC_SUM = 0 } hocRedOp_t;

/* How chunk moves are executed. */
typedef enum {
  HOC_PATH_AUTO = 0,  /* allreduce -> FUSED (CE under an SM budget, reduce_max_sms > 0); moves -> CE */
  HOC_PATH_CE = 1,    /* cudaMemcpyAsync on internal copy streams: zero SMs */
  HOC_PATH_TMA = 2,   /* cp.async.bulk kernel: SM-driven comparison path */
  HOC_PATH_FUSED = 3  /* allreduce only: one kernel reduces and writes all k outputs */
} hocPath_t;

/* How the k-way reduce kernel moves its bytes. */
typedef enum {
  HOC_REDUCE_AUTO = 0, /* LSU (measured faster on GB300 with and without an SM budget) */
  HOC_REDUCE_LSU = 1,  /* every thread issues 16-byte vector loads and stores */
  HOC_REDUCE_TMA = 2   /* bulk async copies through shared memory; one CTA per SM */
} hocReduceEngine_t;

/* Communicator configuration; hoc_config_default() fills the defaults.
 * Environment variables HOC_PATH (ce|tma|fused|auto), HOC_CHUNK_BYTES,
 * HOC_COPY_STREAMS, HOC_USE_GRAPHS, HOC_REDUCE_MAX_SMS, HOC_REDUCE_ENGINE
 * (lsu|tma|auto), HOC_DEBUG override the values passed in. */
typedef struct {
  int path;              /* hocPath_t */
  size_t chunk_bytes;    /* pipeline unit inside a block / flow; 0 (default): the scheduler
                            picks -- allreduce chunks by move path and rank count k (copy
                            engines 32 MiB / k within 2-8 MiB, a power of two, at most 16 MiB in flight
                            over the copy queues, TMA kernel 64 MiB / k^2 within 4-16 MiB),
                            4 MiB copies for the other collectives */
  int n_copy_streams;    /* internal copy streams (the multi-QP analogue), max 16; 0 (default):
                            the scheduler picks per call -- 8 while every copy of the call is at
                            most 2 MiB (small messages: per-copy startup dominates), else 4.
                            They run at the default stream priority, the lowest: a caller's
                            compute stream created with a higher priority gets its kernel
                            launches served ahead of the moves' work, which keeps the moves'
                            cost to short compute kernels beside them lowest */
  int pipeline_depth;    /* allreduce CE/TMA: reduce of chunk q waits for the moves of
                            chunk q - depth; 0 = no limit */
  int reduce_max_sms;    /* cap on CTAs of reduce kernels (one 1024-thread CTA per SM); 0 = whole GPU */
  int copy_max_sms;      /* CTAs of the TMA copy kernel; 0 = whole GPU */
  int use_graphs;        /* 1: cache each call's issue sequence as a CUDA graph and replay it */
  int a2a_interleave;    /* 1: flow-size-aware chunk interleave per copy queue; 0: per-flow FIFO */
  int a2a_stage_sync;    /* 1: all copy queues join between all-to-all shift stages */
  const int* ring_order; /* k ranks in ring order (a permutation); NULL = identity; copied */
  int reduce_engine;     /* hocReduceEngine_t */
} hocConfig_t;

typedef struct hocComm* hocComm_t;

/* Statistics of the last collective issued on a communicator. */
typedef struct {
  int path;             /* path actually taken (hocPath_t) */
  int kernels;          /* kernels of this library launched by the call */
  int copies;           /* copy-engine copies issued by the call */
  int max_ctas;         /* largest grid among those kernels */
  int sms_used;         /* SMs those kernels can occupy: min(max_ctas, SM count); 0 on pure CE */
  int graph_replayed;   /* 1 if the call replayed a cached CUDA graph */
  size_t bytes_exec;    /* algorithmic HBM bytes of the executed schedule */
  size_t bytes_min;     /* lower bound: read every input and write every output once */
} hocOpStats_t;

/* Kernel classes for hoc_profile_read(). */
typedef enum { HOC_KERNEL_REDUCE = 0, HOC_KERNEL_FUSED = 1, HOC_KERNEL_TMA = 2 } hocKernel_t;

/* Fill `cfg` with the defaults listed in hocConfig_t. Never fails for non-NULL cfg. */
hocResult_t hoc_config_default(hocConfig_t* cfg);

/* Create a communicator for `nranks` (1..HOC_MAX_RANKS) simulated ranks on CUDA
 * device `device`.  `cfg` may be NULL (defaults).  The communicator owns its
 * internal streams, events, plan and graph caches and a small device status
 * buffer.  Returns HOC_ERR_NO_DEVICE without a GPU. */
hocResult_t hoc_init(hocComm_t* comm, int nranks, int device, const hocConfig_t* cfg);

/* Wait for the communicator's internal work, then free everything it owns. */
hocResult_t hoc_destroy(hocComm_t comm);

/* AllReduce (sum).  send[r], recv[r]: `count` elements each.  Each rank buffer
 * is split into k blocks, B_r = floor(count/k) + (r < count mod k) elements,
 * owned by rank r.  Block r is folded in ring order: start from rank succ(r),
 * add succ^2(r), ..., end with r's own input (textbook ring reduce-scatter
 * hop order; succ follows cfg.ring_order).  fp32 adds in binary32 with round to
 * nearest even; bf16 widens to binary32, adds in binary32 and rounds once to
 * bf16; int32 wraps modulo 2^32.  Every rank then receives every block (ring
 * all-gather, section 6.2 "AllGather").  In place: send[r] == recv[r]. */
hocResult_t hoc_allreduce(hocComm_t comm, const void* const* send, void* const* recv, size_t count,
                          hocDataType_t dtype, hocRedOp_t op, void* stream);

/* AllReduce over HOST buffers: h_send[r], h_recv[r] are host pointers.  Same
 * fold and bits as hoc_allreduce.  Two modes:
 *  - direct (cfg.path AUTO or FUSED, when the device can address every buffer:
 *    pinned memory, or pageable memory on a device with pageable memory access
 *    such as a Grace-attached GPU): one fused reduce launch loads the inputs
 *    from host memory and stores the results there; no staging, no copies.
 *    With cfg.path FUSED and a buffer the device cannot address, the call
 *    returns HOC_ERR_UNSUPPORTED.
 *  - staged (cfg.path CE or TMA, or AUTO with a buffer the device cannot
 *    address): the element range is cut into 8 MiB chunks per rank; the
 *    host->device copies of chunk q+1, the reduce of chunk q and the
 *    device->host copies of chunk q-1 overlap on copy engines and SMs, through
 *    two device staging slots the communicator allocates on first use.  Calls
 *    that run at the same time on the GPU (different streams without ordering
 *    between them) share those slots and race.
 * Stream-ordered like every call; in place: h_send[r] == h_recv[r]. */
hocResult_t hoc_allreduce_host(hocComm_t comm, const void* const* h_send, void* const* h_recv, size_t count,
                               hocDataType_t dtype, hocRedOp_t op, void* stream);

/* ReduceScatter (sum).  send[r] holds k*recvcount elements, recv[r] recvcount.
 * recv[r] = block r of the fold above (block size recvcount for every rank).
 * In place: recv[r] == (elem*)send[r] + r*recvcount. */
hocResult_t hoc_reduce_scatter(hocComm_t comm, const void* const* send, void* const* recv,
                               size_t recvcount, hocDataType_t dtype, hocRedOp_t op, void* stream);

/* AllGather (section 6.2, "AllGather").  recv[d][r*sendcount ...] = send[r][0 .. sendcount).
 * In place: send[r] == (elem*)recv[r] + r*sendcount. */
hocResult_t hoc_allgather(hocComm_t comm, const void* const* send, void* const* recv,
                          size_t sendcount, hocDataType_t dtype, void* stream);

/* All-to-all(v) (section 6.2 "All-to-All"; traffic matrix C of section 3.4).
 * sendcounts: k*k host array, row = source: rank s sends sendcounts[s*k+d]
 * elements from send[s] + sdispls[s*k+d] to recv[d] + rdispls[d*k+s].
 * sendcounts == NULL means the uniform exchange of `count_if_uniform`
 * elements per pair.  sdispls / rdispls == NULL mean prefix sums in rank
 * order.  Receive regions must not overlap each other or any send region. */
hocResult_t hoc_alltoall(hocComm_t comm, const void* const* send, const size_t* sendcounts,
                         const size_t* sdispls, void* const* recv, const size_t* rdispls,
                         size_t count_if_uniform, hocDataType_t dtype, void* stream);

/* Send/recv (section 3.3.2): move `count` elements from rank src_rank's buffer
 * `send` into rank dst_rank's buffer `recv` with one direct copy on `stream`
 * (messages above 64 MiB are split into chunks striped over the copy queues).
 * src_rank may equal dst_rank. */
hocResult_t hoc_sendrecv(hocComm_t comm, int src_rank, const void* send, int dst_rank, void* recv,
                         size_t count, hocDataType_t dtype, void* stream);

/* Send/recv whose completion is signalled by an event instead of the caller's
 * stream (HOCCL section 3.2: the stream manager orders communication against
 * the kernels around it with events).  The copy waits for the work issued on
 * `stream` before this call, runs on one of the communicator's copy streams
 * (consecutive calls rotate over them) and records `done_event`, a
 * cudaEvent_t the caller created, when the data is in `recv`.  Later work on
 * `stream` does NOT wait for it, so the sender keeps computing while the copy
 * engine moves the data; consumers wait on `done_event`.  The caller leaves
 * `send` unchanged and does not touch `recv` until `done_event` has completed.
 * With nothing to move, `done_event` is recorded on `stream`.  Not allowed
 * while `stream` is being captured into a graph (HOC_ERR_UNSUPPORTED). */
hocResult_t hoc_sendrecv_async(hocComm_t comm, int src_rank, const void* send, int dst_rank, void* recv,
                               size_t count, hocDataType_t dtype, void* stream, void* done_event);

/* Bounded host wait: polls until all work on `stream` (and the communicator's
 * internal streams) has finished, or `timeout_ms` ms pass (HOC_ERR_TIMEOUT).
 * Also reports device-side timeouts of the TMA copy kernel (HOC_ERR_TIMEOUT). */
hocResult_t hoc_wait(hocComm_t comm, void* stream, int timeout_ms);

/* Statistics of the last collective issued on `comm`. */
hocResult_t hoc_last_stats(hocComm_t comm, hocOpStats_t* stats);

/* Per-kernel timing.  While enabled, every kernel this communicator launches
 * is bracketed by CUDA events on the stream it is launched on (graphs are not
 * used while enabled).  hoc_profile_read() waits for those events and returns,
 * for one kernel class, the number of launches and their summed duration in
 * milliseconds since the last read, then clears that class. */
hocResult_t hoc_profile_enable(hocComm_t comm, int enable);
hocResult_t hoc_profile_read(hocComm_t comm, hocKernel_t kernel, int* launches, double* total_ms);

/* Per-stream finish times of the last call issued while profiling was
 * enabled, when it forked onto internal copy streams: finish_ms[i] = time from
 * the fork on the caller's stream to the end of copy stream i's last
 * operation, for i < min(*n_streams, max_streams).  Waits for those events.
 * *n_streams = 0 if the last profiled call ran on the caller's stream alone.
 * Their spread is the schedule's tail: how unevenly the moves were spread
 * over the copy engines (HOCCL section 3.3 on skewed all-to-all flows). */
hocResult_t hoc_profile_stream_finish(hocComm_t comm, float* finish_ms, int max_streams, int* n_streams);

/* Per-step timeline of the last call issued while profiling was enabled: one
 * item per plan step (a reduce or fused kernel, a bulk-copy kernel, or the
 * copy-engine copies of one copy queue for one chunk), in issue order, with
 * start and end in milliseconds from the moment the caller's stream reached
 * the call.  A step's start is recorded on its stream after the waits it
 * depends on, so start..end is when the step could run and when it finished.
 * Waits for those events.  Writes at most `cap` items; *n_items = all of them.
 * Used to see how the chunks of a pipelined allreduce overlap (HOCCL section
 * 3.3.1 on chunk pipelining).  A profiled call that the caller captures into a
 * CUDA graph records these events as external event nodes: after a replay of
 * that graph, this call returns the replay's timeline. */
typedef struct {
  int kind;     /* hocItemKind_t: HOC_ITEM_REDUCE, HOC_ITEM_FUSED, HOC_ITEM_COPY or HOC_ITEM_TMA */
  int stream;   /* 0 = caller stream, 1..n = internal copy streams */
  int stage;    /* chunk index (allreduce, allgather) or shift stage (alltoall) */
  float start_ms;
  float end_ms;
} hocStepTime_t;
hocResult_t hoc_profile_timeline(hocComm_t comm, hocStepTime_t* items, size_t cap, size_t* n_items);

/* Static description of a result code. */
const char* hoc_error_string(hocResult_t result);

/* Text of the last CUDA or argument error seen by this process (thread-local). */
const char* hoc_last_error_detail(void);

/* ---------------------------------------------------------------------------
 * Allocation-free moves.  The paper has no counterpart to this call.
 *
 * Everything above needs a communicator, and hoc_init allocates device memory
 * (a status word for the bulk-copy kernel's bounded waits).  Some callers
 * cannot call cudaMalloc: a plug-in running inside a runtime that has already
 * claimed the device's memory with its own allocator, code that must not own
 * device memory, or a step that must not risk the device-wide
 * synchronisation cudaMalloc / cudaFree can cause.  hoc_tma_moves_noalloc
 * moves `n` byte ranges, src[i] -> dst[i] of bytes[i] bytes (device pointers
 * on the current device, any alignment), with the TMA bulk-copy kernel and
 * allocates nothing: its scratch is a file-scope device array of
 * HOC_NOALLOC_SCRATCH_BYTES (256) bytes that every GPU loading the library
 * holds until the process exits.
 *   - At most HOC_NOALLOC_MAX_MOVES moves per call (what one launch's
 *     parameters carry); more returns HOC_ERR_INVALID_ARG.  A move whose
 *     source and destination overlap, a non-empty move with a NULL pointer and
 *     a move of more than 2^40 bytes are rejected the same way, before
 *     anything is queued.
 *   - The first call on a device sets that device up (kernel attributes and
 *     the scratch array's device address); make that first call before any
 *     stream capture.
 *   - All calls share the scratch array: calls that overlap on the GPU (on
 *     different streams without ordering between them) race on it.  Each call
 *     clears it on `stream` before its launch.
 *   - max_ctas caps the kernel's CTAs (0 = one per SM).  With wait != 0 the
 *     call waits for `stream` and returns HOC_ERR_TIMEOUT if a bounded wait in
 *     the kernel gave up; with wait == 0 it returns once the work is queued.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 * ------------------------------------------------------------------------- */
#define HOC_NOALLOC_MAX_MOVES 192
#define HOC_NOALLOC_SCRATCH_BYTES 256
hocResult_t hoc_tma_moves_noalloc(const void* const* src, void* const* dst, const size_t* bytes, int n,
                                  int max_ctas, void* stream, int wait);

/* ---------------------------------------------------------------------------
 * Plan introspection (host only, needs no GPU).  Builds the plan a
 * communicator with `cfg` would execute and returns it as a flat item list:
 * one item per reduce segment, per copy, or per join.  Used to test the
 * scheduler on machines without a GPU.
 * ------------------------------------------------------------------------- */
typedef enum { HOC_OP_ALLREDUCE = 0, HOC_OP_REDUCE_SCATTER = 1, HOC_OP_ALLGATHER = 2,
               HOC_OP_ALLTOALL = 3, HOC_OP_SENDRECV = 4 } hocOp_t;
typedef enum { HOC_ITEM_REDUCE = 0, HOC_ITEM_FUSED = 1, HOC_ITEM_COPY = 2, HOC_ITEM_TMA = 3,
               HOC_ITEM_JOIN = 4 } hocItemKind_t;
typedef enum { HOC_BUF_SEND = 0, HOC_BUF_RECV = 1 } hocBuf_t;

typedef struct {
  int kind;       /* hocItemKind_t */
  int step;       /* index of the launch / copy step the item belongs to */
  int stream;     /* 0 = caller stream, 1..n = internal copy streams */
  int stage;      /* chunk index (allreduce, allgather) or shift stage (alltoall) */
  int src_rank;   /* REDUCE/FUSED: -1 (all ranks are read) */
  int dst_rank;   /* REDUCE/FUSED: block owner; FUSED writes every rank */
  int src_buf;    /* hocBuf_t */
  int dst_buf;    /* hocBuf_t */
  size_t src_off; /* bytes from the start of the source rank buffer */
  size_t dst_off; /* bytes from the start of the destination rank buffer */
  size_t bytes;
  int n_waits;    /* number of earlier steps this step waits on (cross-stream) */
  int wait0;      /* first of them, -1 if none */
} hocPlanItem_t;

/* `op` is hocOp_t; `count` as in the matching call (recvcount for reduce
 * scatter, sendcount for allgather, count_if_uniform for alltoall, count for
 * sendrecv); `counts` is the k*k sendcounts matrix for alltoall or NULL.
 * For sendrecv, src/dst ranks are 0 and 1 % nranks.  Writes at most `cap`
 * items to `items` (may be NULL) and the full count to `n_items`. */
hocResult_t hoc_plan_query(int nranks, const hocConfig_t* cfg, int op, size_t count,
                           hocDataType_t dtype, const size_t* counts, hocPlanItem_t* items,
                           size_t cap, size_t* n_items);

#ifdef __cplusplus
}
#endif

#endif /* HOC_H */
