// Collective scheduler: turns one collective call into a plan of steps.
//
// HOCCL section 3.4 (Fig. 6): a collective becomes a traffic matrix of flows,
// the flows are grouped into contention-free stages, and each flow is cut into
// fixed-size chunks that share the DMA-engine work queues.  Here a plan is an
// ordered list of steps; each step runs on one stream (0 = the caller's
// stream, 1..n = internal copy streams) and may wait on earlier steps of
// other streams.  Plans depend only on the shape of the call (op, k, counts,
// dtype, configuration), never on buffer addresses, so they are cached.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "hoc.h"
#include "hoc_internal.h"

namespace hoc {

struct Cfg {
  int path = HOC_PATH_AUTO;
  size_t chunk_bytes = 0;  // 0: by move path (chunk_for)
  int n_copy = 4;          // copy streams created per caller stream (the most a plan uses)
  int n_copy_auto = 0;     // 1: each plan picks its copy-queue count by copy size (copy_queues)
  int depth = 0;
  int reduce_max_sms = 0;
  int copy_max_sms = 0;
  int use_graphs = 1;
  int a2a_interleave = 1;
  int a2a_stage_sync = 0;
  std::vector<int> order;  // ring order, size k
  int reduce_engine = HOC_REDUCE_AUTO;
  int debug = 0;
  int fault = 0;           // host-side fault injection (Fault)
};

// Copy size of the all-gather, all-to-all and send/recv moves when the
// configuration leaves chunk_bytes at 0: 4 MiB on both move paths.
constexpr size_t kAutoChunkCe = size_t(4) << 20;
constexpr size_t kAutoChunkTma = size_t(4) << 20;
inline size_t chunk_for(const Cfg& cfg, int path) {
  return cfg.chunk_bytes ? cfg.chunk_bytes : (path == HOC_PATH_TMA ? kAutoChunkTma : kAutoChunkCe);
}


// Copy queues of a plan when the configuration leaves their number to the
// scheduler: copies are started back to back on each queue at about 4 us per
// dependent copy, so many small copies want more queues, while the cost of the
// moves to kernels running beside them grows with the bytes the queues hold in
// flight.  Measured on GB300 (8 ranks, HBM-resident): 8 queues against 4 lift
// all-gathers of 2 and 8 MB by 28-30 % and all-to-alls by 49-58 %, and change
// nothing from 32 MB (4 MiB copies) up; so 8 queues while every copy of the
// call is at most 2 MiB (no more bytes in flight than 4 queues of 4 MiB), else 4.
constexpr int kAutoQueuesSmall = 8;
constexpr int kAutoQueuesLarge = 4;
constexpr size_t kAutoSmallCopyBytes = size_t(2) << 20;
inline int copy_queues(const Cfg& cfg, size_t largest_copy) {
  if (!cfg.n_copy_auto) return cfg.n_copy;
  return largest_copy <= kAutoSmallCopyBytes ? kAutoQueuesSmall : kAutoQueuesLarge;
}

// Pipeline chunk of the copy-engine and TMA allreduce when the configuration
// leaves chunk_bytes at 0, by move path and rank count.  Each chunk costs a
// reduce kernel and a round of k(k-1) copies; with few ranks a chunk's kernel
// is small and its launch and tail show, with many the copies are many and
// small.  From sweeps of 1-64 MiB chunks (bf16, 16 / 64 / 256 MiB per rank,
// k = 2..16, GB300): copy engines want 32 MiB / k within 2-8 MiB, rounded down
// to a power of two (k = 2: 8 MiB, 0.180 ms at 256 MiB against 0.243 at 4 MiB;
// k = 9 and 12: 2 MiB on 8 queues, 1.12 and 1.69 ms against 1.20 and 1.77 at
// 3-4 MiB on 4; k = 16: 2 MiB, 0.490 ms at 64 MiB against 0.543), the TMA
// kernel 64 MiB / k^2 within 4-16 MiB (k = 2: 16 MiB, 0.199 ms at 256 MiB
// against 0.278).  The copy engines' chunk is
// also held to 16 MiB in flight over the queues one chunk's copies spread
// over -- what 4 queues of the 4 MiB all-gather copies hold: a compute kernel
// beside the moves slows with the bytes in flight (k = 4 keeps 4 MiB, which
// 8 MiB beat by at most 6 %).  A block smaller than the chunk is one chunk.
constexpr size_t kArChunkCeBytesTimesK = size_t(32) << 20;
constexpr size_t kArChunkTmaBytesTimesK2 = size_t(64) << 20;
constexpr size_t kArCeInFlightBytes = size_t(16) << 20;
constexpr size_t kArChunkMinBytes = size_t(2) << 20;  // the smallest chunk the scheduler picks
inline size_t allreduce_chunk(const Cfg& cfg, int path, int k) {
  if (cfg.chunk_bytes) return cfg.chunk_bytes;
  const size_t kk = size_t(k < 1 ? 1 : k);
  const size_t lo = kArChunkMinBytes;
  if (path == HOC_PATH_TMA)
    return std::min(size_t(16) << 20, std::max(size_t(4) << 20, kArChunkTmaBytesTimesK2 / (kk * kk)));
  size_t c = std::min(size_t(8) << 20, std::max(lo, kArChunkCeBytesTimesK / kk));
  while (c & (c - 1)) c &= c - 1;  // the power of two at or below
  const size_t spread = std::min(kk * (kk - 1), size_t(std::max(1, copy_queues(cfg, c))));
  if (spread > 0) c = std::min(c, std::max(lo, kArCeInFlightBytes / spread));
  return c;
}

// Chunks and pieces of moves are cut on multiples of this many bytes into
// the destination buffers.  A copy-engine copy whose destination starts off
// such a boundary runs slower throughout, while the source's offset costs
// little: an all-to-all of 4 MiB flows (8 ranks) took 0.122 ms aligned, 0.191
// ms with the destinations 16 B off, 0.408 ms 2 B off, and 0.122 / 0.147 ms
// with the sources 16 B / 2 B off; the copy-engine allreduce of 256 MiB bf16
// per rank at k = 6 took 1.046 ms with its blocks 32 B aligned and 0.699 ms
// with them 4 KiB aligned (64 KiB and 2 MiB: 0.699 and 0.688 ms).
constexpr size_t kCopyAlignBytes = 4096;

// Send/recv messages up to this size go as one copy on the caller's stream;
// larger ones are chunked and striped over the copy queues.
constexpr size_t kSendrecvStripeBytes = size_t(64) << 20;

enum Fault {
  kFaultNone = 0,
  kFaultDropChunk = 1,
  kFaultDupChunk = 2,
  kFaultWrongOrder = 3,
  kFaultProxyStall = 4,
  kFaultTmaStall = 5,   // the TMA kernel's mbarriers expect bytes that never arrive
  kFaultProxyBlock = 6,  // the proxy thread is held up past a task's deadline (host sleep)
  kFaultProxyMemop = 7,  // the first device-count call: its wait for FINISH fails to queue
  kFaultProxyMemopReset = 8  // the first device-count call: its reset of end_flag fails to queue
};

enum StepKind { kStepReduce = 0, kStepFused = 1, kStepCopy = 2, kStepTma = 3 };

struct Move {
  int src_rank, dst_rank;
  int src_buf, dst_buf;  // hocBuf_t
  size_t src_off, dst_off, bytes;
};

struct Step {
  int kind = kStepCopy;
  int stream = 0;
  int stage = 0;
  std::vector<ReduceSeg> segs;  // reduce / fused (vec is filled in at bind time)
  std::vector<Move> moves;      // copy / tma
  std::vector<int> waits;       // earlier steps on other streams
  bool record = false;          // some later step waits on this one
};

struct Plan {
  int op = 0, k = 0, dtype = 0, path = 0;
  size_t count = 0;
  int n_streams = 1;  // streams used including stream 0
  std::vector<Step> steps;
  size_t bytes_exec = 0, bytes_min = 0;
  int kernels = 0, copies = 0;
};

struct CallShape {
  int op = 0;
  int k = 0;
  int dtype = 0;
  size_t count = 0;
  std::vector<size_t> counts;  // alltoall: k*k sendcounts (elements); empty = uniform
  std::vector<size_t> sdispls, rdispls;
  int src_rank = 0, dst_rank = 0;  // sendrecv
  int path = -1;                   // allreduce: path override (-1: the communicator's)
  size_t chunk = 0;                // chunk override in bytes (0: the communicator's)
};

size_t dtype_bytes(int dtype);
int dtype_lanes(int dtype);  // elements per 16-byte vector

// The moves of a TMA step that read the same source bytes (same rank, buffer,
// offset and length), grouped in order of first appearance, at most kMaxRanks
// per group: the copy kernel loads such a group's bytes once and stores them to
// every destination (a broadcast job).
std::vector<std::vector<int>> source_groups(const std::vector<Move>& moves);

// Builds the plan; returns HOC_ERR_INVALID_ARG / UNSUPPORTED for bad shapes.
// Largest span of one rank's buffer a call may name (1 TiB, beyond any one
// device's memory) and most pipeline chunks one rank's span may be cut into:
// together they keep every size and offset sum far from overflow and the
// plan's host memory bounded.  build_plan rejects a shape past either with
// HOC_ERR_INVALID_ARG, before anything is issued.
constexpr uint64_t kMaxSpanBytes = uint64_t(1) << 40;
constexpr uint64_t kMaxChunksPerSpan = uint64_t(1) << 24;

// Builds the plan of a call shape.  Returns HOC_ERR_OOM (never throws) if the
// host runs out of memory while building it.
hocResult_t build_plan(const Cfg& cfg, const CallShape& shape, Plan* plan);

void set_error_detail(const char* what);

// Block partition of n elements over k owners (sizes differ by at most one).
void block_partition(size_t n, int k, std::vector<size_t>* sizes, std::vector<size_t>* offs);

// Order in which a copy queue serves the chunks of several flows.  Input: the
// chunk count of each flow.  Output: (flow, chunk) pairs.  Flow-size-aware:
// chunk j of flow f is due at virtual time (j + 1) / n_f and chunks are served
// in due order (ties by flow index), so every flow advances in proportion to
// its size.  FIFO: all chunks of flow 0, then flow 1, ...
std::vector<std::pair<int, size_t>> interleave_chunks(const std::vector<size_t>& chunks_per_flow, bool size_aware);

// Key that identifies a plan (shape + configuration).
std::string plan_key(const CallShape& s);

}  // namespace hoc
