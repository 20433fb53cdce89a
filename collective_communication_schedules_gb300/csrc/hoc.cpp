// C ABI of the collective library: communicator, stream manager and
// point-to-point executor.
//
// Stream manager (HOCCL section 3.2, Fig. 4): the paper keeps communication
// ordered against the kernels before and after it on a GPU stream through a
// CPU-GPU flag handshake.  On one GPU the same ordering comes from CUDA
// events: the caller's stream records a fork event that the internal copy
// streams wait on, cross-stream plan edges are event waits, and the caller's
// stream waits on a join event of every internal stream.  No host thread ever
// blocks, and no device-side wait is unbounded.  hoc_sendrecv_async skips the
// join and completes a caller's event instead.  The one call whose sizes the
// host cannot know, an all-to-all with device-computed counts, uses the
// paper's flag handshake with a host proxy (proxy.cpp).
//
// P2P executor (section 3.3): a move is one cudaMemcpyAsync on an internal
// copy stream (copy engines, zero SMs) or a job of the TMA bulk-copy kernel.
// Chunks striped over several copy streams play the role of the paper's
// multi-QP striping (section 3.3.1): several chunks in flight hide per-copy
// startup latency.  Each call's issue sequence can be captured once as a CUDA
// graph and replayed, which removes the per-chunk host launch cost the paper
// measures in Fig. 9.
#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <list>
#include <mutex>
#include <string>
#include <thread>
#include <unordered_map>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "comm.h"
#include "hoc.h"
#include "hoc_internal.h"
#include "plan.h"

namespace hoc {
namespace {

thread_local std::string g_detail;

void set_detail(const char* what, cudaError_t e) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s (%d)", what, cudaGetErrorString(e), int(e));
  g_detail = buf;
}
void set_detail(const char* what) { g_detail = what; }

#define HOC_CK(call)                  \
  do {                                \
    cudaError_t e_ = (call);          \
    if (e_ != cudaSuccess) {          \
      set_detail(#call, e_);          \
      return HOC_ERR_CUDA;            \
    }                                 \
  } while (0)

#define HOC_TRY(expr)                 \
  do {                                \
    hocResult_t r_ = (expr);          \
    if (r_ != HOC_SUCCESS) return r_; \
  } while (0)

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

int env_int(const char* name, int dflt) {
  const char* v = getenv(name);
  return v && *v ? atoi(v) : dflt;
}

}  // namespace

}  // namespace hoc

namespace hoc {
namespace {

constexpr size_t kMaxGraphs = 64;
constexpr uint64_t kReduceWaves = 8;
constexpr size_t kMaxStreamSets = 16;

// The copy streams serving caller stream `s0` (created on first use).
hocResult_t copy_streams_for(hocComm* c, cudaStream_t s0, std::vector<cudaStream_t>** out) {
  for (auto& set : c->sets)
    if (set.owner == s0) {
      *out = &set.copy;
      return HOC_SUCCESS;
    }
  if (c->sets.size() >= kMaxStreamSets) {
    // more caller streams than sets: share one (still correct, may serialise)
    *out = &c->sets[reinterpret_cast<uintptr_t>(s0) % c->sets.size()].copy;
    return HOC_SUCCESS;
  }
  hocComm::StreamSet set;
  set.owner = s0;
  for (int i = 0; i < c->cfg.n_copy; ++i) {
    cudaStream_t s;
    HOC_CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    set.copy.push_back(s);
  }
  c->sets.push_back(std::move(set));
  *out = &c->sets.back().copy;
  return HOC_SUCCESS;
}

hocResult_t get_event(hocComm* c, std::vector<cudaEvent_t>& pool, size_t i) {
  while (pool.size() <= i) {
    cudaEvent_t e;
    HOC_CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    pool.push_back(e);
  }
  (void)c;
  return HOC_SUCCESS;
}

hocResult_t prof_event(hocComm* c, cudaEvent_t* e) {
  if (!c->prof_free.empty()) {
    *e = c->prof_free.back();
    c->prof_free.pop_back();
    return HOC_SUCCESS;
  }
  HOC_CK(cudaEventCreate(e));
  return HOC_SUCCESS;
}

int ctas_per_sm(hocComm* c, int dtype, int k, int broadcast) {
  int& v = c->reduce_ctas_per_sm[dtype == HOC_BFLOAT16 ? 2 : dtype == HOC_FLOAT32 ? 1 : 0][k][broadcast];
  if (v == 0) v = reduce_ctas_per_sm(dtype, k, broadcast);
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernel launch with optional timing events and debug checks.
template <class F>
hocResult_t timed_launch(hocComm* c, int kind, cudaStream_t s, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  unsigned flags = cudaEventRecordDefault;  // external event nodes when the caller captures the call
  if (c->profiling) {
    HOC_TRY(prof_event(c, &a));
    HOC_TRY(prof_event(c, &b));
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    HOC_CK(cudaStreamIsCapturing(s, &cap));
    if (cap != cudaStreamCaptureStatusNone) flags = cudaEventRecordExternal;
    HOC_CK(cudaEventRecordWithFlags(a, s, flags));
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) {
    set_detail("kernel launch", e);
    return HOC_ERR_CUDA;
  }
  if (c->profiling) {
    HOC_CK(cudaEventRecordWithFlags(b, s, flags));
    c->prof_pending.push_back(ProfPair{a, b, kind});
  }
  if (c->cfg.debug) {
    HOC_CK(cudaStreamSynchronize(s));
    HOC_CK(cudaGetLastError());
  }
  return HOC_SUCCESS;
}

const void* buf_ptr(const Bind& b, int rank, int which) {
  return which == HOC_BUF_SEND ? b.send[rank] : b.recv[rank];
}

hocResult_t run_reduce(hocComm* c, const Plan& p, const Step& st, const Bind& bd, cudaStream_t s, int* max_ctas) {
  ReduceParams rp;
  memset(&rp, 0, sizeof rp);
  const int k = p.k;
  rp.k = k;
  rp.dtype = p.dtype;
  rp.broadcast = st.kind == kStepFused ? 1 : 0;
  const int lanes = dtype_lanes(p.dtype);
  const size_t b = dtype_bytes(p.dtype);
  bool bases_aligned = true;
  for (int r = 0; r < k; ++r) {
    rp.in[r] = bd.send[r];
    rp.out[r] = bd.recv[r];
    bases_aligned = bases_aligned && aligned16(bd.send[r]) && aligned16(bd.recv[r]);
  }
  // operand order of block `owner`: succ(owner), succ^2(owner), ..., owner
  std::vector<int> pos(k);
  for (int i = 0; i < k; ++i) pos[c->cfg.order[i]] = i;
  for (int o = 0; o < k; ++o)
    for (int j = 0; j < k; ++j) rp.seq[o][j] = uint8_t(c->cfg.order[(pos[o] + 1 + j) % k]);
  rp.nseg = int(st.segs.size());
  bool all_vec = true;
  for (int i = 0; i < rp.nseg; ++i) {
    ReduceSeg g = st.segs[i];
    g.vec = (bases_aligned && (g.out_off % lanes) == (g.elem_off % lanes)) ? 1u : 0u;
    all_vec = all_vec && g.vec;
    rp.seg[i] = g;
  }
  (void)b;
  const int budget = c->cfg.reduce_max_sms;
  int engine = c->cfg.reduce_engine;
  if (engine == HOC_REDUCE_AUTO) engine = HOC_REDUCE_LSU;  // measured faster in both shapes
  const bool wide = budget > 0;  // one CTA per SM: the 1024-thread shape
  if (!all_vec) engine = HOC_REDUCE_LSU;  // bulk copies need co-aligned 16-byte rows
  rp.tile_start[0] = 0;
  for (int i = 0; i < rp.nseg; ++i)
    rp.tile_start[i + 1] = rp.tile_start[i] + (engine == HOC_REDUCE_TMA ? reduce_tma_seg_tiles(p.dtype, rp.seg[i], k)
                                                                       : reduce_seg_tiles(p.dtype, rp.seg[i], wide));
  const uint64_t tiles = rp.tile_start[rp.nseg];
  if (tiles == 0) return HOC_SUCCESS;
  const int kind = rp.broadcast ? HOC_KERNEL_FUSED : HOC_KERNEL_REDUCE;
  if (engine == HOC_REDUCE_TMA) {
    const uint64_t cap = uint64_t(budget > 0 ? std::min(budget, c->sms) : c->sms);
    const int grid = int(std::min<uint64_t>(tiles, cap));
    *max_ctas = std::max(*max_ctas, grid);
    const bool stall = c->cfg.fault == kFaultTmaStall;  // host-injected: mbarriers that never complete
    return timed_launch(c, kind, s, [&] {
      return launch_reduce_tma(rp, grid, c->status, s, stall ? 16u : 0u, stall ? 100000000ull : 2000000000ull);
    });
  }
  // Whole GPU: several waves of CTAs rather than one persistent wave, so a CTA
  // that finishes its tiles is replaced at once and loads keep streaming.
  uint64_t cap;
  if (budget > 0) cap = uint64_t(std::min(budget, c->sms));
  else cap = uint64_t(c->sms) * ctas_per_sm(c, p.dtype, k, rp.broadcast) * kReduceWaves;
  const int grid = int(std::min<uint64_t>(tiles, cap));
  *max_ctas = std::max(*max_ctas, grid);
  const bool overlap = !wide && uint64_t(grid) > uint64_t(c->sms) * ctas_per_sm(c, p.dtype, k, rp.broadcast);
  return timed_launch(c, kind, s, [&] { return launch_reduce(rp, grid, wide, s, overlap); });
}

// The copy jobs of a TMA step: one job per group of moves that read the same
// source (source_groups), all of whose destinations share the job's
// alignment class (co-aligned with the source modulo 16, or not); a member in
// the other class gets a job of its own.  `more[i]` lists job i's destinations
// beyond the first.
void tma_jobs(const Step& st, const Bind& bd, std::vector<CopyJob>* jobs, std::vector<std::vector<char*>>* more) {
  auto co = [](const char* a, const char* b) {
    return ((reinterpret_cast<uintptr_t>(a) ^ reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
  };
  for (const auto& g : source_groups(st.moves)) {
    const size_t first = jobs->size();  // jobs of this group start here
    for (int idx : g) {
      const Move& m = st.moves[idx];
      const char* src = static_cast<const char*>(buf_ptr(bd, m.src_rank, m.src_buf)) + m.src_off;
      char* dst = static_cast<char*>(const_cast<void*>(buf_ptr(bd, m.dst_rank, m.dst_buf))) + m.dst_off;
      if (!m.bytes || src == dst) continue;  // nothing to move (in-place self block)
      bool placed = false;
      for (size_t q = first; q < jobs->size() && !placed; ++q) {
        if (co(src, (*jobs)[q].dst) == co(src, dst)) {
          (*more)[q].push_back(dst);
          placed = true;
        }
      }
      if (!placed) {
        CopyJob j{};
        j.src = src;
        j.dst = dst;
        j.bytes = m.bytes;
        jobs->push_back(j);
        more->emplace_back();
      }
    }
  }
}

hocResult_t run_tma(hocComm* c, const Step& st, const Bind& bd, cudaStream_t s, int* max_ctas) {
  const uint32_t pb = tma_piece_bytes();
  std::vector<CopyJob> jobs;
  std::vector<std::vector<char*>> more;
  tma_jobs(st, bd, &jobs, &more);
  size_t i = 0;
  while (i < jobs.size()) {
    CopyParams cp;
    memset(&cp, 0, sizeof cp);
    cp.piece_bytes = pb;
    cp.status = c->status;
    cp.tx_pad = c->cfg.fault == kFaultTmaStall ? 16u : 0u;
    cp.wait_ns = c->cfg.fault == kFaultTmaStall ? 100000000ull : 2000000000ull;  // 0.1 s under injection, else 2 s
    int nj = 0, nm = 0;
    for (; i < jobs.size() && nj < kMaxCopyJobs; ++i) {
      // the pool is full: the next launch takes this job (a job has fewer than
      // kMaxRanks extra destinations, so a fresh pool always holds it)
      if (size_t(nm) + more[i].size() > size_t(kMaxMoreDst)) break;
      CopyJob j = jobs[i];
      j.nmore = int32_t(more[i].size());
      j.more_at = nm;
      for (char* d : more[i]) cp.more_dst[nm++] = d;
      cp.job[nj] = j;
      cp.piece_start[nj + 1] = cp.piece_start[nj] + tma_job_pieces(j, pb);
      ++nj;
    }
    cp.njobs = nj;
    if (!nj) continue;
    const uint64_t pieces = cp.piece_start[nj];
    const int cap = c->cfg.copy_max_sms > 0 ? std::min(c->cfg.copy_max_sms, c->sms) : c->sms * tma_ctas_per_sm();
    const int grid = int(std::min<uint64_t>(pieces, uint64_t(cap)));
    *max_ctas = std::max(*max_ctas, grid);
    HOC_TRY(timed_launch(c, HOC_KERNEL_TMA, s, [&] { return launch_tma_copy(cp, grid, s); }));
  }
  return HOC_SUCCESS;
}

// Issue the plan: stream 0 is `s0`; 1..n are the internal copy streams
// (those of `s0`'s set, or `given` when the caller picked them).
hocResult_t issue(hocComm* c, const Plan& p, const Bind& bd, cudaStream_t s0, const std::vector<cudaStream_t>* given,
                  int* max_ctas) {
  std::vector<cudaStream_t> st(p.n_streams);
  st[0] = s0;
  if (p.n_streams > 1) {
    std::vector<cudaStream_t>* copy = nullptr;
    if (given) {
      if (given->size() < size_t(p.n_streams - 1)) return HOC_ERR_INVALID_ARG;
    } else {
      HOC_TRY(copy_streams_for(c, s0, &copy));
    }
    for (int i = 1; i < p.n_streams; ++i) st[i] = given ? (*given)[i - 1] : (*copy)[i - 1];
  }
  const bool prof_streams = c->profiling && p.n_streams > 1;
  // Timeline events of a call the caller is capturing into a graph are
  // recorded as external event nodes, so that they can be read after a replay.
  unsigned tl_flags = cudaEventRecordDefault;
  if (c->profiling) {
    c->prof_streams = 0;
    c->prof_steps.clear();
    if (!c->prof_origin) HOC_CK(cudaEventCreate(&c->prof_origin));
    while (c->prof_step_events.size() < 2 * p.steps.size()) {
      cudaEvent_t e;
      HOC_CK(cudaEventCreate(&e));
      c->prof_step_events.push_back(e);
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    HOC_CK(cudaStreamIsCapturing(s0, &cap));
    if (cap != cudaStreamCaptureStatusNone) tl_flags = cudaEventRecordExternal;
    HOC_CK(cudaEventRecordWithFlags(c->prof_origin, s0, tl_flags));
  }
  if (prof_streams) {
    if (!c->prof_fork) HOC_CK(cudaEventCreate(&c->prof_fork));
    while (c->prof_stream_end.size() < size_t(p.n_streams)) {
      cudaEvent_t e;
      HOC_CK(cudaEventCreate(&e));
      c->prof_stream_end.push_back(e);
    }
    HOC_CK(cudaEventRecord(c->prof_fork, s0));
  }
  if (p.n_streams > 1) {
    HOC_CK(cudaEventRecord(c->fork, s0));
    for (int i = 1; i < p.n_streams; ++i) HOC_CK(cudaStreamWaitEvent(st[i], c->fork, 0));
  }
  HOC_TRY(get_event(c, c->ev, p.steps.size()));
  for (size_t i = 0; i < p.steps.size(); ++i) {
    const Step& step = p.steps[i];
    cudaStream_t s = st[step.stream];
    for (int w : step.waits)
      if (p.steps[w].stream != step.stream) HOC_CK(cudaStreamWaitEvent(s, c->ev[w], 0));
    if (c->profiling) {
      hocComm::StepTiming t{step.kind, step.stream, step.stage, c->prof_step_events[2 * i],
                            c->prof_step_events[2 * i + 1]};
      HOC_CK(cudaEventRecordWithFlags(t.start, s, tl_flags));
      c->prof_steps.push_back(t);
    }
    switch (step.kind) {
      case kStepReduce:
      case kStepFused: HOC_TRY(run_reduce(c, p, step, bd, s, max_ctas)); break;
      case kStepTma: HOC_TRY(run_tma(c, step, bd, s, max_ctas)); break;
      case kStepCopy:
        for (const Move& m : step.moves) {
          const char* src = static_cast<const char*>(buf_ptr(bd, m.src_rank, m.src_buf)) + m.src_off;
          char* dst = static_cast<char*>(const_cast<void*>(buf_ptr(bd, m.dst_rank, m.dst_buf))) + m.dst_off;
          if (!m.bytes || src == dst) continue;  // nothing to move (in-place self block)
          HOC_CK(cudaMemcpyAsync(dst, src, m.bytes, cudaMemcpyDeviceToDevice, s));
        }
        if (c->cfg.debug) {
          HOC_CK(cudaStreamSynchronize(s));
          HOC_CK(cudaGetLastError());
        }
        break;
      default: return HOC_ERR_INVALID_ARG;
    }
    if (c->profiling) HOC_CK(cudaEventRecordWithFlags(c->prof_steps.back().end, s, tl_flags));
    if (step.record) HOC_CK(cudaEventRecord(c->ev[i], s));
  }
  if (prof_streams) {
    for (int i = 1; i < p.n_streams; ++i) HOC_CK(cudaEventRecord(c->prof_stream_end[i - 1], st[i]));
    c->prof_streams = p.n_streams - 1;
  }
  if (p.n_streams > 1) {
    HOC_TRY(get_event(c, c->join, size_t(p.n_streams)));
    for (int i = 1; i < p.n_streams; ++i) {
      HOC_CK(cudaEventRecord(c->join[i], st[i]));
      HOC_CK(cudaStreamWaitEvent(s0, c->join[i], 0));
    }
  }
  return HOC_SUCCESS;
}

}  // namespace

hocResult_t issue_plan(hocComm* c, const Plan& p, const Bind& bd, cudaStream_t s0,
                       const std::vector<cudaStream_t>* copy_streams, int* max_ctas) {
  return issue(c, p, bd, s0, copy_streams, max_ctas);
}

hocResult_t get_plan(hocComm* c, const CallShape& shape, const Plan** plan) {
  const std::string pkey = plan_key(shape);
  auto it = c->plans.find(pkey);
  if (it == c->plans.end()) {
    Plan p;
    HOC_TRY(build_plan(c->cfg, shape, &p));
    if (c->plans.size() > 256) c->plans.clear();
    it = c->plans.emplace(pkey, std::move(p)).first;
  }
  *plan = &it->second;
  return HOC_SUCCESS;
}

void set_error_detail(const char* what) { set_detail(what); }

namespace {

std::string graph_key(const std::string& pkey, const Bind& bd, int k) {
  std::string key = pkey;
  key.append(reinterpret_cast<const char*>(bd.send), sizeof(void*) * k);
  key.append(reinterpret_cast<const char*>(bd.recv), sizeof(void*) * k);
  return key;
}

hocResult_t execute(hocComm* c, const CallShape& shape, const Bind& bd, cudaStream_t stream) {
  const std::string pkey = plan_key(shape);
  const Plan* pp = nullptr;
  HOC_TRY(get_plan(c, shape, &pp));
  const Plan& p = *pp;
  hocOpStats_t stats{};
  stats.path = p.path;
  stats.kernels = p.kernels;
  stats.copies = p.copies;
  stats.bytes_exec = p.bytes_exec;
  stats.bytes_min = p.bytes_min;
  int max_ctas = 0;
  if (p.steps.empty()) {
    c->last = stats;
    return HOC_SUCCESS;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  HOC_CK(cudaStreamIsCapturing(stream, &cs));
  // Graphs pay off when a call issues many operations over several streams;
  // a single copy or kernel is cheaper to issue directly (and a graph per
  // distinct buffer address would only churn the cache).
  const bool worth = p.n_streams > 1 && p.copies + p.kernels >= 8;
  const bool use_graph = c->cfg.use_graphs && !c->profiling && !c->cfg.debug && cs == cudaStreamCaptureStatusNone && worth;
  if (!use_graph) {
    HOC_TRY(issue(c, p, bd, stream, nullptr, &max_ctas));
  } else {
    const std::string gkey = graph_key(pkey, bd, p.k);
    auto g = c->graphs.find(gkey);
    if (g == c->graphs.end()) {
      HOC_CK(cudaStreamBeginCapture(c->capture, cudaStreamCaptureModeThreadLocal));
      hocResult_t r = issue(c, p, bd, c->capture, nullptr, &max_ctas);
      cudaGraph_t graph = nullptr;
      cudaError_t e = cudaStreamEndCapture(c->capture, &graph);
      if (r != HOC_SUCCESS) {
        if (graph) cudaGraphDestroy(graph);
        return r;
      }
      if (e != cudaSuccess) {
        set_detail("cudaStreamEndCapture", e);
        return HOC_ERR_CUDA;
      }
      cudaGraphExec_t exec = nullptr;
      e = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      if (e != cudaSuccess) {
        set_detail("cudaGraphInstantiate", e);
        return HOC_ERR_CUDA;
      }
      if (c->graphs.size() >= kMaxGraphs) {
        const std::string victim = c->lru.back();
        c->lru.pop_back();
        auto v = c->graphs.find(victim);
        if (v != c->graphs.end()) {
          cudaGraphExecDestroy(v->second.exec);
          c->graphs.erase(v);
        }
      }
      c->lru.push_front(gkey);
      g = c->graphs.emplace(gkey, hocComm::GraphEntry{exec, c->lru.begin(), max_ctas}).first;
    } else {
      c->lru.splice(c->lru.begin(), c->lru, g->second.lru);
      stats.graph_replayed = 1;
      max_ctas = g->second.max_ctas;
    }
    HOC_CK(cudaGraphLaunch(g->second.exec, stream));
  }
  stats.max_ctas = max_ctas;
  stats.sms_used = std::min(max_ctas, c->sms);
  c->last = stats;
  return HOC_SUCCESS;
}

}  // namespace
}  // namespace hoc

// ============================================================== C ABI
namespace hoc {
namespace {

hocResult_t read_cfg(const hocConfig_t* in, int k, Cfg* out) {
  Cfg c;
  if (in) {
    c.path = in->path;
    if (in->chunk_bytes) c.chunk_bytes = in->chunk_bytes;
    if (in->n_copy_streams) c.n_copy = in->n_copy_streams;
    else c.n_copy_auto = 1;
    c.depth = in->pipeline_depth;
    c.reduce_max_sms = in->reduce_max_sms;
    c.copy_max_sms = in->copy_max_sms;
    c.use_graphs = in->use_graphs;
    c.a2a_interleave = in->a2a_interleave;
    c.a2a_stage_sync = in->a2a_stage_sync;
    if (in->ring_order) c.order.assign(in->ring_order, in->ring_order + k);
    c.reduce_engine = in->reduce_engine;
  }
  if (const char* v = getenv("HOC_PATH")) {
    if (!strcmp(v, "ce")) c.path = HOC_PATH_CE;
    else if (!strcmp(v, "tma")) c.path = HOC_PATH_TMA;
    else if (!strcmp(v, "fused")) c.path = HOC_PATH_FUSED;
    else if (!strcmp(v, "auto")) c.path = HOC_PATH_AUTO;
  }
  if (const char* v = getenv("HOC_CHUNK_BYTES")) c.chunk_bytes = size_t(strtoull(v, nullptr, 10));
  if (!in) c.n_copy_auto = 1;
  if (getenv("HOC_COPY_STREAMS")) {
    c.n_copy = env_int("HOC_COPY_STREAMS", c.n_copy);
    c.n_copy_auto = 0;
  }
  if (c.n_copy_auto) c.n_copy = std::max(kAutoQueuesSmall, kAutoQueuesLarge);  // streams for either choice
  c.use_graphs = env_int("HOC_USE_GRAPHS", c.use_graphs);
  c.reduce_max_sms = env_int("HOC_REDUCE_MAX_SMS", c.reduce_max_sms);
  c.copy_max_sms = env_int("HOC_COPY_MAX_SMS", c.copy_max_sms);
  c.depth = env_int("HOC_PIPELINE_DEPTH", c.depth);
  if (const char* v = getenv("HOC_REDUCE_ENGINE")) {
    if (!strcmp(v, "lsu")) c.reduce_engine = HOC_REDUCE_LSU;
    else if (!strcmp(v, "tma")) c.reduce_engine = HOC_REDUCE_TMA;
    else if (!strcmp(v, "auto")) c.reduce_engine = HOC_REDUCE_AUTO;
  }
  c.debug = env_int("HOC_DEBUG", 0);
  if (const char* v = getenv("HOC_FAULT")) {
    if (!strcmp(v, "drop_chunk")) c.fault = kFaultDropChunk;
    else if (!strcmp(v, "dup_chunk")) c.fault = kFaultDupChunk;
    else if (!strcmp(v, "wrong_order")) c.fault = kFaultWrongOrder;
    else if (!strcmp(v, "proxy_stall")) c.fault = kFaultProxyStall;
    else if (!strcmp(v, "tma_stall")) c.fault = kFaultTmaStall;
    else if (!strcmp(v, "proxy_block")) c.fault = kFaultProxyBlock;
    else if (!strcmp(v, "proxy_memop")) c.fault = kFaultProxyMemop;
    else if (!strcmp(v, "proxy_memop_reset")) c.fault = kFaultProxyMemopReset;
  }
  if (c.order.empty())
    for (int i = 0; i < k; ++i) c.order.push_back(i);
  std::vector<int> seen(k, 0);
  for (int v : c.order) {
    if (v < 0 || v >= k || seen[v]) {
      set_detail("ring_order is not a permutation of 0..k-1");
      return HOC_ERR_INVALID_ARG;
    }
    seen[v] = 1;
  }
  if (c.path < HOC_PATH_AUTO || c.path > HOC_PATH_FUSED || c.n_copy < 1 || c.n_copy > 16 || (c.chunk_bytes != 0 && c.chunk_bytes < 256) ||
      c.depth < 0 || c.reduce_max_sms < 0 || c.copy_max_sms < 0 || c.reduce_engine < HOC_REDUCE_AUTO ||
      c.reduce_engine > HOC_REDUCE_TMA) {
    set_detail("configuration value out of range");
    return HOC_ERR_INVALID_ARG;
  }
  c.use_graphs = c.use_graphs ? 1 : 0;
  *out = c;
  return HOC_SUCCESS;
}

void free_comm(hocComm* c) {
  if (!c) return;
  host_ar_free(c);
  for (auto& g : c->graphs) cudaGraphExecDestroy(g.second.exec);
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  for (cudaEvent_t e : c->join) cudaEventDestroy(e);
  for (cudaEvent_t e : c->prof_free) cudaEventDestroy(e);
  for (auto& pp : c->prof_pending) {
    cudaEventDestroy(pp.start);
    cudaEventDestroy(pp.stop);
  }
  if (c->fork) cudaEventDestroy(c->fork);
  if (c->prof_fork) cudaEventDestroy(c->prof_fork);
  for (cudaEvent_t e : c->prof_stream_end) cudaEventDestroy(e);
  for (auto& set : c->sets)
    for (cudaStream_t s : set.copy) cudaStreamDestroy(s);
  if (c->capture) cudaStreamDestroy(c->capture);
  if (c->status) cudaFree(c->status);
  delete c;
}

bool dtype_ok(int dtype, bool reduction) {
  if (reduction) return dtype == HOC_INT32 || dtype == HOC_FLOAT32 || dtype == HOC_BFLOAT16;
  return dtype_bytes(dtype) != 0;
}

bool elem_aligned(const void* p, size_t b) { return (reinterpret_cast<uintptr_t>(p) % b) == 0; }

struct Range {
  uintptr_t lo, hi;
  bool writable;
  int rank;
};

// Writable ranges may not overlap any other range; read-only ranges may
// overlap each other.  `same_ok(a, b)` names the allowed in-place pairs.
template <class F>
hocResult_t check_overlaps(const std::vector<Range>& rs, F&& same_ok) {
  for (size_t i = 0; i < rs.size(); ++i)
    for (size_t j = i + 1; j < rs.size(); ++j) {
      const Range &a = rs[i], &b = rs[j];
      if (!(a.writable || b.writable)) continue;
      if (a.lo >= b.hi || b.lo >= a.hi) continue;
      if (same_ok(a, b)) continue;
      set_detail("rank buffers overlap");
      return HOC_ERR_INVALID_ARG;
    }
  return HOC_SUCCESS;
}

hocResult_t check_array(const void* const* a, int k, size_t b) {
  if (!a) {
    set_detail("NULL buffer array");
    return HOC_ERR_INVALID_ARG;
  }
  for (int r = 0; r < k; ++r) {
    if (!a[r]) {
      set_detail("NULL rank buffer");
      return HOC_ERR_INVALID_ARG;
    }
    if (!elem_aligned(a[r], b)) {
      set_detail("rank buffer not aligned to its element size");
      return HOC_ERR_INVALID_ARG;
    }
  }
  return HOC_SUCCESS;
}

hocResult_t check_reduce_args(hocComm* c, int dtype, int op) {
  if (!c) return HOC_ERR_NOT_INITIALIZED;
  if (!dtype_ok(dtype, true)) {
    set_detail(dtype == HOC_UINT8 ? "reductions take int32, float32 or bfloat16" : "unknown dtype");
    return dtype == HOC_UINT8 ? HOC_ERR_UNSUPPORTED : HOC_ERR_INVALID_ARG;
  }
  if (op != HOC_SUM) {
    set_detail("only HOC_SUM is implemented");
    return HOC_ERR_UNSUPPORTED;
  }
  return HOC_SUCCESS;
}

uintptr_t U(const void* p) { return reinterpret_cast<uintptr_t>(p); }

const char* op_name(int op) {
  switch (op) {
    case HOC_OP_ALLREDUCE: return "hoc_allreduce";
    case HOC_OP_REDUCE_SCATTER: return "hoc_reduce_scatter";
    case HOC_OP_ALLGATHER: return "hoc_allgather";
    case HOC_OP_ALLTOALL: return "hoc_alltoall";
    default: return "hoc_sendrecv";
  }
}

// NVTX range around the host side of every call (visible in any profiler that
// records NVTX; a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

hocResult_t run(hocComm* c, const CallShape& shape, const Bind& bd, void* stream) {
  NvtxRange range(op_name(shape.op));
  std::lock_guard<std::mutex> lock(c->mu);
  DeviceGuard g(c->device);
  if (!g.ok) {
    set_detail("cudaSetDevice failed");
    return HOC_ERR_CUDA;
  }
  return execute(c, shape, bd, static_cast<cudaStream_t>(stream));
}

// The plan on one of the caller stream's copy streams: it waits for the work
// before the call on `stream`, and `done` is recorded when it completes;
// `stream` itself is not joined.
hocResult_t run_detached(hocComm* c, const CallShape& shape, const Bind& bd, void* stream, void* done) {
  NvtxRange range("hoc_sendrecv_async");
  std::lock_guard<std::mutex> lock(c->mu);
  DeviceGuard g(c->device);
  if (!g.ok) {
    set_detail("cudaSetDevice failed");
    return HOC_ERR_CUDA;
  }
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  HOC_CK(cudaStreamIsCapturing(s0, &cs));
  if (cs != cudaStreamCaptureStatusNone) {
    set_detail("hoc_sendrecv_async cannot be captured into a graph (its copy is not joined to the stream)");
    return HOC_ERR_UNSUPPORTED;
  }
  const Plan* pp = nullptr;
  HOC_TRY(get_plan(c, shape, &pp));
  std::vector<cudaStream_t>* copy = nullptr;
  HOC_TRY(copy_streams_for(c, s0, &copy));
  cudaStream_t cs0 = (*copy)[c->detached_next++ % copy->size()];  // spread consecutive sends over the queues
  HOC_CK(cudaEventRecord(c->fork, s0));
  HOC_CK(cudaStreamWaitEvent(cs0, c->fork, 0));
  int max_ctas = 0;
  HOC_TRY(issue(c, *pp, bd, cs0, copy, &max_ctas));
  HOC_CK(cudaEventRecord(static_cast<cudaEvent_t>(done), cs0));
  hocOpStats_t stats{};
  stats.path = pp->path;
  stats.kernels = pp->kernels;
  stats.copies = pp->copies;
  stats.bytes_exec = pp->bytes_exec;
  stats.bytes_min = pp->bytes_min;
  stats.max_ctas = max_ctas;
  stats.sms_used = std::min(max_ctas, c->sms);
  c->last = stats;
  return HOC_SUCCESS;
}

// hoc_allreduce with the plan's path set by `path` (-1: the communicator's).
hocResult_t allreduce_on(hocComm_t comm, const void* const* send, void* const* recv, size_t count,
                         hocDataType_t dtype, hocRedOp_t op, void* stream, int path) {
  HOC_TRY(check_reduce_args(comm, dtype, op));
  if (count == 0) return HOC_SUCCESS;
  const int k = comm->k;
  const size_t b = dtype_bytes(dtype);
  HOC_TRY(check_array(send, k, b));
  HOC_TRY(check_array(const_cast<const void* const*>(reinterpret_cast<void* const*>(recv)), k, b));
  std::vector<Range> rs;
  for (int r = 0; r < k; ++r) {
    rs.push_back(Range{U(send[r]), U(send[r]) + count * b, false, r});
    rs.push_back(Range{U(recv[r]), U(recv[r]) + count * b, true, r});
  }
  HOC_TRY(check_overlaps(rs, [](const Range& a, const Range& b2) {
    return a.rank == b2.rank && a.writable != b2.writable && a.lo == b2.lo;  // in place: send[r] == recv[r]
  }));
  CallShape s;
  s.op = HOC_OP_ALLREDUCE;
  s.k = k;
  s.dtype = dtype;
  s.count = count;
  s.path = path;
  Bind bd;
  for (int r = 0; r < k; ++r) {
    bd.send[r] = send[r];
    bd.recv[r] = recv[r];
  }
  return run(comm, s, bd, stream);
}
hocResult_t sendrecv_shape(hocComm_t comm, int src_rank, const void* send, int dst_rank, void* recv, size_t count,
                           hocDataType_t dtype, CallShape* out, Bind* bind, bool* nothing) {
  *nothing = false;
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!dtype_ok(dtype, false)) {
    set_detail("unknown dtype");
    return HOC_ERR_INVALID_ARG;
  }
  if (src_rank < 0 || src_rank >= comm->k || dst_rank < 0 || dst_rank >= comm->k) {
    set_detail("rank out of range");
    return HOC_ERR_INVALID_ARG;
  }
  if (count == 0) {
    *nothing = true;
    return HOC_SUCCESS;
  }
  const size_t b = dtype_bytes(dtype);
  if (!send || !recv || !elem_aligned(send, b) || !elem_aligned(recv, b)) {
    set_detail("NULL or misaligned buffer");
    return HOC_ERR_INVALID_ARG;
  }
  if (send == recv) {
    *nothing = true;
    return HOC_SUCCESS;
  }
  const uintptr_t a = U(send), d = U(recv);
  if (a < d + count * b && d < a + count * b) {
    set_detail("send and recv overlap");
    return HOC_ERR_INVALID_ARG;
  }
  out->op = HOC_OP_SENDRECV;
  out->k = comm->k;
  out->dtype = dtype;
  out->count = count;
  out->src_rank = src_rank;
  out->dst_rank = dst_rank;
  bind->send[src_rank] = send;
  bind->recv[dst_rank] = recv;
  return HOC_SUCCESS;
}
}  // namespace

hocResult_t allreduce_fused(hocComm* comm, const void* const* send, void* const* recv, size_t count, int dtype,
                            cudaStream_t stream) {
  return allreduce_on(comm, send, recv, count, hocDataType_t(dtype), HOC_SUM, stream, HOC_PATH_FUSED);
}

}  // namespace hoc

using namespace hoc;

extern "C" {

hocResult_t hoc_config_default(hocConfig_t* cfg) {
  if (!cfg) return HOC_ERR_INVALID_ARG;
  memset(cfg, 0, sizeof *cfg);
  cfg->path = HOC_PATH_AUTO;
  cfg->chunk_bytes = 0;  // by move path
  cfg->n_copy_streams = 0;  // the scheduler picks per call (copy_queues)
  cfg->pipeline_depth = 0;
  cfg->reduce_max_sms = 0;
  cfg->copy_max_sms = 0;
  cfg->use_graphs = 1;
  cfg->a2a_interleave = 1;
  cfg->a2a_stage_sync = 0;
  cfg->ring_order = nullptr;
  cfg->reduce_engine = HOC_REDUCE_AUTO;
  return HOC_SUCCESS;
}

hocResult_t hoc_init(hocComm_t* comm, int nranks, int device, const hocConfig_t* cfg) {
  if (!comm) return HOC_ERR_INVALID_ARG;
  *comm = nullptr;
  if (nranks < 1 || nranks > kMaxRanks) {
    set_detail("nranks must be 1..HOC_MAX_RANKS");
    return HOC_ERR_INVALID_ARG;
  }
  Cfg c;
  HOC_TRY(read_cfg(cfg, nranks, &c));
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    set_detail("no CUDA device");
    return HOC_ERR_NO_DEVICE;
  }
  if (device < 0 || device >= ndev) {
    set_detail("device index out of range");
    return HOC_ERR_INVALID_ARG;
  }
  DeviceGuard g(device);
  if (!g.ok) {
    set_detail("cudaSetDevice failed");
    return HOC_ERR_CUDA;
  }
  hocComm* h = new (std::nothrow) hocComm();
  if (!h) return HOC_ERR_OOM;
  h->k = nranks;
  h->device = device;
  h->cfg = c;
  auto fail = [&](const char* what, cudaError_t e) {
    set_detail(what, e);
    free_comm(h);
    return e == cudaErrorMemoryAllocation ? HOC_ERR_OOM : HOC_ERR_CUDA;
  };
  cudaError_t e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return fail("cudaDeviceGetAttribute", e);
  e = cudaStreamCreateWithFlags(&h->capture, cudaStreamNonBlocking);
  if (e != cudaSuccess) return fail("cudaStreamCreateWithFlags", e);
  {
    std::vector<cudaStream_t>* unused = nullptr;  // the set graph captures fork into
    if (copy_streams_for(h, h->capture, &unused) != HOC_SUCCESS) {
      free_comm(h);
      return HOC_ERR_CUDA;
    }
  }
  e = cudaEventCreateWithFlags(&h->fork, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail("cudaEventCreateWithFlags", e);
  e = cudaMalloc(&h->status, 256);
  if (e != cudaSuccess) return fail("cudaMalloc(status)", e);
  e = cudaMemset(h->status, 0, 256);
  if (e != cudaSuccess) return fail("cudaMemset(status)", e);
  e = tma_prepare();
  if (e != cudaSuccess) return fail("tma_prepare", e);
  e = reduce_tma_prepare();
  if (e != cudaSuccess) return fail("reduce_tma_prepare", e);
  // occupancy of every reduce kernel this communicator can launch, queried
  // now so that nothing but stream work happens while a graph is captured
  for (int dt : {int(HOC_INT32), int(HOC_FLOAT32), int(HOC_BFLOAT16)})
    for (int bc = 0; bc < 2; ++bc) ctas_per_sm(h, dt, nranks, bc);
  *comm = h;
  return HOC_SUCCESS;
}

hocResult_t hoc_destroy(hocComm_t comm) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  proxy_shutdown(comm);
  {
    DeviceGuard g(comm->device);
    for (auto& set : comm->sets)
      for (cudaStream_t s : set.copy) cudaStreamSynchronize(s);
    free_comm(comm);
  }
  return HOC_SUCCESS;
}

hocResult_t hoc_allreduce(hocComm_t comm, const void* const* send, void* const* recv, size_t count,
                          hocDataType_t dtype, hocRedOp_t op, void* stream) {
  return allreduce_on(comm, send, recv, count, dtype, op, stream, -1);
}

hocResult_t hoc_reduce_scatter(hocComm_t comm, const void* const* send, void* const* recv, size_t recvcount,
                               hocDataType_t dtype, hocRedOp_t op, void* stream) {
  HOC_TRY(check_reduce_args(comm, dtype, op));
  if (recvcount == 0) return HOC_SUCCESS;
  const int k = comm->k;
  const size_t b = dtype_bytes(dtype);
  HOC_TRY(check_array(send, k, b));
  HOC_TRY(check_array(const_cast<const void* const*>(reinterpret_cast<void* const*>(recv)), k, b));
  std::vector<Range> rs;
  for (int r = 0; r < k; ++r) {
    rs.push_back(Range{U(send[r]), U(send[r]) + size_t(k) * recvcount * b, false, r});
    rs.push_back(Range{U(recv[r]), U(recv[r]) + recvcount * b, true, r});
  }
  HOC_TRY(check_overlaps(rs, [&](const Range& a, const Range& b2) {
    if (a.rank != b2.rank || a.writable == b2.writable) return false;
    const Range& w = a.writable ? a : b2;
    const Range& ro = a.writable ? b2 : a;
    return w.lo == ro.lo + size_t(a.rank) * recvcount * b;  // in place: recv[r] = send[r] + r*recvcount
  }));
  CallShape s;
  s.op = HOC_OP_REDUCE_SCATTER;
  s.k = k;
  s.dtype = dtype;
  s.count = recvcount;
  Bind bd;
  for (int r = 0; r < k; ++r) {
    bd.send[r] = send[r];
    bd.recv[r] = recv[r];
  }
  return run(comm, s, bd, stream);
}

hocResult_t hoc_allgather(hocComm_t comm, const void* const* send, void* const* recv, size_t sendcount,
                          hocDataType_t dtype, void* stream) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!dtype_ok(dtype, false)) {
    set_detail("unknown dtype");
    return HOC_ERR_INVALID_ARG;
  }
  if (sendcount == 0) return HOC_SUCCESS;
  const int k = comm->k;
  const size_t b = dtype_bytes(dtype);
  HOC_TRY(check_array(send, k, b));
  HOC_TRY(check_array(const_cast<const void* const*>(reinterpret_cast<void* const*>(recv)), k, b));
  std::vector<Range> rs;
  for (int r = 0; r < k; ++r) {
    rs.push_back(Range{U(send[r]), U(send[r]) + sendcount * b, false, r});
    rs.push_back(Range{U(recv[r]), U(recv[r]) + size_t(k) * sendcount * b, true, r});
  }
  HOC_TRY(check_overlaps(rs, [&](const Range& a, const Range& b2) {
    if (a.rank != b2.rank || a.writable == b2.writable) return false;
    const Range& w = a.writable ? a : b2;
    const Range& ro = a.writable ? b2 : a;
    return ro.lo == w.lo + size_t(a.rank) * sendcount * b;  // in place: send[r] = recv[r] + r*sendcount
  }));
  CallShape s;
  s.op = HOC_OP_ALLGATHER;
  s.k = k;
  s.dtype = dtype;
  s.count = sendcount;
  Bind bd;
  for (int r = 0; r < k; ++r) {
    bd.send[r] = send[r];
    bd.recv[r] = recv[r];
  }
  return run(comm, s, bd, stream);
}

hocResult_t hoc_alltoall(hocComm_t comm, const void* const* send, const size_t* sendcounts, const size_t* sdispls,
                         void* const* recv, const size_t* rdispls, size_t count_if_uniform, hocDataType_t dtype,
                         void* stream) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!dtype_ok(dtype, false)) {
    set_detail("unknown dtype");
    return HOC_ERR_INVALID_ARG;
  }
  const int k = comm->k;
  const size_t b = dtype_bytes(dtype);
  const size_t kk = size_t(k) * k;
  std::vector<size_t> cnt(kk), sd(kk), rd(kk);
  size_t total = 0;
  for (size_t i = 0; i < kk; ++i) {
    cnt[i] = sendcounts ? sendcounts[i] : count_if_uniform;
    total += cnt[i];
  }
  if (total == 0) return HOC_SUCCESS;
  for (int a = 0; a < k; ++a)
    for (int d = 0; d < k; ++d)
      sd[size_t(a) * k + d] = sdispls ? sdispls[size_t(a) * k + d] : (d ? sd[size_t(a) * k + d - 1] + cnt[size_t(a) * k + d - 1] : 0);
  for (int d = 0; d < k; ++d)
    for (int a = 0; a < k; ++a)
      rd[size_t(d) * k + a] = rdispls ? rdispls[size_t(d) * k + a] : (a ? rd[size_t(d) * k + a - 1] + cnt[size_t(a - 1) * k + d] : 0);
  HOC_TRY(check_array(send, k, b));
  HOC_TRY(check_array(const_cast<const void* const*>(reinterpret_cast<void* const*>(recv)), k, b));
  std::vector<Range> rs;
  for (int a = 0; a < k; ++a)
    for (int d = 0; d < k; ++d) {
      const size_t n = cnt[size_t(a) * k + d] * b;
      if (!n) continue;
      rs.push_back(Range{U(send[a]) + sd[size_t(a) * k + d] * b, U(send[a]) + sd[size_t(a) * k + d] * b + n, false, a});
      rs.push_back(Range{U(recv[d]) + rd[size_t(d) * k + a] * b, U(recv[d]) + rd[size_t(d) * k + a] * b + n, true, d});
    }
  HOC_TRY(check_overlaps(rs, [](const Range&, const Range&) { return false; }));
  CallShape s;
  s.op = HOC_OP_ALLTOALL;
  s.k = k;
  s.dtype = dtype;
  if (sendcounts) s.counts = cnt;
  else s.count = count_if_uniform;
  if (sdispls) s.sdispls = sd;
  if (rdispls) s.rdispls = rd;
  Bind bd;
  for (int r = 0; r < k; ++r) {
    bd.send[r] = send[r];
    bd.recv[r] = recv[r];
  }
  return run(comm, s, bd, stream);
}

hocResult_t hoc_sendrecv(hocComm_t comm, int src_rank, const void* send, int dst_rank, void* recv, size_t count,
                         hocDataType_t dtype, void* stream) {
  CallShape s;
  Bind bd;
  bool nothing = false;
  HOC_TRY(sendrecv_shape(comm, src_rank, send, dst_rank, recv, count, dtype, &s, &bd, &nothing));
  if (nothing) return HOC_SUCCESS;
  return run(comm, s, bd, stream);
}

hocResult_t hoc_sendrecv_async(hocComm_t comm, int src_rank, const void* send, int dst_rank, void* recv, size_t count,
                               hocDataType_t dtype, void* stream, void* done_event) {
  if (comm && !done_event) {
    set_detail("hoc_sendrecv_async: NULL done_event");
    return HOC_ERR_INVALID_ARG;
  }
  CallShape s;
  Bind bd;
  bool nothing = false;
  HOC_TRY(sendrecv_shape(comm, src_rank, send, dst_rank, recv, count, dtype, &s, &bd, &nothing));
  if (nothing) {  // nothing to move: the event completes with the work before the call
    DeviceGuard g(comm->device);
    HOC_CK(cudaEventRecord(static_cast<cudaEvent_t>(done_event), static_cast<cudaStream_t>(stream)));
    return HOC_SUCCESS;
  }
  return run_detached(comm, s, bd, stream, done_event);
}


hocResult_t hoc_wait(hocComm_t comm, void* stream, int timeout_ms) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  DeviceGuard g(comm->device);
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms < 0 ? 0 : timeout_ms);
  std::vector<cudaStream_t> all;
  {
    std::lock_guard<std::mutex> lock(comm->mu);  // another thread's call may add a stream set
    for (auto& set : comm->sets) all.insert(all.end(), set.copy.begin(), set.copy.end());
  }
  all.push_back(static_cast<cudaStream_t>(stream));
  for (cudaStream_t s : all) {
    for (;;) {
      cudaError_t e = cudaStreamQuery(s);
      if (e == cudaSuccess) break;
      if (e != cudaErrorNotReady) {
        set_detail("cudaStreamQuery", e);
        return HOC_ERR_CUDA;
      }
      if (std::chrono::steady_clock::now() >= deadline) {
        set_detail("hoc_wait: work still running at the deadline");
        return HOC_ERR_TIMEOUT;
      }
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  std::string why;
  if (const int perr = proxy_take_error(comm, &why)) {
    set_detail(("a device-count all-to-all was released by the proxy: " + why).c_str());
    return hocResult_t(perr);
  }
  if (comm->cfg.fault == kFaultProxyStall && !comm->proxy) {
    // Injected on the host: a completion that never arrives.
    std::this_thread::sleep_until(deadline);
    set_detail("hoc_wait: injected proxy stall");
    return HOC_ERR_TIMEOUT;
  }
  int st = 0;
  HOC_CK(cudaMemcpy(&st, comm->status, sizeof st, cudaMemcpyDeviceToHost));
  if (st != 0) {
    HOC_CK(cudaMemset(comm->status, 0, sizeof st));
    char buf[96];
    snprintf(buf, sizeof buf, "TMA copy kernel gave up on a bounded wait (status 0x%x)", st);
    set_detail(buf);
    return HOC_ERR_TIMEOUT;
  }
  return HOC_SUCCESS;
}

hocResult_t hoc_last_stats(hocComm_t comm, hocOpStats_t* stats) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!stats) return HOC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(comm->mu);
  *stats = comm->last;
  return HOC_SUCCESS;
}

hocResult_t hoc_profile_enable(hocComm_t comm, int enable) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  std::lock_guard<std::mutex> lock(comm->mu);
  comm->profiling = enable != 0;
  return HOC_SUCCESS;
}

hocResult_t hoc_profile_read(hocComm_t comm, hocKernel_t kernel, int* launches, double* total_ms) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (kernel < HOC_KERNEL_REDUCE || kernel > HOC_KERNEL_TMA || !launches || !total_ms) return HOC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(comm->mu);
  DeviceGuard g(comm->device);
  for (const ProfPair& pp : comm->prof_pending) {
    HOC_CK(cudaEventSynchronize(pp.stop));
    float ms = 0.f;
    HOC_CK(cudaEventElapsedTime(&ms, pp.start, pp.stop));
    comm->prof_launches[pp.kind] += 1;
    comm->prof_ms[pp.kind] += ms;
    comm->prof_free.push_back(pp.start);
    comm->prof_free.push_back(pp.stop);
  }
  comm->prof_pending.clear();
  *launches = comm->prof_launches[kernel];
  *total_ms = comm->prof_ms[kernel];
  comm->prof_launches[kernel] = 0;
  comm->prof_ms[kernel] = 0;
  return HOC_SUCCESS;
}

hocResult_t hoc_profile_stream_finish(hocComm_t comm, float* finish_ms, int max_streams, int* n_streams) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!n_streams || (max_streams > 0 && !finish_ms)) return HOC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(comm->mu);
  DeviceGuard g(comm->device);
  *n_streams = comm->prof_streams;
  for (int i = 0; i < comm->prof_streams && i < max_streams; ++i) {
    HOC_CK(cudaEventSynchronize(comm->prof_stream_end[i]));
    HOC_CK(cudaEventElapsedTime(&finish_ms[i], comm->prof_fork, comm->prof_stream_end[i]));
  }
  return HOC_SUCCESS;
}

hocResult_t hoc_profile_timeline(hocComm_t comm, hocStepTime_t* items, size_t cap, size_t* n_items) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!n_items || (cap > 0 && !items)) return HOC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(comm->mu);
  DeviceGuard g(comm->device);
  *n_items = comm->prof_steps.size();
  for (size_t i = 0; i < comm->prof_steps.size() && i < cap; ++i) {
    const hocComm::StepTiming& t = comm->prof_steps[i];
    hocStepTime_t& o = items[i];
    o.kind = t.kind == kStepReduce ? HOC_ITEM_REDUCE : t.kind == kStepFused ? HOC_ITEM_FUSED
           : t.kind == kStepTma ? HOC_ITEM_TMA : HOC_ITEM_COPY;
    o.stream = t.stream;
    o.stage = t.stage;
    HOC_CK(cudaEventSynchronize(t.end));
    HOC_CK(cudaEventElapsedTime(&o.start_ms, comm->prof_origin, t.start));
    HOC_CK(cudaEventElapsedTime(&o.end_ms, comm->prof_origin, t.end));
  }
  return HOC_SUCCESS;
}

const char* hoc_error_string(hocResult_t r) {
  switch (r) {
    case HOC_SUCCESS: return "success";
    case HOC_ERR_INVALID_ARG: return "invalid argument";
    case HOC_ERR_CUDA: return "CUDA error";
    case HOC_ERR_OOM: return "out of memory";
    case HOC_ERR_NOT_INITIALIZED: return "communicator not initialized";
    case HOC_ERR_UNSUPPORTED: return "unsupported";
    case HOC_ERR_TIMEOUT: return "timeout";
    case HOC_ERR_NO_DEVICE: return "no CUDA device";
    default: return "unknown result code";
  }
}

const char* hoc_last_error_detail(void) { return g_detail.c_str(); }

hocResult_t hoc_plan_query(int nranks, const hocConfig_t* cfg, int op, size_t count, hocDataType_t dtype,
                           const size_t* counts, hocPlanItem_t* items, size_t cap, size_t* n_items) {
  if (!n_items) return HOC_ERR_INVALID_ARG;
  *n_items = 0;
  if (nranks < 1 || nranks > kMaxRanks) return HOC_ERR_INVALID_ARG;
  Cfg c;
  HOC_TRY(read_cfg(cfg, nranks, &c));
  CallShape s;
  s.op = op;
  s.k = nranks;
  s.dtype = dtype;
  s.count = count;
  if (op == HOC_OP_ALLTOALL && counts) s.counts.assign(counts, counts + size_t(nranks) * nranks);
  if (op == HOC_OP_SENDRECV) {
    s.src_rank = 0;
    s.dst_rank = 1 % nranks;
  }
  Plan p;
  HOC_TRY(build_plan(c, s, &p));
  const size_t b = dtype_bytes(dtype);
  size_t n = 0;
  auto put = [&](const hocPlanItem_t& it) {
    if (items && n < cap) items[n] = it;
    ++n;
  };
  for (size_t i = 0; i < p.steps.size(); ++i) {
    const Step& st = p.steps[i];
    hocPlanItem_t base{};
    base.step = int(i);
    base.stream = st.stream;
    base.stage = st.stage;
    base.n_waits = int(st.waits.size());
    base.wait0 = st.waits.empty() ? -1 : st.waits[0];
    if (st.kind == kStepReduce || st.kind == kStepFused) {
      for (const ReduceSeg& g : st.segs) {
        hocPlanItem_t it = base;
        it.kind = st.kind == kStepFused ? HOC_ITEM_FUSED : HOC_ITEM_REDUCE;
        it.src_rank = -1;
        it.dst_rank = int(g.owner);
        it.src_buf = HOC_BUF_SEND;
        it.dst_buf = HOC_BUF_RECV;
        it.src_off = g.elem_off * b;
        it.dst_off = g.out_off * b;
        it.bytes = g.elems * b;
        put(it);
      }
    } else {
      for (const Move& m : st.moves) {
        hocPlanItem_t it = base;
        it.kind = st.kind == kStepTma ? HOC_ITEM_TMA : HOC_ITEM_COPY;
        it.src_rank = m.src_rank;
        it.dst_rank = m.dst_rank;
        it.src_buf = m.src_buf;
        it.dst_buf = m.dst_buf;
        it.src_off = m.src_off;
        it.dst_off = m.dst_off;
        it.bytes = m.bytes;
        put(it);
      }
    }
  }
  *n_items = n;
  return HOC_SUCCESS;
}

}  // extern "C"
