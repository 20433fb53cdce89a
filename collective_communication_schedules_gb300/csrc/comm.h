// The communicator object, shared by the C ABI (hoc.cpp) and the host proxy
// (proxy.cpp).  Internal: not part of the C ABI.
#pragma once

#include <list>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "hoc.h"
#include "hoc_internal.h"
#include "plan.h"

namespace hoc {

struct ProfPair {
  cudaEvent_t start, stop;
  int kind;
};

struct Bind {
  const void* send[kMaxRanks] = {};
  void* recv[kMaxRanks] = {};
};

struct Proxy;  // host proxy of the flag handshake (proxy.cpp)

}  // namespace hoc

struct hocComm {
  int k = 0;
  int device = 0;
  int sms = 0;
  hoc::Cfg cfg;
  std::mutex mu;
  // Internal copy streams, one set per caller stream (the paper's stream
  // manager keeps its handshake state per GPU stream): calls issued on
  // different caller streams never queue behind each other.
  struct StreamSet {
    cudaStream_t owner;
    std::vector<cudaStream_t> copy;
  };
  std::vector<StreamSet> sets;
  cudaStream_t capture = nullptr;  // origin stream for graph capture
  std::vector<cudaEvent_t> ev;     // plan edges (timing disabled)
  std::vector<cudaEvent_t> join;   // one per internal stream
  cudaEvent_t fork = nullptr;
  int* status = nullptr;           // device status word(s) of the TMA kernel
  std::unordered_map<std::string, hoc::Plan> plans;
  struct GraphEntry {
    cudaGraphExec_t exec;
    std::list<std::string>::iterator lru;
    int max_ctas;
  };
  std::unordered_map<std::string, GraphEntry> graphs;
  std::list<std::string> lru;
  hocOpStats_t last{};
  bool profiling = false;
  std::vector<hoc::ProfPair> prof_pending;
  std::vector<cudaEvent_t> prof_free;
  int prof_launches[3] = {0, 0, 0};
  double prof_ms[3] = {0, 0, 0};
  // While profiling: timing events at the fork of the last multi-stream call
  // and after the last operation of each of its copy streams.
  cudaEvent_t prof_fork = nullptr;
  std::vector<cudaEvent_t> prof_stream_end;
  int prof_streams = 0;  // copy streams the last profiled call used (0: none)
  // While profiling: the fork of the last profiled call (recorded on the
  // caller's stream before anything else) and an event pair around each of its
  // steps, recorded on the step's stream after its waits.
  cudaEvent_t prof_origin = nullptr;
  struct StepTiming {
    int kind, stream, stage;
    cudaEvent_t start, end;
  };
  std::vector<StepTiming> prof_steps;
  std::vector<cudaEvent_t> prof_step_events;  // pool, reused call after call
  int reduce_ctas_per_sm[3][hoc::kMaxRanks + 1][2] = {};
  hoc::Proxy* proxy = nullptr;  // created by the first device-count all-to-all
  unsigned detached_next = 0;   // copy stream of the next hoc_sendrecv_async
  void* host_ar = nullptr;      // staging and streams of hoc_allreduce_host (host_ar.cpp)
};

namespace hoc {

// Build (or fetch from the cache) the plan of a call shape.
hocResult_t get_plan(hocComm* c, const CallShape& shape, const Plan** plan);
// Issue a plan with stream 0 = s0, forking to and joining from the copy
// streams `copy_streams` (at least n_streams - 1 of them), or s0's own set
// when that is null.
hocResult_t issue_plan(hocComm* c, const Plan& p, const Bind& bd, cudaStream_t s0,
                       const std::vector<cudaStream_t>* copy_streams, int* max_ctas);
// One fused allreduce launch on the given rank buffers, whatever the
// communicator's path (the buffers may be any memory the device can address).
hocResult_t allreduce_fused(hocComm* c, const void* const* send, void* const* recv, size_t count, int dtype,
                            cudaStream_t stream);
// Release the proxy (waits, bounded, for its tasks; see proxy.cpp).
void proxy_shutdown(hocComm* c);
// Free what hoc_allreduce_host set up (staging slots, streams, graphs).
void host_ar_free(hocComm* c);
// First error of a proxy task since the last call (0 if none) and, in `why`
// when non-null, what it was; both are then cleared.
int proxy_take_error(hocComm* c, std::string* why);
void set_error_detail(const char* what);

}  // namespace hoc
