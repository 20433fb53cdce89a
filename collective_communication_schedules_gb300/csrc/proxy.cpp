// Host proxy of the stream-memory-operation handshake (HOCCL section 3.2,
// Fig. 4, Listing 1), serving all-to-all(v) exchanges whose counts are
// computed on the device.  See include/hoc_proxy.h for the contract.
//
// Per task the caller's stream runs, in order:
//   copy counts device -> pinned host slot;
//   write start_flag = START; wait start_flag == 0      (the proxy's ack)
//   wait end_flag == FINISH; write end_flag = 0          (the proxy's release)
// The proxy thread polls the start flags of its queued tasks, acknowledges,
// plans and issues the moves on copy engines, polls their completion event and
// writes FINISH -- on success, on error, or when the deadline passes (the
// watchdog) -- so the stream is always released.  Slots are reused once the
// stream has reset end_flag.
//
// A stream held at a wait blocks the hardware queue it was mapped to, and
// every other stream mapped to that queue with it (CUDA maps streams onto a
// fixed number of queues, CUDA_DEVICE_MAX_CONNECTIONS, in creation order).
// So before acknowledging, while the caller's stream is known to be held at
// the start flag, the proxy records a probe event on each of its candidate
// streams and issues the moves only on streams whose probe completed: a
// queue that lets an event through while the caller waits is not behind it.
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstring>
#include <thread>

#include <cuda.h>  // CUstream / CUdeviceptr types and memop flags; entry points are resolved at run time

#include "comm.h"
#include "hoc_proxy.h"

namespace hoc {

namespace {

using MemOpFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

constexpr uint32_t kStartValue = 1;
constexpr uint32_t kFinishValue = 1;
constexpr int kSlots = 16;
constexpr size_t kFlagBytes = 64;
constexpr auto kTaskDeadline = std::chrono::seconds(10);
constexpr auto kShutdownWait = std::chrono::seconds(60);
constexpr size_t kMaxCandidates = 64;                       // probe streams the proxy may create
constexpr auto kProbePoll = std::chrono::milliseconds(20);   // wait for probes before adding streams
constexpr auto kProbeGiveUp = std::chrono::milliseconds(500);

enum SlotState { kFree = 0, kQueued = 1, kRunning = 2, kReleasing = 3 };

}  // namespace

struct Slot {
  volatile uint32_t* start = nullptr;  // host view of the flags
  volatile uint32_t* end = nullptr;
  CUdeviceptr d_start = 0, d_end = 0;  // device view
  uint64_t* counts = nullptr;          // pinned, k*k
  int state = kFree;
  Bind bind;
  int dtype = 0;
  std::vector<size_t> cap;
  int transpose = 0;
  cudaEvent_t done = nullptr;
  bool stalled = false;  // host-injected: the moves are never reported complete
  std::chrono::steady_clock::time_point deadline;
};

struct Proxy {
  hocComm* c = nullptr;
  int k = 0;
  int device = 0;
  std::mutex mu;
  std::condition_variable cv;
  std::thread th;
  bool closing = false;
  bool orphaned = false;   // the communicator is gone: release tasks without moving data
  bool using_comm = false; // start_task is working with the communicator
  void* pinned = nullptr;
  Slot slots[kSlots];
  size_t next = 0;
  struct Candidate {
    cudaStream_t s = nullptr;
    cudaEvent_t probe = nullptr;
    bool pending = false;  // the last probe has not completed yet
  };
  std::vector<Candidate> cand;
  std::atomic<uint64_t> probes_blocked{0};  // probes found behind a held queue
  uint64_t n_cand = 0;                       // cand.size(), read under mu by other threads
  MemOpFn write32 = nullptr, wait32 = nullptr;
  std::atomic<uint64_t> completed{0}, released{0};
  std::atomic<int> first_error{0};
};

namespace {

void note_error(Proxy* P, int err) {
  int zero = 0;
  P->first_error.compare_exchange_strong(zero, err);
}

void release(Proxy* P, Slot& s, int err) {
  std::atomic_thread_fence(std::memory_order_seq_cst);
  *s.end = kFinishValue;  // always: the stream is never left waiting
  std::atomic_thread_fence(std::memory_order_seq_cst);
  if (err) {
    P->released.fetch_add(1);
    note_error(P, err);
  } else {
    P->completed.fetch_add(1);
  }
  std::lock_guard<std::mutex> lock(P->mu);
  s.state = kReleasing;
}

hocResult_t add_candidate(Proxy* P) {
  Proxy::Candidate q;
  if (cudaStreamCreateWithFlags(&q.s, cudaStreamNonBlocking) != cudaSuccess) return HOC_ERR_CUDA;
  if (cudaEventCreateWithFlags(&q.probe, cudaEventDisableTiming) != cudaSuccess) {
    cudaStreamDestroy(q.s);
    return HOC_ERR_CUDA;
  }
  P->cand.push_back(q);
  std::lock_guard<std::mutex> lock(P->mu);
  P->n_cand = P->cand.size();
  return HOC_SUCCESS;
}

// `need` streams whose queues are not held by any waiting stream right now.
// Called while the caller's stream is held at its start flag.
hocResult_t pick_streams(Proxy* P, size_t need, std::vector<cudaStream_t>* out) {
  const auto give_up = std::chrono::steady_clock::now() + kProbeGiveUp;
  for (;;) {
    for (auto& q : P->cand)
      if (!q.pending) {
        if (cudaEventRecord(q.probe, q.s) != cudaSuccess) return HOC_ERR_CUDA;
        q.pending = true;
      }
    const auto poll_end = std::chrono::steady_clock::now() + kProbePoll;
    for (;;) {
      out->clear();
      for (auto& q : P->cand) {
        if (q.pending) {
          const cudaError_t e = cudaEventQuery(q.probe);
          if (e == cudaSuccess) q.pending = false;
          else if (e != cudaErrorNotReady) return HOC_ERR_CUDA;
        }
        if (!q.pending) out->push_back(q.s);
      }
      if (out->size() >= need) {
        out->resize(need);
        return HOC_SUCCESS;
      }
      if (std::chrono::steady_clock::now() > poll_end) break;
      std::this_thread::yield();
    }
    P->probes_blocked.fetch_add(P->cand.size() - out->size());
    if (std::chrono::steady_clock::now() > give_up || P->cand.size() >= kMaxCandidates) {
      set_error_detail("the proxy found no copy streams outside the held hardware queues");
      return HOC_ERR_UNSUPPORTED;
    }
    for (size_t i = out->size(); i < need + 2 && P->cand.size() < kMaxCandidates; ++i) {
      const hocResult_t r = add_candidate(P);
      if (r != HOC_SUCCESS) return r;
    }
  }
}

// The stream reached the start flag: pick streams, acknowledge, plan and
// issue the moves.
void start_task(Proxy* P, Slot& s) {
  std::atomic_thread_fence(std::memory_order_acquire);
  const int k = P->k;
  std::vector<size_t> cnt(size_t(k) * k);
  for (int a = 0; a < k; ++a)
    for (int b = 0; b < k; ++b)
      cnt[size_t(a) * k + b] = size_t(s.transpose ? s.counts[size_t(b) * k + a] : s.counts[size_t(a) * k + b]);
  std::vector<cudaStream_t> streams;
  const hocResult_t picked = pick_streams(P, size_t(P->c->cfg.n_copy) + 1, &streams);
  *s.start = 0;  // acknowledge: the stream moves on to wait for the end flag
  std::atomic_thread_fence(std::memory_order_seq_cst);
  if (picked != HOC_SUCCESS) {
    release(P, s, picked);
    return;
  }
  {
    std::unique_lock<std::mutex> lock(P->mu);
    if (P->orphaned) {
      lock.unlock();
      release(P, s, HOC_ERR_NOT_INITIALIZED);
      return;
    }
    P->using_comm = true;  // the communicator stays alive until this is cleared
  }
  struct Done {
    Proxy* P;
    ~Done() {
      std::lock_guard<std::mutex> lock(P->mu);
      P->using_comm = false;
      P->cv.notify_all();
    }
  } done_guard{P};
  for (int d = 0; d < k; ++d) {
    size_t col = 0;
    for (int a = 0; a < k; ++a) col += cnt[size_t(a) * k + d];
    if (col > s.cap[d]) {
      release(P, s, HOC_ERR_INVALID_ARG);
      return;
    }
  }
  CallShape shape;
  shape.op = HOC_OP_ALLTOALL;
  shape.k = k;
  shape.dtype = s.dtype;
  shape.counts = cnt;
  hocResult_t r;
  if (P->c->cfg.fault == kFaultProxyStall) {  // injected on the host: a completion that never arrives
    std::lock_guard<std::mutex> lock(P->mu);
    s.stalled = true;
    s.deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(200);
    s.state = kRunning;
    return;
  }
  {
    std::lock_guard<std::mutex> lock(P->c->mu);
    const Plan* plan = nullptr;
    r = get_plan(P->c, shape, &plan);
    int mx = 0;
    const std::vector<cudaStream_t> copy(streams.begin() + 1, streams.end());
    if (r == HOC_SUCCESS) r = issue_plan(P->c, *plan, s.bind, streams[0], &copy, &mx);
    if (r == HOC_SUCCESS && cudaEventRecord(s.done, streams[0]) != cudaSuccess) r = HOC_ERR_CUDA;
  }
  if (r != HOC_SUCCESS) {
    release(P, s, r);
    return;
  }
  std::lock_guard<std::mutex> lock(P->mu);
  s.stalled = false;
  s.deadline = std::chrono::steady_clock::now() + kTaskDeadline;
  s.state = kRunning;
}

void free_resources(Proxy* P) {
  for (Slot& s : P->slots)
    if (s.done) cudaEventDestroy(s.done);
  for (auto& q : P->cand) {
    cudaEventDestroy(q.probe);
    cudaStreamDestroy(q.s);
  }
  P->cand.clear();
  if (P->pinned) cudaFreeHost(P->pinned);
}

void proxy_loop(Proxy* P) {
  cudaSetDevice(P->device);
  for (;;) {
    bool busy = false, all_free = true;
    for (Slot& s : P->slots) {
      int st;
      {
        std::lock_guard<std::mutex> lock(P->mu);
        st = s.state;
      }
      if (st == kFree) continue;
      all_free = false;
      if (st == kQueued) {
        if (*s.start == kStartValue) {
          start_task(P, s);
          busy = true;
        }
      } else if (st == kRunning) {
        const cudaError_t e = s.stalled ? cudaErrorNotReady : cudaEventQuery(s.done);
        if (e == cudaSuccess) {
          release(P, s, 0);
          busy = true;
        } else if (e != cudaErrorNotReady) {
          release(P, s, HOC_ERR_CUDA);
        } else if (std::chrono::steady_clock::now() > s.deadline) {
          release(P, s, HOC_ERR_TIMEOUT);  // watchdog
        }
      } else if (st == kReleasing) {
        if (*s.end == 0) {  // the stream has passed the end flag: slot reusable
          std::lock_guard<std::mutex> lock(P->mu);
          s.state = kFree;
          P->cv.notify_all();
          busy = true;
        }
      }
    }
    bool stop;
    {
      std::lock_guard<std::mutex> lock(P->mu);
      stop = P->closing && all_free;
      if (stop) P->cv.notify_all();
    }
    if (stop) break;
    if (!busy) std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
  bool orphaned;
  {
    std::lock_guard<std::mutex> lock(P->mu);
    orphaned = P->orphaned;
  }
  if (orphaned) {  // nobody else will free the proxy
    free_resources(P);
    delete P;
  }
}

hocResult_t proxy_create(hocComm* c, Proxy** out) {
  Proxy* P = new (std::nothrow) Proxy();
  if (!P) return HOC_ERR_OOM;
  P->c = c;
  P->k = c->k;
  P->device = c->device;
  cudaDriverEntryPointQueryResult q;
  void* fw = nullptr;
  void* fv = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fw, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess ||
      cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &fv, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fw || !fv) {
    delete P;
    set_error_detail("stream memory operations are not available from the driver");
    return HOC_ERR_UNSUPPORTED;
  }
  P->write32 = reinterpret_cast<MemOpFn>(fw);
  P->wait32 = reinterpret_cast<MemOpFn>(fv);
  const size_t counts_bytes = size_t(c->k) * c->k * sizeof(uint64_t);
  const size_t slot_bytes = kFlagBytes + ((counts_bytes + 63) / 64) * 64;
  if (cudaHostAlloc(&P->pinned, slot_bytes * kSlots, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    delete P;
    set_error_detail("cudaHostAlloc of the proxy flags failed");
    return HOC_ERR_OOM;
  }
  memset(P->pinned, 0, slot_bytes * kSlots);
  for (int i = 0; i < kSlots; ++i) {
    char* base = static_cast<char*>(P->pinned) + size_t(i) * slot_bytes;
    Slot& s = P->slots[i];
    s.start = reinterpret_cast<volatile uint32_t*>(base);
    s.end = reinterpret_cast<volatile uint32_t*>(base + 4);
    s.counts = reinterpret_cast<uint64_t*>(base + kFlagBytes);
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, base, 0) != cudaSuccess || cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) {
      free_resources(P);
      delete P;
      set_error_detail("mapping the proxy flags failed");
      return HOC_ERR_CUDA;
    }
    s.d_start = reinterpret_cast<CUdeviceptr>(d);
    s.d_end = reinterpret_cast<CUdeviceptr>(d) + 4;
  }
  for (int i = 0; i < c->cfg.n_copy + 3; ++i)
    if (add_candidate(P) != HOC_SUCCESS) {
      free_resources(P);
      delete P;
      set_error_detail("creating the proxy's copy streams failed");
      return HOC_ERR_CUDA;
    }
  P->th = std::thread(proxy_loop, P);
  *out = P;
  return HOC_SUCCESS;
}

}  // namespace

void proxy_shutdown(hocComm* c) {
  Proxy* P = c->proxy;
  if (!P) return;
  c->proxy = nullptr;
  std::unique_lock<std::mutex> lock(P->mu);
  P->closing = true;
  auto all_free = [P] {
    for (const Slot& s : P->slots)
      if (s.state != kFree) return false;
    return true;
  };
  if (P->cv.wait_for(lock, kShutdownWait, all_free)) {
    lock.unlock();
    P->th.join();
    free_resources(P);
    delete P;
    return;
  }
  // Tasks whose stream never reached its start flag: keep a detached proxy
  // that acknowledges and releases them without moving data (the
  // communicator is gone), so no stream can wait forever on a flag.
  P->orphaned = true;
  P->cv.wait(lock, [P] { return !P->using_comm; });
  lock.unlock();
  P->th.detach();
}

int proxy_take_error(hocComm* c) { return c->proxy ? c->proxy->first_error.exchange(0) : 0; }

}  // namespace hoc

using namespace hoc;

extern "C" hocResult_t hoc_alltoall_device_counts(hocComm_t comm, const void* const* send, void* const* recv,
                                                  const uint64_t* d_sendcounts, int transpose,
                                                  const size_t* recv_capacity, hocDataType_t dtype, void* stream) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!send || !recv || !d_sendcounts || !recv_capacity || dtype_bytes(dtype) == 0) return HOC_ERR_INVALID_ARG;
  const int k = comm->k;
  for (int r = 0; r < k; ++r)
    if (!send[r] || !recv[r]) return HOC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != comm->device) cudaSetDevice(comm->device);
  struct Restore {
    int p, d;
    ~Restore() {
      if (p >= 0 && p != d) cudaSetDevice(p);
    }
  } restore{prev, comm->device};
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return HOC_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) {
    set_error_detail("the device-count all-to-all cannot be captured into a graph");
    return HOC_ERR_UNSUPPORTED;
  }
  {
    std::lock_guard<std::mutex> lock(comm->mu);
    if (!comm->proxy) {
      Proxy* P = nullptr;
      hocResult_t r = proxy_create(comm, &P);
      if (r != HOC_SUCCESS) return r;
      comm->proxy = P;
    }
  }
  Proxy* P = comm->proxy;
  Slot* slot = nullptr;
  {
    std::unique_lock<std::mutex> lock(P->mu);
    Slot& cand = P->slots[P->next % kSlots];
    if (!P->cv.wait_for(lock, std::chrono::seconds(30), [&] { return cand.state == kFree; })) {
      set_error_detail("no free proxy slot within 30 s");
      return HOC_ERR_TIMEOUT;
    }
    ++P->next;
    slot = &cand;
    for (int r = 0; r < k; ++r) {
      slot->bind.send[r] = send[r];
      slot->bind.recv[r] = recv[r];
    }
    slot->dtype = dtype;
    slot->transpose = transpose != 0;
    slot->cap.assign(recv_capacity, recv_capacity + k);
    slot->state = kQueued;
  }
  const size_t counts_bytes = size_t(k) * k * sizeof(uint64_t);
  if (cudaMemcpyAsync(slot->counts, d_sendcounts, counts_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    std::lock_guard<std::mutex> lock(P->mu);
    slot->state = kFree;  // nothing was queued on the stream
    set_error_detail("cudaMemcpyAsync of the device counts failed");
    return HOC_ERR_CUDA;
  }
  CUstream cu = reinterpret_cast<CUstream>(s);
  bool ok = P->write32(cu, slot->d_start, kStartValue, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
  ok = ok && P->wait32(cu, slot->d_start, 0, CU_STREAM_WAIT_VALUE_EQ) == CUDA_SUCCESS;
  ok = ok && P->wait32(cu, slot->d_end, kFinishValue, CU_STREAM_WAIT_VALUE_EQ) == CUDA_SUCCESS;
  ok = ok && P->write32(cu, slot->d_end, 0, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
  if (!ok) {
    set_error_detail("queueing the stream memory operations failed");
    return HOC_ERR_CUDA;
  }
  return HOC_SUCCESS;
}

extern "C" hocResult_t hoc_proxy_status(hocComm_t comm, uint64_t* completed, uint64_t* released_on_error,
                                        hocResult_t* first_error) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  Proxy* P = comm->proxy;
  if (completed) *completed = P ? P->completed.load() : 0;
  if (released_on_error) *released_on_error = P ? P->released.load() : 0;
  if (first_error) *first_error = P ? hocResult_t(P->first_error.exchange(0)) : HOC_SUCCESS;
  return HOC_SUCCESS;
}

extern "C" hocResult_t hoc_proxy_queue_stats(hocComm_t comm, uint64_t* candidates, uint64_t* probes_not_clear) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  Proxy* P = comm->proxy;
  if (candidates) {
    uint64_t n = 0;
    if (P) {
      std::lock_guard<std::mutex> lock(P->mu);
      n = P->n_cand;
    }
    *candidates = n;
  }
  if (probes_not_clear) *probes_not_clear = P ? P->probes_blocked.load() : 0;
  return HOC_SUCCESS;
}
