// Host proxy of the stream-memory-operation handshake (HOCCL section 3.2,
// Fig. 4, Listing 1), serving all-to-all(v) exchanges whose counts are
// computed on the device.  See include/hoc_proxy.h for the contract.
//
// Per task the caller's stream runs, in order:
//   copy counts device -> pinned host slot;
//   write start_flag = START; wait start_flag == 0      (the proxy's ack)
//   wait end_flag == FINISH; write end_flag = 0          (the proxy's release)
//
// Two host threads serve the slots.  The proxy thread polls the start flags of
// queued tasks, acknowledges, plans and issues the moves on its own streams,
// polls their completion event and writes FINISH.  The watchdog thread makes
// no CUDA call at all: when a task is still unreleased at its deadline it
// writes the ack and FINISH itself.  So the stream is released even when the
// proxy thread is stuck inside a driver call that cannot return before the
// held stream drains -- a kernel's first launch under lazy module loading can
// wait for the whole context, and a pageable host copy queued behind the held
// stream blocks its caller until the stream gets past the flags.  Slots are
// reused once the stream has reset end_flag.
//
// Slot states: Free -> Queued (handed to the proxy; the stream has not reached
// the start flag) -> Starting (start flag seen; planning and issuing) ->
// Running (moves issued) -> Releasing (FINISH written) -> Free (the stream
// reset end_flag).  Every transition happens under Proxy::mu; the release
// writes happen under it too, so exactly one thread releases a task.
// If queueing the four stream operations fails part way, the call returns
// HOC_ERR_CUDA and the slot is abandoned: once the stream writes the start
// flag the proxy acknowledges it and, without moving anything, frees the
// slot -- or retires it for good when the stream waits for FINISH but the
// reset of end_flag was never queued (nothing would ever reset it), or when
// not even the start flag was queued (the counts copy may still land in it).
// Retired slots are skipped when a call picks its slot.
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <thread>

#include <cuda.h>  // CUstream / CUdeviceptr types and memop flags; entry points are resolved at run time

#include "comm.h"
#include "hoc_internal.h"
#include "hoc_proxy.h"

namespace hoc {

namespace {

using MemOpFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
using Clock = std::chrono::steady_clock;

constexpr uint32_t kStartValue = 1;
constexpr uint32_t kFinishValue = 1;
constexpr int kSlots = 16;
constexpr size_t kFlagBytes = 64;
constexpr auto kTaskDeadline = std::chrono::seconds(10);
constexpr auto kInjectedDeadline = std::chrono::milliseconds(200);
constexpr auto kInjectedBlock = std::chrono::milliseconds(1500);
constexpr auto kShutdownWait = std::chrono::seconds(60);
// The proxy issues a task's copies only once the stream is at the start flag,
// so the exchange is bound by whichever is longer: issuing the copies (about
// 1.5 us of host time each) or moving the bytes (copy engines, ~5.8 TB/s).
// It sizes the chunks so that a task takes at most about this many copies.
// Measured on the EP round trip (2 x 805 MB exchanges): 96 -> 0.96 ms,
// 48 -> 0.90 ms, 32 -> 0.92 ms.
constexpr size_t kProxyTaskCopies = 48;
constexpr size_t kChunkGrain = size_t(1) << 20;

enum SlotState { kFree = 0, kQueued = 1, kStarting = 2, kRunning = 3, kReleasing = 4, kRetired = 5 };
constexpr int kStreamOps = 4;  // write start, wait ack, wait finish, reset end

const char* const kWhyDeadline =
    "the moves did not finish within 10 s of the stream reaching the start flag; launching a kernel for the first "
    "time while the stream is held (lazy module loading) or queueing a pageable host copy behind it stalls them: "
    "load such kernels beforehand (or set CUDA_MODULE_LOADING=EAGER) and keep blocking copies off the held stream";

}  // namespace

struct Slot {
  volatile uint32_t* start = nullptr;  // host view of the flags
  volatile uint32_t* end = nullptr;
  CUdeviceptr d_start = 0, d_end = 0;  // device view
  uint64_t* counts = nullptr;          // pinned, k*k
  int state = kFree;
  Bind bind;
  int dtype = 0;
  std::vector<size_t> cap;   // receive capacities, elements
  std::vector<size_t> scap;  // send capacities, elements
  int abandoned_ops = 0;     // > 0: queueing failed after this many stream operations
  int transpose = 0;
  cudaEvent_t done = nullptr;
  bool stalled = false;  // host-injected: the moves are never reported complete
  uint64_t task = 0;
  Clock::time_point deadline;
};

struct Proxy {
  hocComm* c = nullptr;
  int k = 0;
  int device = 0;
  int fault = 0;  // the communicator's injected fault, copied: the proxy may outlive it
  bool memop_fault_used = false;  // the stream-operation fault is injected into the first call only
  std::mutex mu;
  std::condition_variable cv;
  std::thread th;        // the proxy thread
  std::thread watchdog;  // host memory only
  bool closing = false;
  bool orphaned = false;    // the communicator is gone: release tasks without moving data
  bool using_comm = false;  // start_task is working with the communicator
  bool stop_watchdog = false;
  void* pinned = nullptr;
  Slot slots[kSlots];
  size_t next = 0;
  cudaStream_t origin = nullptr;   // stream 0 of the proxy's plans
  std::vector<cudaStream_t> copy;  // its copy streams
  MemOpFn write32 = nullptr, wait32 = nullptr;
  std::atomic<uint64_t> completed{0}, released{0};
  int first_error = 0;  // under mu
  std::string why;      // under mu: what the first error was
  bool trace = false;   // HOC_PROXY_TRACE=1: one stderr line per task phase
  uint64_t tasks = 0;
  Clock::time_point t0 = Clock::now();
};

namespace {

void trace(Proxy* P, const Slot& s, const char* what) {
  if (!P->trace) return;
  const double ms = std::chrono::duration<double, std::milli>(Clock::now() - P->t0).count();
  fprintf(stderr, "[hoc proxy %.3f ms] task %llu slot %d: %s\n", ms, (unsigned long long)s.task, int(&s - P->slots),
          what);
}

// Write the release (ack and FINISH) of a task the proxy still holds.  The
// caller holds P->mu.  Returns false if the task was already released.
bool release_locked(Proxy* P, Slot& s, int err, const char* why) {
  if (s.state != kStarting && s.state != kRunning) return false;
  std::atomic_thread_fence(std::memory_order_seq_cst);
  *s.start = 0;  // no-op once acknowledged; frees a stream still at the start flag
  *s.end = kFinishValue;
  std::atomic_thread_fence(std::memory_order_seq_cst);
  s.state = kReleasing;
  if (err) {
    P->released.fetch_add(1);
    if (!P->first_error) {
      P->first_error = err;
      P->why = why ? why : "";
    }
  } else {
    P->completed.fetch_add(1);
  }
  return true;
}

void release(Proxy* P, Slot& s, int err, const char* why) {
  std::lock_guard<std::mutex> lock(P->mu);
  release_locked(P, s, err, why);
}

// The stream reached the start flag: acknowledge, plan and issue the moves.
void start_task(Proxy* P, Slot& s) {
  bool block = false;
  {
    std::lock_guard<std::mutex> lock(P->mu);
    if (s.state != kQueued) return;
    s.state = kStarting;
    s.task = ++P->tasks;
    block = P->fault == kFaultProxyBlock;
    const bool injected = P->fault == kFaultProxyStall || block;
    s.deadline = Clock::now() + (injected ? Clock::duration(kInjectedDeadline) : Clock::duration(kTaskDeadline));
  }
  trace(P, s, "start flag seen");
  std::atomic_thread_fence(std::memory_order_acquire);
  const int k = P->k;
  std::vector<size_t> cnt(size_t(k) * k);
  for (int a = 0; a < k; ++a)
    for (int b = 0; b < k; ++b)
      cnt[size_t(a) * k + b] = size_t(s.transpose ? s.counts[size_t(b) * k + a] : s.counts[size_t(a) * k + b]);
  // Injected on the host: the proxy thread is held up past the deadline, as in
  // a driver call that waits for the held stream; the watchdog must release.
  if (block) std::this_thread::sleep_for(kInjectedBlock);
  {
    std::lock_guard<std::mutex> lock(P->mu);
    if (s.state != kStarting) return;  // the watchdog released it meanwhile
    *s.start = 0;                      // acknowledge: the stream moves on to wait for the end flag
    std::atomic_thread_fence(std::memory_order_seq_cst);
    if (P->orphaned) {
      release_locked(P, s, HOC_ERR_NOT_INITIALIZED, "the communicator was destroyed before the task started");
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
    size_t col = 0;  // stays <= cap[d]: each count is compared with the room left, so no sum wraps
    for (int a = 0; a < k; ++a) {
      const size_t c = cnt[size_t(a) * k + d];
      if (c > s.cap[d] - col) {
        release(P, s, HOC_ERR_INVALID_ARG, "a receiver's total count exceeds its capacity; nothing was moved");
        return;
      }
      col += c;
    }
  }
  for (int a = 0; a < k; ++a) {  // the same for what each source reads from its send buffer
    size_t row = 0;
    for (int d = 0; d < k; ++d) {
      const size_t c = cnt[size_t(a) * k + d];
      if (c > s.scap[a] - row) {
        release(P, s, HOC_ERR_INVALID_ARG, "a sender's total count exceeds its send buffer; nothing was moved");
        return;
      }
      row += c;
    }
  }
  if (P->fault == kFaultProxyStall) {  // injected on the host: a completion that never arrives
    std::lock_guard<std::mutex> lock(P->mu);
    if (s.state == kStarting) {
      s.stalled = true;
      s.state = kRunning;
    }
    return;
  }
  CallShape shape;
  shape.op = HOC_OP_ALLTOALL;
  shape.k = k;
  shape.dtype = s.dtype;
  size_t total = 0;
  for (size_t v : cnt) total += v;
  total *= dtype_bytes(s.dtype);
  const size_t want = (total / kProxyTaskCopies + kChunkGrain - 1) / kChunkGrain * kChunkGrain;
  if (want > chunk_for(P->c->cfg, HOC_PATH_CE)) shape.chunk = want;
  shape.counts = cnt;
  hocResult_t r;
  {
    std::lock_guard<std::mutex> lock(P->c->mu);
    const Plan* plan = nullptr;
    r = get_plan(P->c, shape, &plan);
    int mx = 0;
    if (r == HOC_SUCCESS) r = issue_plan(P->c, *plan, s.bind, P->origin, &P->copy, &mx);
    if (r == HOC_SUCCESS && cudaEventRecord(s.done, P->origin) != cudaSuccess) r = HOC_ERR_CUDA;
  }
  if (r != HOC_SUCCESS) {
    release(P, s, r, "planning or issuing the moves failed");
    return;
  }
  trace(P, s, "moves issued");
  std::lock_guard<std::mutex> lock(P->mu);
  if (s.state == kStarting) {
    s.stalled = false;
    s.state = kRunning;
  }
}

// The stream of an abandoned slot reached its start flag: let it pass without
// moving anything.  The caller holds P->mu.
void abandon_locked(Proxy* P, Slot& s) {
  std::atomic_thread_fence(std::memory_order_seq_cst);
  *s.start = 0;                   // the ack, if the stream waits for it
  if (s.abandoned_ops >= 3) {     // the stream waits for FINISH, but nothing will reset end_flag
    *s.end = kFinishValue;
    s.state = kRetired;
  } else {                        // nothing waits on end_flag
    s.state = kFree;
  }
  std::atomic_thread_fence(std::memory_order_seq_cst);
  s.abandoned_ops = 0;
  P->cv.notify_all();
}

void free_resources(Proxy* P) {
  for (Slot& s : P->slots)
    if (s.done) cudaEventDestroy(s.done);
  for (cudaStream_t s : P->copy) cudaStreamDestroy(s);
  P->copy.clear();
  if (P->origin) cudaStreamDestroy(P->origin);
  if (P->pinned) cudaFreeHost(P->pinned);
}

void watchdog_loop(Proxy* P) {
  std::unique_lock<std::mutex> lock(P->mu);
  while (!P->stop_watchdog) {
    const auto now = Clock::now();
    for (Slot& s : P->slots) {
      if ((s.state != kStarting && s.state != kRunning) || now <= s.deadline) continue;
      const bool issued = s.state == kRunning;
      release_locked(P, s, HOC_ERR_TIMEOUT, issued ? kWhyDeadline : "the proxy did not issue the moves before the deadline");
      if (P->trace)
        fprintf(stderr, "[hoc proxy] task %llu slot %d: deadline passed, the watchdog released the stream\n",
                (unsigned long long)s.task, int(&s - P->slots));
    }
    P->cv.wait_for(lock, std::chrono::milliseconds(1));
  }
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
      if (st == kFree || st == kRetired) continue;
      all_free = false;
      if (st == kQueued) {
        if (*s.start == kStartValue) {
          bool abandoned;
          {
            std::lock_guard<std::mutex> lock(P->mu);
            abandoned = s.abandoned_ops > 0;
            if (abandoned) abandon_locked(P, s);
          }
          if (!abandoned) start_task(P, s);
          busy = true;
        }
      } else if (st == kRunning) {
        const cudaError_t e = s.stalled ? cudaErrorNotReady : cudaEventQuery(s.done);
        if (e == cudaSuccess) {
          trace(P, s, "moves complete, releasing");
          release(P, s, 0, nullptr);
          busy = true;
        } else if (e != cudaErrorNotReady) {
          release(P, s, HOC_ERR_CUDA, "querying the completion event of the moves failed");
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
      std::unique_lock<std::mutex> lock(P->mu);
      stop = P->closing && all_free;
      if (stop) {
        P->stop_watchdog = true;
        P->cv.notify_all();
      } else if (all_free) {
        // idle: sleep until a task is queued (or shutdown), re-checking every ms
        P->cv.wait_for(lock, std::chrono::milliseconds(1));
      }
    }
    if (stop) break;
    if (!busy && !all_free) std::this_thread::yield();  // tasks in flight: poll their flags closely
  }
  P->watchdog.join();
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

// Every kernel of the library, loaded once per device before the first task.
hocResult_t preload_kernels(int device) {
  static std::mutex mu;
  static uint64_t loaded = 0;  // bit per device
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t bit = device < 64 ? (uint64_t(1) << device) : 0;
  if (loaded & bit) return HOC_SUCCESS;
  cudaError_t e = reduce_preload();
  if (e == cudaSuccess) e = tma_preload();
  if (e == cudaSuccess) e = ep_preload();
  if (e == cudaSuccess) e = workload_preload();
  if (e != cudaSuccess) {
    set_error_detail("loading the library's kernels before starting the proxy failed");
    return HOC_ERR_CUDA;
  }
  loaded |= bit;
  return HOC_SUCCESS;
}

hocResult_t proxy_create(hocComm* c, Proxy** out) {
  const hocResult_t pre = preload_kernels(c->device);
  if (pre != HOC_SUCCESS) return pre;
  Proxy* P = new (std::nothrow) Proxy();
  if (!P) return HOC_ERR_OOM;
  P->c = c;
  P->k = c->k;
  P->device = c->device;
  P->fault = c->cfg.fault;
  const char* tr = getenv("HOC_PROXY_TRACE");
  P->trace = tr && atoi(tr) != 0;
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
    if (cudaHostGetDevicePointer(&d, base, 0) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) {
      free_resources(P);
      delete P;
      set_error_detail("mapping the proxy flags failed");
      return HOC_ERR_CUDA;
    }
    s.d_start = reinterpret_cast<CUdeviceptr>(d);
    s.d_end = reinterpret_cast<CUdeviceptr>(d) + 4;
  }
  bool ok = cudaStreamCreateWithFlags(&P->origin, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < c->cfg.n_copy; ++i) {
    cudaStream_t s = nullptr;
    ok = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess;
    if (ok) P->copy.push_back(s);
  }
  if (!ok) {
    free_resources(P);
    delete P;
    set_error_detail("creating the proxy's streams failed");
    return HOC_ERR_CUDA;
  }
  P->watchdog = std::thread(watchdog_loop, P);
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
      if (s.state != kFree && s.state != kRetired) return false;
    return true;
  };
  if (P->cv.wait_for(lock, kShutdownWait, all_free)) {
    lock.unlock();
    P->th.join();  // the proxy thread joins the watchdog before it returns
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

int proxy_take_error(hocComm* c, std::string* why) {
  Proxy* P = c->proxy;
  if (!P) return 0;
  std::lock_guard<std::mutex> lock(P->mu);
  const int e = P->first_error;
  if (why) *why = P->why;
  P->first_error = 0;
  P->why.clear();
  return e;
}

}  // namespace hoc

using namespace hoc;

extern "C" hocResult_t hoc_alltoall_device_counts(hocComm_t comm, const void* const* send, void* const* recv,
                                                  const uint64_t* d_sendcounts, int transpose,
                                                  const size_t* send_capacity, const size_t* recv_capacity,
                                                  hocDataType_t dtype, void* stream) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (!send || !recv || !d_sendcounts || !send_capacity || !recv_capacity || dtype_bytes(dtype) == 0)
    return HOC_ERR_INVALID_ARG;
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
  int inject_fail_at = 0;  // host-injected: the stream operation of this number (1-based) fails to queue
  {
    std::unique_lock<std::mutex> lock(P->mu);
    const auto give_up = Clock::now() + std::chrono::seconds(30);
    while (!slot) {  // the next slot in turn that is not retired, once it is free
      Slot* cand = nullptr;
      for (int i = 0; i < kSlots && !cand; ++i) {
        Slot& c2 = P->slots[(P->next + i) % kSlots];
        if (c2.state != kRetired) {
          cand = &c2;
          P->next += i;
        }
      }
      if (!cand) {
        set_error_detail("every proxy slot was retired after stream operations failed to queue");
        return HOC_ERR_CUDA;
      }
      if (!P->cv.wait_until(lock, give_up, [&] { return cand->state == kFree || cand->state == kRetired; })) {
        set_error_detail("no free proxy slot within 30 s");
        return HOC_ERR_TIMEOUT;
      }
      if (cand->state == kFree) slot = cand;
    }
    ++P->next;
    if ((P->fault == kFaultProxyMemop || P->fault == kFaultProxyMemopReset) && !P->memop_fault_used) {
      P->memop_fault_used = true;
      inject_fail_at = P->fault == kFaultProxyMemop ? 3 : 4;
    }
    for (int r = 0; r < k; ++r) {
      slot->bind.send[r] = send[r];
      slot->bind.recv[r] = recv[r];
    }
    slot->dtype = dtype;
    slot->transpose = transpose != 0;
    slot->cap.assign(recv_capacity, recv_capacity + k);
    slot->scap.assign(send_capacity, send_capacity + k);
    slot->abandoned_ops = 0;
    slot->state = kQueued;
    P->cv.notify_all();  // wake an idle proxy thread
  }
  const size_t counts_bytes = size_t(k) * k * sizeof(uint64_t);
  if (cudaMemcpyAsync(slot->counts, d_sendcounts, counts_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    std::lock_guard<std::mutex> lock(P->mu);
    slot->state = kFree;  // nothing was queued on the stream
    set_error_detail("cudaMemcpyAsync of the device counts failed");
    return HOC_ERR_CUDA;
  }
  CUstream cu = reinterpret_cast<CUstream>(s);
  int queued = 0;  // stream operations queued so far, in order
  for (int op = 1; op <= kStreamOps; ++op) {
    if (op == inject_fail_at) break;
    CUresult e;
    switch (op) {
      case 1: e = P->write32(cu, slot->d_start, kStartValue, CU_STREAM_WRITE_VALUE_DEFAULT); break;
      case 2: e = P->wait32(cu, slot->d_start, 0, CU_STREAM_WAIT_VALUE_EQ); break;
      case 3: e = P->wait32(cu, slot->d_end, kFinishValue, CU_STREAM_WAIT_VALUE_EQ); break;
      default: e = P->write32(cu, slot->d_end, 0, CU_STREAM_WRITE_VALUE_DEFAULT); break;
    }
    if (e != CUDA_SUCCESS) break;
    ++queued;
  }
  if (queued < kStreamOps) {
    std::lock_guard<std::mutex> lock(P->mu);
    if (queued == 0) {
      // The stream will never write the start flag, but the counts copy queued
      // on it may still land in the slot: retire it rather than hand it out.
      slot->state = kRetired;
    } else {
      slot->abandoned_ops = queued;  // the proxy lets the stream pass its flags and moves nothing
    }
    P->cv.notify_all();
    set_error_detail("queueing the stream memory operations failed; nothing will be moved");
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
  if (first_error) *first_error = hocResult_t(proxy_take_error(comm, nullptr));
  return HOC_SUCCESS;
}
