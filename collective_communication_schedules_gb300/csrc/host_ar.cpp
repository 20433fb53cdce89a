// AllReduce over host buffers.
//
// Direct mode (path AUTO or FUSED, when the device can address every host
// buffer: pinned memory, or any memory over a coherent host link with
// pageable access such as Grace's NVLink-C2C): one fused reduce launch loads
// the k inputs from host memory and stores the k results there -- the same
// kernel, fold and bits as the device allreduce, and no staging.
//
// Staged mode (path CE or TMA, or host buffers the device cannot address):
// the k-way reduce pipelined with copy-engine copies that bring the inputs in
// and the results out.
//
// The element range is cut into chunks.  Chunk q runs three steps on three
// internal streams: the host->device copies of the k input chunks into a
// staging slot (copy engine, one direction), the ring-order reduce of that
// slot into one output chunk (SMs, the same fold and bits as hoc_allreduce),
// and the device->host copies of the output chunk into the k host results
// (copy engine, other direction).  Two staging slots let the input copies of
// chunk q+1, the reduce of chunk q and the output copies of chunk q-1 run at
// the same time.  Ordering against the caller's stream uses events (fork and
// join), as for every other call; each call's issue sequence is captured once
// as a CUDA graph and replayed.
#include <algorithm>
#include <cstring>

#include "comm.h"
#include "hoc.h"

namespace hoc {
namespace {

constexpr size_t kHostChunkBytes = size_t(8) << 20;  // per rank and chunk

// The address under which the device loads and stores host buffer `p`, if it
// has one: registered (pinned) memory, device or managed memory, or pageable
// memory when the device can access pageable memory.
bool device_view(const void* p, bool pageable_ok, const void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  switch (a.type) {
    case cudaMemoryTypeHost:
      if (!a.devicePointer) return false;
      *out = a.devicePointer;
      return true;
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged: *out = p; return true;
    default:
      if (!pageable_ok) return false;
      *out = p;
      return true;
  }
}
constexpr int kEventRing = 4;

struct HostArState {
  cudaStream_t h2d = nullptr, red = nullptr, d2h = nullptr, origin = nullptr;
  void* stage = nullptr;  // 2 slots x (k inputs + 1 output) x kHostChunkBytes
  std::vector<cudaEvent_t> ev;  // 3 kinds x kEventRing, then fork / joins
  std::unordered_map<std::string, cudaGraphExec_t> graphs;
  int ctas_per_sm = 0;  // of the reduce kernel for the dtype of the current call
};

#define HCK(call)                                  \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) {                       \
      set_error_detail(#call);                     \
      return HOC_ERR_CUDA;                         \
    }                                              \
  } while (0)

hocResult_t ensure_state(hocComm* c, HostArState** out) {
  if (c->host_ar) {
    *out = static_cast<HostArState*>(c->host_ar);
    return HOC_SUCCESS;
  }
  HostArState* st = new (std::nothrow) HostArState();
  if (!st) return HOC_ERR_OOM;
  c->host_ar = st;  // freed by host_ar_free even if set-up stops half way
  HCK(cudaStreamCreateWithFlags(&st->h2d, cudaStreamNonBlocking));
  HCK(cudaStreamCreateWithFlags(&st->red, cudaStreamNonBlocking));
  HCK(cudaStreamCreateWithFlags(&st->d2h, cudaStreamNonBlocking));
  HCK(cudaStreamCreateWithFlags(&st->origin, cudaStreamNonBlocking));
  const size_t bytes = 2 * size_t(c->k + 1) * kHostChunkBytes;
  if (cudaMalloc(&st->stage, bytes) != cudaSuccess) {
    cudaGetLastError();
    set_error_detail("cudaMalloc of the host-allreduce staging slots failed");
    return HOC_ERR_OOM;
  }
  st->ev.resize(3 * kEventRing + 4, nullptr);
  for (auto& e : st->ev) HCK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  *out = st;
  return HOC_SUCCESS;
}

char* slot_in(HostArState* st, int k, int slot, int r) {
  return static_cast<char*>(st->stage) + (size_t(slot) * (k + 1) + r) * kHostChunkBytes;
}
char* slot_out(HostArState* st, int k, int slot) { return slot_in(st, k, slot, k); }

// Issue the whole pipeline with stream 0 = s0.
hocResult_t issue_host_ar(hocComm* c, HostArState* st, const void* const* hs, void* const* hr, size_t count,
                          int dtype, cudaStream_t s0, int* kernels, int* copies, int* max_ctas) {
  const int k = c->k;
  const size_t b = dtype_bytes(dtype);
  const int lanes = dtype_lanes(dtype);
  size_t ce = kHostChunkBytes / b;
  ce -= ce % 16;
  std::vector<size_t> sz, off;
  block_partition(count, k, &sz, &off);
  std::vector<int> pos(k);
  for (int i = 0; i < k; ++i) pos[c->cfg.order[i]] = i;
  cudaEvent_t* evH = &st->ev[0];
  cudaEvent_t* evC = &st->ev[kEventRing];
  cudaEvent_t* evD = &st->ev[2 * kEventRing];
  cudaEvent_t fork = st->ev[3 * kEventRing], jH = st->ev[3 * kEventRing + 1], jC = st->ev[3 * kEventRing + 2],
              jD = st->ev[3 * kEventRing + 3];
  HCK(cudaEventRecord(fork, s0));
  HCK(cudaStreamWaitEvent(st->h2d, fork, 0));
  HCK(cudaStreamWaitEvent(st->red, fork, 0));
  HCK(cudaStreamWaitEvent(st->d2h, fork, 0));
  const size_t nq = (count + ce - 1) / ce;
  for (size_t q = 0; q < nq; ++q) {
    const int slot = int(q & 1);
    const size_t lo = q * ce, len = std::min(ce, count - lo);
    // inputs of chunk q into the slot, once the reduce of chunk q-2 has read it
    if (q >= 2) HCK(cudaStreamWaitEvent(st->h2d, evC[(q - 2) % kEventRing], 0));
    for (int r = 0; r < k; ++r) {
      HCK(cudaMemcpyAsync(slot_in(st, k, slot, r), static_cast<const char*>(hs[r]) + lo * b, len * b,
                          cudaMemcpyHostToDevice, st->h2d));
      ++*copies;
    }
    HCK(cudaEventRecord(evH[q % kEventRing], st->h2d));
    // reduce: one segment per block the chunk touches, all into the output chunk
    HCK(cudaStreamWaitEvent(st->red, evH[q % kEventRing], 0));
    if (q >= 2) HCK(cudaStreamWaitEvent(st->red, evD[(q - 2) % kEventRing], 0));
    ReduceParams rp;
    memset(&rp, 0, sizeof rp);
    rp.k = k;
    rp.dtype = dtype;
    rp.broadcast = 0;
    for (int r = 0; r < k; ++r) {
      rp.in[r] = slot_in(st, k, slot, r);
      rp.out[r] = slot_out(st, k, slot);
      for (int j = 0; j < k; ++j) rp.seq[r][j] = uint8_t(c->cfg.order[(pos[r] + 1 + j) % k]);
    }
    for (int r = 0; r < k; ++r) {
      const size_t a = std::max(lo, off[r]), z = std::min(lo + len, off[r] + sz[r]);
      if (a >= z) continue;
      ReduceSeg g{a - lo, z - a, a - lo, uint32_t(r), 0};
      g.vec = (g.elem_off % lanes) == (g.out_off % lanes) ? 1u : 0u;  // staging slots are 256-byte aligned
      rp.seg[rp.nseg] = g;
      rp.tile_start[rp.nseg + 1] = rp.tile_start[rp.nseg] + reduce_seg_tiles(dtype, g, false);
      ++rp.nseg;
    }
    const uint64_t tiles = rp.tile_start[rp.nseg];
    const int grid = int(std::min<uint64_t>(tiles, uint64_t(c->sms) * st->ctas_per_sm));
    if (grid > 0) {
      HCK(launch_reduce(rp, grid, false, st->red, false));
      ++*kernels;
      *max_ctas = std::max(*max_ctas, grid);
    }
    HCK(cudaEventRecord(evC[q % kEventRing], st->red));
    // results of chunk q out to every rank's host buffer
    HCK(cudaStreamWaitEvent(st->d2h, evC[q % kEventRing], 0));
    for (int r = 0; r < k; ++r) {
      HCK(cudaMemcpyAsync(static_cast<char*>(hr[r]) + lo * b, slot_out(st, k, slot), len * b, cudaMemcpyDeviceToHost,
                          st->d2h));
      ++*copies;
    }
    HCK(cudaEventRecord(evD[q % kEventRing], st->d2h));
  }
  HCK(cudaEventRecord(jH, st->h2d));
  HCK(cudaEventRecord(jC, st->red));
  HCK(cudaEventRecord(jD, st->d2h));
  HCK(cudaStreamWaitEvent(s0, jH, 0));
  HCK(cudaStreamWaitEvent(s0, jC, 0));
  HCK(cudaStreamWaitEvent(s0, jD, 0));
  return HOC_SUCCESS;
}

}  // namespace

void host_ar_free(hocComm* c) {
  HostArState* st = static_cast<HostArState*>(c->host_ar);
  if (!st) return;
  for (auto& g : st->graphs) cudaGraphExecDestroy(g.second);
  for (cudaEvent_t e : st->ev)
    if (e) cudaEventDestroy(e);
  for (cudaStream_t s : {st->h2d, st->red, st->d2h, st->origin})
    if (s) cudaStreamDestroy(s);
  if (st->stage) cudaFree(st->stage);
  delete st;
  c->host_ar = nullptr;
}

}  // namespace hoc

using namespace hoc;

extern "C" hocResult_t hoc_allreduce_host(hocComm_t comm, const void* const* h_send, void* const* h_recv,
                                          size_t count, hocDataType_t dtype, hocRedOp_t op, void* stream) {
  if (!comm) return HOC_ERR_NOT_INITIALIZED;
  if (dtype != HOC_INT32 && dtype != HOC_FLOAT32 && dtype != HOC_BFLOAT16) return HOC_ERR_INVALID_ARG;
  if (op != HOC_SUM) return HOC_ERR_UNSUPPORTED;
  if (count == 0) return HOC_SUCCESS;
  const int k = comm->k;
  if (!h_send || !h_recv) return HOC_ERR_INVALID_ARG;
  const size_t b = dtype_bytes(dtype);
  for (int r = 0; r < k; ++r)
    if (!h_send[r] || !h_recv[r]) return HOC_ERR_INVALID_ARG;
  if (count > kMaxSpanBytes / b) {  // the staged pipeline issues its copies without a plan
    set_error_detail("a rank's buffer span exceeds 2^40 bytes");
    return HOC_ERR_INVALID_ARG;
  }
  // A result buffer may only coincide with its own input (in place); it may
  // not overlap any other input or result.
  for (int r = 0; r < k; ++r) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(h_recv[r]);
    for (int s = 0; s < k; ++s) {
      const uintptr_t ri = reinterpret_cast<uintptr_t>(h_recv[s]);
      const uintptr_t si = reinterpret_cast<uintptr_t>(h_send[s]);
      const bool hit_recv = s != r && a < ri + count * b && ri < a + count * b;
      const bool hit_send = !(s == r && si == a) && a < si + count * b && si < a + count * b;
      if (hit_recv || hit_send) {
        set_error_detail("host result buffers overlap");
        return HOC_ERR_INVALID_ARG;
      }
    }
  }
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != comm->device) cudaSetDevice(comm->device);
  struct Restore {
    int p, d;
    ~Restore() {
      if (p >= 0 && p != d) cudaSetDevice(p);
    }
  } restore{prev, comm->device};
  const int path = comm->cfg.path;
  if (path == HOC_PATH_AUTO || path == HOC_PATH_FUSED) {
    int pageable = 0;
    cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, comm->device);
    std::vector<const void*> ds(k), dr(k);
    std::vector<void*> drw(k);
    bool direct = true;
    for (int r = 0; r < k && direct; ++r)
      direct = device_view(h_send[r], pageable != 0, &ds[r]) && device_view(h_recv[r], pageable != 0, &dr[r]);
    for (int r = 0; r < k && direct; ++r) drw[r] = const_cast<void*>(dr[r]);
    if (direct) return allreduce_fused(comm, ds.data(), drw.data(), count, dtype, static_cast<cudaStream_t>(stream));
    if (path == HOC_PATH_FUSED) {
      set_error_detail("the FUSED host allreduce needs host buffers the device can address (pinned, or pageable memory on a device with pageable access)");
      return HOC_ERR_UNSUPPORTED;
    }
  }
  std::lock_guard<std::mutex> lock(comm->mu);
  HostArState* st = nullptr;
  hocResult_t r0 = ensure_state(comm, &st);
  if (r0 != HOC_SUCCESS) return r0;
  st->ctas_per_sm = reduce_ctas_per_sm(dtype, k, 0);  // an occupancy query: never inside a capture
  cudaStream_t s0 = static_cast<cudaStream_t>(stream);
  hocOpStats_t stats{};
  stats.path = HOC_PATH_FUSED;
  stats.bytes_exec = 2 * size_t(k) * count * b + (size_t(k) + 1) * count * b;  // copies in/out + reduce
  stats.bytes_min = stats.bytes_exec;
  int kernels = 0, copies = 0, max_ctas = 0;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s0, &cs) != cudaSuccess) return HOC_ERR_CUDA;
  if (!comm->cfg.use_graphs || comm->profiling || cs != cudaStreamCaptureStatusNone) {
    hocResult_t r = issue_host_ar(comm, st, h_send, h_recv, count, dtype, s0, &kernels, &copies, &max_ctas);
    if (r != HOC_SUCCESS) return r;
  } else {
    std::string key(reinterpret_cast<const char*>(&count), sizeof count);
    key.append(reinterpret_cast<const char*>(&dtype), sizeof dtype);
    key.append(reinterpret_cast<const char*>(h_send), sizeof(void*) * k);
    key.append(reinterpret_cast<const char*>(h_recv), sizeof(void*) * k);
    auto it = st->graphs.find(key);
    if (it == st->graphs.end()) {
      if (st->graphs.size() >= 8) {
        for (auto& old : st->graphs) cudaGraphExecDestroy(old.second);
        st->graphs.clear();
      }
      if (cudaStreamBeginCapture(st->origin, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return HOC_ERR_CUDA;
      hocResult_t r = issue_host_ar(comm, st, h_send, h_recv, count, dtype, st->origin, &kernels, &copies, &max_ctas);
      cudaGraph_t g = nullptr;
      const cudaError_t e = cudaStreamEndCapture(st->origin, &g);
      if (r != HOC_SUCCESS || e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return r != HOC_SUCCESS ? r : HOC_ERR_CUDA;
      }
      cudaGraphExec_t exec = nullptr;
      const cudaError_t ei = cudaGraphInstantiate(&exec, g, 0);
      cudaGraphDestroy(g);
      if (ei != cudaSuccess) return HOC_ERR_CUDA;
      it = st->graphs.emplace(key, exec).first;
    } else {
      stats.graph_replayed = 1;
      const size_t ce = (kHostChunkBytes / b) - (kHostChunkBytes / b) % 16;
      const size_t nq = (count + ce - 1) / ce;
      kernels = int(nq);
      copies = int(2 * nq * k);
      max_ctas = comm->sms * st->ctas_per_sm;
    }
    if (cudaGraphLaunch(it->second, s0) != cudaSuccess) return HOC_ERR_CUDA;
  }
  stats.kernels = kernels;
  stats.copies = copies;
  stats.max_ctas = max_ctas;
  stats.sms_used = std::min(max_ctas, comm->sms);
  comm->last = stats;
  return HOC_SUCCESS;
}
