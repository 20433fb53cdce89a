// SM-driven chunk mover: bulk asynchronous copies (cp.async.bulk) through
// shared memory, the comparison path to the copy-engine executor.
//
// HOCCL's point-to-point executor (section 3.3) moves every chunk with a DMA
// engine so that no SM takes part.  This kernel does the same moves from SMs,
// the way SM-based communication libraries do (section 2.2.1, Fig. 1a), but
// with the Blackwell tensor-memory accelerator: one thread per CTA issues
// global->shared bulk loads that complete on an mbarrier, then shared->global
// bulk stores, keeping kStages pieces in flight.  A CTA has two warps: lane 0
// of warp 0 drives the bulk pipeline; warp 1 copies the bytes a bulk copy
// cannot take (heads and tails that are not 16-byte aligned, and jobs whose
// source and destination are aligned differently).
//
// Every wait is bounded by the global timer (p.wait_ns).  On a timeout the
// kernel writes a status code to p.status, waits (again bounded) for its own
// copies in flight and returns; the host reports HOC_ERR_TIMEOUT.  A host-side
// fault injection (p.tx_pad > 0) makes every mbarrier expect more bytes than
// its load delivers, so the phase never completes and this path runs without
// any fault on the GPU.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "hoc_internal.h"
#include "ptx_async.cuh"

namespace hoc {
namespace {

// Pieces in flight per CTA (one CTA per SM, 192 KiB of shared memory).  Measured on GB300: the
// all-gather moves of 8 x 32 MiB blocks run at 5.93-5.96 TB/s with 4, 6 or 8 stages alike, and the
// TMA allreduce, whose moves interleave with the reduce kernels, takes 0.679 ms with 6 stages
// against 0.695 with 4 (3 stages on two CTAs per SM: 0.685; 8 x 16 KiB: 0.714).  Neither 2-3 CTAs
// per SM (2-4 stages of 16-32 KiB each) nor 2-3 store groups in flight moved the all-gather or a
// 1-SM copy, which stays at about 52 GB/s: one SM writes at most about 63 GB/s, by bulk stores or
// by plain 16-byte stores alike.
constexpr int kStages = 6;
constexpr uint32_t kPieceBytes = 32768;
constexpr int kCopyThreads = 64;

using namespace ptx;

__host__ __device__ inline bool co_aligned(const CopyJob& j) {
  return ((reinterpret_cast<uintptr_t>(j.src) ^ reinterpret_cast<uintptr_t>(j.dst)) & 15u) == 0;
}
__host__ __device__ inline uint64_t job_head(const CopyJob& j) {
  const uint64_t mis = reinterpret_cast<uintptr_t>(j.src) & 15u;
  const uint64_t h = mis ? 16 - mis : 0;
  return h > j.bytes ? j.bytes : h;
}
__host__ __device__ inline uint64_t job_body(const CopyJob& j) { return (j.bytes - job_head(j)) & ~uint64_t(15); }
__host__ __device__ inline uint64_t job_pieces(const CopyJob& j, uint32_t pb) {
  if (j.bytes == 0) return 0;
  const uint64_t span = co_aligned(j) ? job_body(j) : j.bytes;
  const uint64_t n = (span + pb - 1) / pb;
  return n ? n : 1;
}

// Which job owns global piece `pc`, and the piece's index inside it.
__device__ __forceinline__ int find_job(const CopyParams& p, uint64_t pc) {
  int lo = 0, hi = p.njobs - 1;
  while (lo < hi) {  // last job with piece_start <= pc
    const int mid = (lo + hi + 1) >> 1;
    if (p.piece_start[mid] <= pc) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bulk part of a piece: `n` bytes at offset `o` of job `j` (n == 0: none).
__device__ __forceinline__ void piece_bulk(const CopyParams& p, uint64_t pc, int& j, uint64_t& o, uint32_t& n) {
  j = find_job(p, pc);
  const CopyJob& jb = p.job[j];
  n = 0;
  if (!co_aligned(jb)) return;
  const uint64_t i = pc - p.piece_start[j];
  const uint64_t body = job_body(jb);
  const uint64_t off = i * p.piece_bytes;
  if (off >= body) return;
  const uint64_t len = body - off < p.piece_bytes ? body - off : p.piece_bytes;
  o = job_head(jb) + off;
  n = static_cast<uint32_t>(len);
}

__device__ __forceinline__ void copy_bytes(const char* src, char* dst, uint64_t n, int lane) {
  for (uint64_t i = lane; i < n; i += 32) dst[i] = src[i];
}

// [off, off + n) of a job's source to the same range of each of its destinations.
__device__ __forceinline__ void copy_bytes_all(const CopyParams& p, const CopyJob& jb, uint64_t off, uint64_t n,
                                               int lane) {
  copy_bytes(jb.src + off, jb.dst + off, n, lane);
  for (int e = 0; e < jb.nmore; ++e) copy_bytes(jb.src + off, p.more_dst[jb.more_at + e] + off, n, lane);
}

__global__ void __launch_bounds__(kCopyThreads, 1) tma_copy_kernel(const __grid_constant__ CopyParams p) {
  extern __shared__ __align__(128) unsigned char stage_mem[];
  __shared__ __align__(8) uint64_t bar[kStages];
  const uint64_t total = p.piece_start[p.njobs];
  const uint64_t mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 1) {
    // Bytes outside the bulk bodies.
    for (uint64_t i = 0; i < mine; ++i) {
      const uint64_t pc = blockIdx.x + i * gridDim.x;
      const int j = find_job(p, pc);
      const CopyJob& jb = p.job[j];
      const uint64_t local = pc - p.piece_start[j];
      if (!co_aligned(jb)) {
        const uint64_t off = local * p.piece_bytes;
        const uint64_t len = jb.bytes - off < p.piece_bytes ? jb.bytes - off : p.piece_bytes;
        copy_bytes_all(p, jb, off, len, lane);
      } else if (local == 0) {
        const uint64_t h = job_head(jb);
        const uint64_t end = h + job_body(jb);
        copy_bytes_all(p, jb, 0, h, lane);
        copy_bytes_all(p, jb, end, jb.bytes - end, lane);
      }
    }
    return;
  }
  if (lane != 0) return;

  // Bulk pipeline: loads run kStages ahead of stores; a piece's stores (one
  // per destination) form one bulk group.
  uint32_t stage_bytes[kStages];
  int stage_job[kStages];
  uint64_t stage_off[kStages];
  uint64_t next = 0;  // next of my pieces to look at for a load
  uint32_t nload = 0, nstore = 0;
  auto issue_next_load = [&]() -> bool {
    while (next < mine) {
      const uint64_t pc = blockIdx.x + next * gridDim.x;
      ++next;
      int j;
      uint64_t o;
      uint32_t n;
      piece_bulk(p, pc, j, o, n);
      if (n == 0) continue;
      const int s = nload % kStages;
      stage_bytes[s] = n;
      stage_job[s] = j;
      stage_off[s] = o;
      mbar_arrive_expect_tx(&bar[s], n + p.tx_pad);
      bulk_load(stage_mem + size_t(s) * p.piece_bytes, p.job[j].src + o, n, &bar[s]);
      ++nload;
      return true;
    }
    return false;
  };
  for (int s = 0; s < kStages; ++s)
    if (!issue_next_load()) break;
  bool failed = false;
  while (nstore < nload) {
    const int s = nstore % kStages;
    if (!mbar_wait_bounded(&bar[s], (nstore / kStages) & 1u, global_ns() + p.wait_ns)) {
      failed = true;
      break;
    }
    const CopyJob& jb = p.job[stage_job[s]];
    const unsigned char* piece = stage_mem + size_t(s) * p.piece_bytes;
    bulk_store(jb.dst + stage_off[s], piece, stage_bytes[s]);
    for (int e = 0; e < jb.nmore; ++e) bulk_store(p.more_dst[jb.more_at + e] + stage_off[s], piece, stage_bytes[s]);
    bulk_commit();
    ++nstore;
    if (nstore >= 2) {
      // once the store before this one has read its stage, refill that stage
      bulk_wait_read_1();
      issue_next_load();
    }
  }
  if (failed) {
    atomicExch(p.status, kStatusTimeoutLoad);
    // Drain: every load still in flight, bounded again.
    const uint64_t deadline = global_ns() + p.wait_ns;
    for (uint32_t b = nstore; b < nload; ++b) {
      if (!mbar_wait_bounded(&bar[b % kStages], (b / kStages) & 1u, deadline)) {
        atomicExch(p.status, kStatusTimeoutDrain);
        break;
      }
    }
  }
  bulk_wait_all();
}

}  // namespace

uint32_t tma_piece_bytes() { return kPieceBytes; }

uint64_t tma_job_pieces(const CopyJob& j, uint32_t piece_bytes) { return job_pieces(j, piece_bytes); }

int tma_ctas_per_sm() { return 1; }

cudaError_t tma_prepare() {
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&tma_copy_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, int(kStages * kPieceBytes));
}

cudaError_t tma_copy_preload() {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, reinterpret_cast<const void*>(&tma_copy_kernel));
}

cudaError_t launch_tma_copy(const CopyParams& p, int grid, cudaStream_t stream) {
  if (grid < 1 || p.njobs < 1) return cudaSuccess;
  if (p.piece_bytes != kPieceBytes) return cudaErrorInvalidValue;
  void* args[] = {const_cast<CopyParams*>(&p)};
  return cudaLaunchKernel(reinterpret_cast<const void*>(&tma_copy_kernel), dim3(grid), dim3(kCopyThreads), args,
                          size_t(kStages) * kPieceBytes, stream);
}

}  // namespace hoc

// ---------------------------------------------------------------------------
// Allocation-free entry point.  The bulk-copy kernel needs one piece of device
// scratch: the status word its bounded waits write on a timeout.  A
// communicator allocates that word with cudaMalloc in hoc_init; callers that
// cannot allocate device memory use this entry point instead, whose status
// words live in the file-scope array below (loaded with the library and held
// by every GPU that loads it until the process exits).
// ---------------------------------------------------------------------------
namespace hoc {
namespace {

constexpr int kNoAllocStatusWords = HOC_NOALLOC_SCRATCH_BYTES / int(sizeof(int));
static __device__ __align__(256) int g_noalloc_status[kNoAllocStatusWords];

constexpr int kMaxDevices = 64;
constexpr uint64_t kMaxMoveBytes = uint64_t(1) << 40;  // the span limit of every other call
std::mutex g_noalloc_mu;
int* g_noalloc_ptr[kMaxDevices] = {};  // device address of g_noalloc_status, per device

// Once per device, with that device current: opt the kernel into its shared
// memory size and resolve the scratch array's device address (in host code
// the symbol itself is only a host-side stand-in).
cudaError_t noalloc_setup(int dev, int** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    cudaError_t e = tma_prepare();
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_status);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace hoc

extern "C" hocResult_t hoc_tma_moves_noalloc(const void* const* src, void* const* dst, const size_t* bytes, int n,
                                             int max_ctas, void* stream, int wait) {
  using namespace hoc;
  if (n > HOC_NOALLOC_MAX_MOVES) {
    set_error_detail("hoc_tma_moves_noalloc: more than HOC_NOALLOC_MAX_MOVES (192) moves in one call");
    return HOC_ERR_INVALID_ARG;
  }
  if (n < 0 || max_ctas < 0) {
    set_error_detail("hoc_tma_moves_noalloc: negative move count or CTA cap");
    return HOC_ERR_INVALID_ARG;
  }
  if (n == 0) return HOC_SUCCESS;
  if (!src || !dst || !bytes) {
    set_error_detail("hoc_tma_moves_noalloc: NULL array");
    return HOC_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HOC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HOC_ERR_CUDA;
  int* status = nullptr;
  if (noalloc_setup(dev, &status) != cudaSuccess) return HOC_ERR_CUDA;
  CopyParams cp;
  memset(&cp, 0, sizeof cp);
  cp.piece_bytes = kPieceBytes;
  // Host-side fault injection (HOC_FAULT=tma_stall), as for the communicator's
  // moves: every mbarrier expects 16 bytes more than its load brings, so the
  // bounded waits give up after 0.1 s and the status word reports it.
  const char* fault = getenv("HOC_FAULT");
  const bool stall = fault && !strcmp(fault, "tma_stall");
  cp.tx_pad = stall ? 16u : 0u;
  cp.wait_ns = stall ? 100000000ull : 2000000000ull;
  cp.status = status;
  int nj = 0;
  for (int i = 0; i < n; ++i) {
    if (bytes[i] == 0) continue;
    if (!src[i] || !dst[i]) {
      set_error_detail("hoc_tma_moves_noalloc: NULL source or destination of a non-empty move");
      return HOC_ERR_INVALID_ARG;
    }
    const uintptr_t a = reinterpret_cast<uintptr_t>(src[i]), d = reinterpret_cast<uintptr_t>(dst[i]);
    const uintptr_t hi = a > d ? a : d;
    if (uint64_t(bytes[i]) > kMaxMoveBytes || bytes[i] > UINTPTR_MAX - hi) {  // no end address below wraps
      set_error_detail("hoc_tma_moves_noalloc: a move of more than 2^40 bytes, or one that runs past the address space");
      return HOC_ERR_INVALID_ARG;
    }
    if (a < d + bytes[i] && d < a + bytes[i]) {  // a move may not overlap itself
      set_error_detail("hoc_tma_moves_noalloc: a move's source and destination overlap");
      return HOC_ERR_INVALID_ARG;
    }
    CopyJob j{};
    j.src = static_cast<const char*>(src[i]);
    j.dst = static_cast<char*>(dst[i]);
    j.bytes = uint64_t(bytes[i]);
    cp.job[nj] = j;
    cp.piece_start[nj + 1] = cp.piece_start[nj] + job_pieces(j, kPieceBytes);
    ++nj;
  }
  cp.njobs = nj;
  if (nj == 0) return HOC_SUCCESS;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status must start at zero.
  if (cudaMemsetAsync(status, 0, sizeof(int) * kNoAllocStatusWords, s) != cudaSuccess) return HOC_ERR_CUDA;
  const int cap = max_ctas > 0 ? (max_ctas < sms ? max_ctas : sms) : sms;
  const uint64_t pieces = cp.piece_start[nj];
  const int grid = int(pieces < uint64_t(cap) ? pieces : uint64_t(cap));
  if (launch_tma_copy(cp, grid, s) != cudaSuccess) return HOC_ERR_CUDA;
  if (!wait) return HOC_SUCCESS;
  int st = 0;
  if (cudaMemcpyAsync(&st, status, sizeof st, cudaMemcpyDeviceToHost, s) != cudaSuccess) return HOC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return HOC_ERR_CUDA;
  return st == 0 ? HOC_SUCCESS : HOC_ERR_TIMEOUT;
}
