// Internal declarations shared by the host runtime and the CUDA kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "hoc.h"

namespace hoc {

constexpr int kMaxRanks = HOC_MAX_RANKS;
constexpr int kMaxCopyJobs = HOC_NOALLOC_MAX_MOVES;  // jobs per TMA copy launch (kernel parameter space)

// ----------------------------------------------------------------- reduce
// One segment = one block's element range of one launch.  Every rank's input
// is read at [elem_off, elem_off + elems); the folded result goes to the
// output buffer(s) at [out_off, out_off + elems).
struct ReduceSeg {
  uint64_t elem_off;
  uint64_t elems;
  uint64_t out_off;
  uint32_t owner;  // block owner: selects the operand order and, without broadcast, the output rank
  uint32_t vec;    // 1 when every input and output pointer of the segment is co-aligned to 16 bytes
};

struct ReduceParams {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  ReduceSeg seg[kMaxRanks];
  uint64_t tile_start[kMaxRanks + 1];  // prefix sums of the tiles of each segment
  uint8_t seq[kMaxRanks][kMaxRanks];   // seq[owner][j] = rank of the j-th operand (ring order)
  int32_t k;
  int32_t nseg;
  int32_t broadcast;  // 1: write the result to out[0..k-1]; 0: to out[owner]
  int32_t dtype;      // hocDataType_t (INT32, FLOAT32, BFLOAT16)
};

// Tiles of a segment (0 for an empty segment) for the whole-GPU shape
// (wide = false) or the one-CTA-per-SM shape used under an SM budget.
uint64_t reduce_seg_tiles(int dtype, const ReduceSeg& s, bool wide);
// Resident CTAs per SM of the whole-GPU reduce kernel for (dtype, k, broadcast).
int reduce_ctas_per_sm(int dtype, int k, int broadcast);
// overlap_launch: programmatic dependent launch (the kernel may be scheduled
// while the grid before it in the stream drains; it waits for that grid's
// completion before touching memory).  Only for multi-wave grids: under an SM
// budget the waiting CTAs would sit on SMs the budget leaves to other work.
cudaError_t launch_reduce(const ReduceParams& p, int grid, bool wide, cudaStream_t stream, bool overlap_launch);

// Force-load every kernel of the library (cudaFuncGetAttributes on each).
// Under lazy module loading the first launch of a kernel loads it, and that
// load can stall work already queued on other streams until the whole
// context drains; the host proxy holds a stream at a flag while its moves run,
// so every kernel that may launch during that window is loaded up front.
cudaError_t reduce_preload();
cudaError_t tma_preload();       // TMA copy kernel and TMA-fed reduce kernel
cudaError_t ep_preload();        // expert-parallel pack and combine kernels
cudaError_t workload_preload();  // probe and stand-in compute kernels

// TMA-fed variant (reduce_tma.cu): same fold, bulk copies through shared memory.
uint64_t reduce_tma_seg_tiles(int dtype, const ReduceSeg& s, int k);
cudaError_t reduce_tma_prepare();  // one-time per device: shared-memory opt-in
// tx_pad: extra bytes every mbarrier expects (0; > 0 only for host-injected
// stalls); wait_ns: the bound of every mbarrier wait.
cudaError_t launch_reduce_tma(const ReduceParams& p, int grid, int* status, cudaStream_t stream, uint32_t tx_pad,
                              uint64_t wait_ns);

// -------------------------------------------------------------- TMA copy
// One copy job of the TMA kernel: `bytes` from `src` to `dst` and, for a
// broadcast, to CopyParams::more_dst[more_at .. more_at + nmore) too (the
// bytes are loaded once and stored to every destination).  Every destination
// is co-aligned with the source modulo 16 bytes, or none is.
struct CopyJob {
  const char* src;
  char* dst;
  uint64_t bytes;
  int32_t nmore;
  int32_t more_at;
};
constexpr int kMaxMoreDst = 256;  // broadcast destinations beyond the first, per launch

struct CopyParams {
  CopyJob job[kMaxCopyJobs];
  uint64_t piece_start[kMaxCopyJobs + 1];  // prefix sums of the pieces of each job
  char* more_dst[kMaxMoreDst];             // further destinations of broadcast jobs
  int32_t njobs;
  uint32_t piece_bytes;  // bytes per piece: one shared-memory stage
  uint32_t tx_pad;       // extra bytes each mbarrier expects (0; >0 only for host-injected stalls)
  uint64_t wait_ns;      // bound of every mbarrier wait
  int* status;           // device word; the kernel writes a non-zero code on a wait timeout
};

uint32_t tma_piece_bytes();
uint64_t tma_job_pieces(const CopyJob& j, uint32_t piece_bytes);
int tma_ctas_per_sm();
cudaError_t tma_prepare();  // one-time per device: shared-memory opt-in
cudaError_t launch_tma_copy(const CopyParams& p, int grid, cudaStream_t stream);
cudaError_t tma_copy_preload();

// Text for hoc_last_error_detail() (defined with the C ABI).
void set_error_detail(const char* what);

// Device status codes written by kernels.
constexpr int kStatusTimeoutLoad = 0x1001;
constexpr int kStatusTimeoutDrain = 0x1002;

}  // namespace hoc
