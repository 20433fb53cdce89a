// Expert-parallel pack and combine around the dispatch / combine all-to-all
// (HOCCL section 2.1 and Table 1: EP token dispatch and combine).
//
// pack   (dispatch side): a stable counting sort of the (token, slot) pairs of
//        one source rank by expert -- experts of a rank are contiguous, so this
//        is the (destination rank, expert, token, slot) order -- followed by a
//        row scatter into the send buffer and the per-destination element counts
//        that the all-to-all needs (on the device, for hoc_alltoall_device_counts).
// combine (unpack): every token's output row is the gate-weighted sum of its
//        topk returned rows, folded in slot order in binary32 (products and sums
//        each rounded to nearest even, no fused multiply-add) and rounded once to
//        bf16.
// Pairs whose expert id lies outside [0, experts) are dropped: they are sent
// nowhere and add nothing to the combine.
//
// Fused with the exchange (hoc_ep_dispatch_fused / hoc_ep_combine_fused): all k
// simulated ranks share one HBM, so the dispatch's row scatter writes each
// token row straight to its place in the destination rank's receive buffer
// -- the place the all-to-all would have copied it to -- and the combine
// reads each of a token's rows straight from the expert rank's buffer.  The
// places follow from the k x k counts on the device: row i of source s's
// packed order, bound for rank d, lands at row rdispl[d][s] + i - sdispl[s][d]
// of rank d's buffer, with rdispl[d][s] = sum of counts[s'][d] over s' < s and
// sdispl[s][d] = sum of counts[s][d'] over d' < d (prefix sums in rank order,
// the all-to-all's default displacements).
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cuda_bf16.h>

#include "hoc_internal.h"
#include "hoc_ep.h"
#include "f32x2.cuh"
#include "ptx_async.cuh"

namespace hoc {
namespace {

constexpr int kEpThreads = 256;
constexpr int kEpWarps = kEpThreads / 32;
// Counting sort by tiles: each CTA owns kTileItems consecutive pairs, each of
// its warps a contiguous kWarpItems of them, so (tile, warp, step, lane) order
// is pair order and the sort stays stable.
constexpr int kTileItems = 2048;
constexpr int kWarpItems = kTileItems / kEpWarps;
constexpr int kMaxTileExperts = 1024;  // per-warp counters of this many experts fit in shared memory
constexpr int kCombineTopk = 8;        // combine: top-k loads issued together up to this k

// Programmatic dependent launch (no-ops for a plain launch): wait until the
// kernel before this one in the stream has completed and its writes are
// visible, then let the next kernel launch.  The pack and combine are chains
// of short kernels, so this hides each launch behind its predecessor's tail.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per-source pointers of the sort kernels; blockIdx.y selects the source, so
// one launch sorts the pairs of every source rank (a single source: y = 0).
struct EpSort {
  const int32_t* ids[kMaxRanks];
  int32_t* perm[kMaxRanks];    // null: not wanted (the fused dispatch needs only pos_of)
  int32_t* pos_of[kMaxRanks];
  unsigned long long* counts;  // [sources][nranks] element counts, row = source
  int32_t* ws;                 // scratch of source s at ws + s * ws_stride
  size_t ws_stride;
};

// One CTA per expert: how many pairs chose it.
__global__ void ep_count_kernel(const __grid_constant__ EpSort P, int n) {
  pdl_enter();
  const int32_t* __restrict__ ids = P.ids[blockIdx.y];
  int32_t* __restrict__ cnt = P.ws + blockIdx.y * P.ws_stride;
  const int e = blockIdx.x;
  int total = 0;
  for (int base = 0; base < n; base += kEpThreads) {
    const int i = base + threadIdx.x;
    total += __syncthreads_count(i < n && ids[i] == e);
  }
  if (threadIdx.x == 0) cnt[e] = total;
}

// One CTA per expert: place its pairs, in (token, slot) order, after the pairs
// of all smaller experts.
__global__ void ep_place_kernel(const __grid_constant__ EpSort P, int n, int hidden, int per_rank, int nranks) {
  pdl_enter();
  const int32_t* __restrict__ ids = P.ids[blockIdx.y];
  const int32_t* __restrict__ cnt = P.ws + blockIdx.y * P.ws_stride;
  int32_t* __restrict__ perm = P.perm[blockIdx.y];
  int32_t* __restrict__ pos_of = P.pos_of[blockIdx.y];
  unsigned long long* __restrict__ dst_counts = P.counts + size_t(blockIdx.y) * nranks;
  __shared__ int warp_n[kEpThreads / 32];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int offset = 0;
  for (int j = 0; j < e; ++j) offset += cnt[j];
  int running = 0;
  for (int base = 0; base < n; base += kEpThreads) {
    const int i = base + threadIdx.x;
    const bool mine = i < n && ids[i] == e;
    const unsigned ballot = __ballot_sync(0xFFFFFFFFu, mine);
    if (lane == 0) warp_n[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, chunk = 0;
    for (int w = 0; w < kEpThreads / 32; ++w) {
      if (w < warp) before += warp_n[w];
      chunk += warp_n[w];
    }
    if (mine) {
      const int pos = offset + running + before + __popc(ballot & ((1u << lane) - 1u));
      if (perm) perm[pos] = i;
      pos_of[i] = pos;
    }
    running += chunk;
    __syncthreads();
  }
  if (threadIdx.x == 0 && cnt[e] > 0) atomicAdd(dst_counts + e / per_rank, (unsigned long long)cnt[e] * hidden);
}

// Tile histogram: hist[b * experts + e] = pairs of tile b that chose expert e.
// A thread issues all of its loads of the tile before counting them.
__global__ void ep_tile_hist_kernel(const __grid_constant__ EpSort P, int n, int experts) {
  pdl_enter();
  const int32_t* __restrict__ ids = P.ids[blockIdx.y];
  int32_t* __restrict__ hist = P.ws + blockIdx.y * P.ws_stride + experts;
  extern __shared__ int sh[];
  for (int e = threadIdx.x; e < experts; e += blockDim.x) sh[e] = 0;
  const int lo = blockIdx.x * kTileItems;
  int ev[kTileItems / kEpThreads];
#pragma unroll
  for (int k = 0; k < kTileItems / kEpThreads; ++k) {
    const int i = lo + k * kEpThreads + int(threadIdx.x);
    ev[k] = i < n ? ids[i] : -1;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kTileItems / kEpThreads; ++k)
    if (ev[k] >= 0 && ev[k] < experts) atomicAdd(&sh[ev[k]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < experts; e += blockDim.x) hist[size_t(blockIdx.x) * experts + e] = sh[e];
}

// One CTA per source: turns the tile histograms into the first output row of
// each (tile, expert) -- all pairs of smaller experts, then those of expert e
// in earlier tiles -- and writes the per-expert totals, the number of valid
// pairs and the per-destination element counts.  With `staged` the histograms and
// totals are copied into shared memory once (coalesced), every scan runs on
// that copy, and the starts go back once; otherwise the scans run in place in
// global memory (shapes whose histograms exceed the shared budget).
constexpr int kScanThreads = 1024;
// Up to this many (tile, expert) histogram cells per source, each placement
// CTA derives its own starts from the raw histograms instead of a separate scan
// launch (at the EP workload: 12 tiles x 64 experts).
constexpr int kPlaceScanCells = 8192;
constexpr int kScanSmemInts = 48 * 1024 / 4 - kScanThreads;  // dynamic ints beside the static warp sums

__global__ void ep_scan_kernel(const __grid_constant__ EpSort P, int tiles, int experts, int nranks, int per_rank,
                               int hidden, int staged) {
  pdl_enter();
  int32_t* __restrict__ total = P.ws + blockIdx.x * P.ws_stride;
  int32_t* __restrict__ hist = total + experts;
  int32_t* __restrict__ nvalid = hist + size_t(tiles) * experts;
  unsigned long long* __restrict__ dst_counts = P.counts + size_t(blockIdx.x) * nranks;
  __shared__ int warp_sum[kScanThreads / 32];
  extern __shared__ int dyn[];  // staged: [experts] totals, then [tiles][experts] histograms
  const size_t cells = size_t(tiles) * experts;
  int* tot = staged ? dyn : total;
  int* h = staged ? dyn + experts : hist;
  if (staged) {
    for (size_t j = threadIdx.x; j < cells; j += blockDim.x) h[j] = hist[j];
    __syncthreads();
  }
  for (int e = threadIdx.x; e < experts; e += blockDim.x) {  // per expert: exclusive scan over tiles
    int run = 0;
    for (int b = 0; b < tiles; ++b) {
      const int c = h[size_t(b) * experts + e];
      h[size_t(b) * experts + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
  // exclusive scan of the totals over experts: thread t owns a contiguous run
  // of experts; a shuffle scan within each warp, then over the warp sums
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int per = (experts + blockDim.x - 1) / blockDim.x;
  const int e0 = min(experts, int(threadIdx.x) * per), e1 = min(experts, e0 + per);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += tot[e];
  int incl = mine;
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < nwarps ? warp_sum[lane] : 0;
    int wi = ws;
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += v;
    }
    if (lane < nwarps) warp_sum[lane] = wi - ws;  // exclusive over warps
    if (lane == nwarps - 1) *nvalid = wi;         // every valid pair
  }
  __syncthreads();
  int base = warp_sum[warp] + incl - mine;
  for (int e = e0; e < e1; ++e) {
    for (int b = 0; b < tiles; ++b) h[size_t(b) * experts + e] += base;
    base += tot[e];
  }
  for (int d = threadIdx.x; d < nranks; d += blockDim.x) {
    unsigned long long c = 0;
    for (int e = d * per_rank; e < (d + 1) * per_rank; ++e) c += (unsigned long long)tot[e];
    dst_counts[d] = c * (unsigned long long)hidden;
  }
  if (staged) {
    __syncthreads();
    for (size_t j = threadIdx.x; j < cells; j += blockDim.x) hist[j] = h[j];
    for (int e = threadIdx.x; e < experts; e += blockDim.x) total[e] = tot[e];
  }
}

// Exclusive prefix sum of v[0, n) in place by the whole CTA (blockDim.x a
// multiple of 32, at most 1024); returns the sum of all n to every thread.
// sh: shared scratch of blockDim.x / 32 + 1 ints.
__device__ int block_exclusive_scan(int* v, int n, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int e0 = min(n, int(threadIdx.x) * per), e1 = min(n, e0 + per);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += v[e];
  int incl = mine;
  for (int off = 1; off < 32; off <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += x;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < nwarps ? sh[lane] : 0;
    int wi = ws;
    for (int off = 1; off < 32; off <<= 1) {
      const int x = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += x;
    }
    if (lane < nwarps) sh[lane] = wi - ws;  // exclusive over warps
    if (lane == 31) sh[nwarps] = wi;        // everything
  }
  __syncthreads();
  int run = sh[warp] + incl - mine;
  for (int e = e0; e < e1; ++e) {
    const int c = v[e];
    v[e] = run;
    run += c;
  }
  const int all = sh[nwarps];
  __syncthreads();
  return all;
}

// Stable placement of one tile: a pair's row is its (tile, expert) start, plus
// the pairs of that expert in earlier warps of the tile, earlier steps of its
// warp and lower lanes of its step.  A warp loads all of its expert ids, and
// later all of their starts, before the dependent counting.
constexpr int kWarpSteps = kWarpItems / 32;
__global__ void ep_tile_place_kernel(const __grid_constant__ EpSort P, int n, int experts, int tiles, int scan_here,
                                     int nranks, int per_rank, int hidden) {
  pdl_enter();
  const int32_t* __restrict__ ids = P.ids[blockIdx.y];
  const int32_t* __restrict__ start = P.ws + blockIdx.y * P.ws_stride + experts;
  const int32_t* __restrict__ nvalid = start + size_t(tiles) * experts;
  int32_t* __restrict__ perm = P.perm[blockIdx.y];
  int32_t* __restrict__ pos_of = P.pos_of[blockIdx.y];
  extern __shared__ int wh[];  // [kEpWarps][experts]; with scan_here then [experts] starts, [experts] totals
  __shared__ int scan_sh[kEpWarps + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j = threadIdx.x; j < kEpWarps * experts; j += blockDim.x) wh[j] = 0;
  int valid_pairs = 0;
  const int32_t* st = start + size_t(blockIdx.x) * experts;
  if (scan_here) {  // this tile's starts from the raw tile histograms (`start` holds them)
    int* my_start = wh + kEpWarps * experts;
    int* tot = my_start + experts;
    for (int e = threadIdx.x; e < experts; e += blockDim.x) {
      int before = 0, all = 0;
      for (int b = 0; b < tiles; ++b) {
        const int c = start[size_t(b) * experts + e];
        before += b < int(blockIdx.x) ? c : 0;
        all += c;
      }
      my_start[e] = before;
      tot[e] = all;
    }
    __syncthreads();
    if (blockIdx.x == 0)  // one CTA per source writes its destination counts
      for (int d = threadIdx.x; d < nranks; d += blockDim.x) {
        unsigned long long c = 0;
        for (int e = d * per_rank; e < (d + 1) * per_rank; ++e) c += (unsigned long long)tot[e];
        P.counts[size_t(blockIdx.y) * nranks + d] = c * (unsigned long long)hidden;
      }
    valid_pairs = block_exclusive_scan(tot, experts, scan_sh);  // tot[e]: pairs of smaller experts
    for (int e = threadIdx.x; e < experts; e += blockDim.x) my_start[e] += tot[e];
    __syncthreads();
    st = my_start;
  } else {
    valid_pairs = *nvalid;
  }
  int* mine = wh + warp * experts;
  const int lo = blockIdx.x * kTileItems + warp * kWarpItems;
  const int hi = min(n, lo + kWarpItems);
  const unsigned below = (1u << lane) - 1u;
  int ev[kWarpSteps];
#pragma unroll
  for (int k = 0; k < kWarpSteps; ++k) {
    const int i = lo + k * 32 + lane;
    const int e = i < hi ? ids[i] : -1;
    ev[k] = e >= 0 && e < experts ? e : -1;  // -1: dropped pair or past the tile
  }
  __syncthreads();
  unsigned grp[kWarpSteps];
#pragma unroll
  for (int k = 0; k < kWarpSteps; ++k) {  // this warp's pairs per expert
    grp[k] = __match_any_sync(0xFFFFFFFFu, ev[k]);
    if (ev[k] >= 0 && (grp[k] & below) == 0) mine[ev[k]] += __popc(grp[k]);  // the group's lowest lane counts it
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < experts; e += blockDim.x) {  // per expert: exclusive scan over warps
    int run = 0;
    for (int w = 0; w < kEpWarps; ++w) {
      const int c = wh[w * experts + e];
      wh[w * experts + e] = run;
      run += c;
    }
  }
  __syncthreads();
  int sv[kWarpSteps];
#pragma unroll
  for (int k = 0; k < kWarpSteps; ++k) sv[k] = ev[k] >= 0 ? st[ev[k]] : 0;
#pragma unroll
  for (int k = 0; k < kWarpSteps; ++k) {
    const int i = lo + k * 32 + lane;
    if (ev[k] >= 0) {
      const int pos = sv[k] + mine[ev[k]] + __popc(grp[k] & below);
      if (perm) perm[pos] = i;
      pos_of[i] = pos;
    } else if (i < hi) {
      pos_of[i] = -1;  // dropped pair
    }
    __syncwarp();
    if (ev[k] >= 0 && (grp[k] & below) == 0) mine[ev[k]] += __popc(grp[k]);
    __syncwarp();
  }
  // rows past the valid pairs have no pair
  if (perm)
    for (int r = valid_pairs + blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) perm[r] = -1;
}

// send[pos_of[t*topk + j]] = x[t] for every valid pair (t, j); rows of `hb`
// bytes.  Each token row is read once and stored to each of its packed rows.
// Vector path: a work item is (token, 1 KiB slice of its row), one per warp
// of the grid; a lane loads two 16-byte vectors of the slice and stores them
// to every destination row.  Byte path: warp per token.
constexpr int kScatterSliceVecs = 64;  // 16-byte vectors per work item
__global__ void ep_scatter_kernel(const char* __restrict__ x, const int32_t* __restrict__ pos_of, int tokens,
                                  int topk, int hb, char* __restrict__ send, int vec) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long first = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (vec) {
    const int nv = hb / 16;
    const int slices = (nv + kScatterSliceVecs - 1) / kScatterSliceVecs;
    const long long items = (long long)tokens * slices;
    for (long long it = first; it < items; it += warps) {
      const int t = int(it / slices);
      const int v0 = int(it % slices) * kScatterSliceVecs + lane;
      const int v1 = v0 + 32;  // still inside the slice
      const bool h0 = v0 < nv, h1 = v1 < nv;
      const uint4* s4 = reinterpret_cast<const uint4*>(x + size_t(t) * hb);
      uint4 a, b;
      if (h0) a = __ldg(s4 + v0);
      if (h1) b = __ldg(s4 + v1);
      for (int j0 = 0; j0 < topk; j0 += 32) {
        const int pl = j0 + lane < topk ? pos_of[size_t(t) * topk + j0 + lane] : -1;
        const int nj = min(32, topk - j0);
        for (int j = 0; j < nj; ++j) {
          const int pos = __shfl_sync(0xFFFFFFFFu, pl, j);
          if (pos < 0) continue;  // dropped pair: nothing to send
          uint4* d4 = reinterpret_cast<uint4*>(send + size_t(pos) * hb);
          if (h0) d4[v0] = a;
          if (h1) d4[v1] = b;
        }
      }
    }
    return;
  }
  for (long long t = first; t < tokens; t += warps) {
    const char* src = x + size_t(t) * hb;
    for (int j = 0; j < topk; ++j) {
      const int pos = pos_of[size_t(t) * topk + j];
      if (pos < 0) continue;
      char* d = send + size_t(pos) * hb;
      for (int b = lane; b < hb; b += 32) d[b] = src[b];
    }
  }
}

// Warp per token: y[t] = bf16(sum_j fp32(w[t,j] * row[pos_of[t*topk + j]])).
__global__ void ep_combine_kernel(const uint16_t* __restrict__ rows, const int32_t* __restrict__ pos_of,
                                  const float* __restrict__ w, int tokens, int topk, int hidden, int n_rows,
                                  uint16_t* __restrict__ y) {
  pdl_enter();
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < tokens; t += gridDim.x * warps) {
    for (int h = lane; h < hidden; h += 32) {
      float acc = 0.f;
      bool any = false;
      for (int j = 0; j < topk; ++j) {
        const int p = pos_of[size_t(t) * topk + j];
        if (p < 0 || p >= n_rows) continue;
        const float r = __uint_as_float(uint32_t(rows[size_t(p) * hidden + h]) << 16);
        const float prod = __fmul_rn(w[size_t(t) * topk + j], r);
        acc = any ? __fadd_rn(acc, prod) : prod;
        any = true;
      }
      y[size_t(t) * hidden + h] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
  }
}

// Same fold, 8 bf16 per lane per step (16-byte loads and stores); needs
// hidden % 8 == 0 and 16-byte-aligned rows and outputs.
__global__ void ep_combine_vec_kernel(const uint16_t* __restrict__ rows, const int32_t* __restrict__ pos_of,
                                      const float* __restrict__ w, int tokens, int topk, int hidden, int n_rows,
                                      uint16_t* __restrict__ y) {
  pdl_enter();
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hv = hidden / 8;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < tokens; t += gridDim.x * warps) {
    for (int v = lane; v < hv; v += 32) {
      float acc[8];
      bool any = false;
      for (int j = 0; j < topk; ++j) {
        const int p = pos_of[size_t(t) * topk + j];
        if (p < 0 || p >= n_rows) continue;
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(rows + size_t(p) * hidden) + v);
        const float wj = w[size_t(t) * topk + j];
        const uint32_t q[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __fmul_rn(wj, __uint_as_float(q[i] << 16));
          const float hi = __fmul_rn(wj, __uint_as_float(q[i] & 0xFFFF0000u));
          acc[2 * i] = any ? __fadd_rn(acc[2 * i], lo) : lo;
          acc[2 * i + 1] = any ? __fadd_rn(acc[2 * i + 1], hi) : hi;
        }
        any = true;
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = any ? acc[2 * i] : 0.f, b = any ? acc[2 * i + 1] : 0.f;
        o[i] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
      }
      reinterpret_cast<uint4*>(y + size_t(t) * hidden)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Same fold with every one of the token's TK row loads issued before the
// ordered fold, so a lane keeps TK 16-byte loads in flight (TK = topk).
// acc + w * x for the two bf16 values packed in q: each product rounded to
// binary32 on its own, then both sums in one instruction.  The products stay
// scalar on purpose (f32x2.cuh): with a packed multiply the code generator
// fused it into the add -- about a quarter of random operands then differed,
// although both instructions name their rounding, and an empty statement
// between them did not stop it -- while a scalar product with its rounding
// named is never fused.
__device__ __forceinline__ unsigned long long mul_add_bf16x2(unsigned long long acc, float w, uint32_t q) {
  return add_f32x2(acc, pack_f32x2(__fmul_rn(w, __uint_as_float(q << 16)), __fmul_rn(w, __uint_as_float(q & 0xFFFF0000u))));
}

template <int TK>
__global__ void ep_combine_vec_ilp_kernel(const uint16_t* __restrict__ rows, const int32_t* __restrict__ pos_of,
                                          const float* __restrict__ w, int tokens, int hidden, int n_rows,
                                          uint16_t* __restrict__ y) {
  pdl_enter();
  // Work item = (token, slice of 32 16-byte vectors of its row): many small
  // items spread evenly over the warps, so no partial last wave of whole rows.
  // A warp walks its items as (token, slice), moved on by the grid's warps at
  // a time in that mixed radix (no division per item).
  const int lane = threadIdx.x & 31;
  const int hv = hidden / 8;
  const uint32_t slices = uint32_t(hv + 31) / 32;
  const long long items = (long long)tokens * slices;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long first = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  long long t = first / slices;
  uint32_t sl = uint32_t(first - t * slices);
  const long long dt = warps / slices;
  const uint32_t dsl = uint32_t(warps - dt * slices);
  for (long long it = first; it < items; it += warps) {
    const int v = int(sl) * 32 + lane;
    const int pl = lane < TK ? pos_of[size_t(t) * TK + lane] : -1;
    const float wl = lane < TK ? w[size_t(t) * TK + lane] : 0.f;
    int p[TK];
    float wj[TK];
    bool ok[TK];
#pragma unroll
    for (int j = 0; j < TK; ++j) {
      p[j] = __shfl_sync(0xFFFFFFFFu, pl, j);
      wj[j] = __shfl_sync(0xFFFFFFFFu, wl, j);
      ok[j] = p[j] >= 0 && p[j] < n_rows && v < hv;
    }
    const long long tt = t;
    sl += dsl;  // the warp's next item
    t += dt + (sl >= slices);
    if (sl >= slices) sl -= slices;
    if (v >= hv) continue;
    uint4 x[TK];
#pragma unroll
    for (int j = 0; j < TK; ++j)
      x[j] = ok[j] ? __ldg(reinterpret_cast<const uint4*>(rows + size_t(p[j]) * hidden) + v) : make_uint4(0, 0, 0, 0);
    unsigned long long acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = 0x8000000080000000ull;  // -0 in both lanes: x + -0 = x
    bool any = false;
#pragma unroll
    for (int j = 0; j < TK; ++j) {
      if (!ok[j]) continue;
      const uint32_t q[4] = {x[j].x, x[j].y, x[j].z, x[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = mul_add_bf16x2(acc[i], wj[j], q[i]);
      any = true;
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = any ? __uint_as_float(uint32_t(acc[i])) : 0.f;
      const float b = any ? __uint_as_float(uint32_t(acc[i] >> 32)) : 0.f;
      o[i] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
             (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
    }
    reinterpret_cast<uint4*>(y + size_t(tt) * hidden)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------------------
// Fused with the exchange (and, in packed mode, the all-rank pack / combine
// around a copy-engine exchange).  Per-source inputs and per-rank buffers of
// one dispatch / combine over all k simulated ranks.
struct EpRoute {
  const char* x[kMaxRanks];         // dispatch: token rows of each source, [tokens, hidden] bf16
  const int32_t* ids[kMaxRanks];    // expert id of every (token, slot) pair of each source
  const int32_t* pos_of[kMaxRanks]; // packed row of every pair (-1: dropped)
  const float* w[kMaxRanks];        // combine: gate weights of every pair
  char* buf[kMaxRanks];             // row buffer of each rank: receive buffers, or (packed) each source's own
  char* y[kMaxRanks];               // combine: output rows of each source
  unsigned long long cap_rows[kMaxRanks];  // rows each buffer holds
  const unsigned long long* counts;        // [k][k] element counts, row = source (unused when packed)
  int32_t* status;  // bit 0: a dispatched row did not fit; bit 1: a combine row out of range;
                    // bit 2: a bounded wait of a bulk-copy kernel gave up
  int k, tokens, topk, hidden, per_rank;
  int packed;  // 1: each source's own buffer buf[s], rows in its packed order (no exchange to fuse)
  // bulk-copy kernels: the limit of each mbarrier wait, and bytes every
  // mbarrier expects beyond its loads (0; 16 under HOC_FAULT=ep_stall, so no
  // wait completes and the timeout path runs with no fault on the GPU)
  unsigned long long wait_ns;
  uint32_t tx_pad;
};

// base[s * k + d] = rdispl[d][s] - sdispl[s][d] in rows: packed row i of source
// s bound for rank d goes to row base[s * k + d] + i of rank d's buffer.
__device__ __forceinline__ void route_bases(const EpRoute& R, long long* base) {
  for (int c = threadIdx.x; !R.packed && c < R.k * R.k; c += blockDim.x) {
    const int s = c / R.k, d = c % R.k;
    unsigned long long rd = 0, sd = 0;
    for (int a = 0; a < s; ++a) rd += R.counts[a * R.k + d];
    for (int b = 0; b < d; ++b) sd += R.counts[s * R.k + b];
    base[c] = (long long)(rd / (unsigned long long)R.hidden) - (long long)(sd / (unsigned long long)R.hidden);
  }
  __syncthreads();
}

// Expert of pair `pr` of source s (routing only: packed mode reads no ids).
__device__ __forceinline__ int pair_expert(const EpRoute& R, int s, size_t pr) { return R.packed ? 0 : R.ids[s][pr]; }

// Where packed row `pos` of source s, a pair with expert e, lives: buffer *b
// (the destination rank e / per_rank, or s itself in packed mode) and the row
// returned; -1 (and the status bit `bit`) when it lies outside that buffer or
// e names no rank (inputs that disagree with the dispatch that made them).
__device__ __forceinline__ long long route_row(const EpRoute& R, const long long* base, int s, int e, int pos,
                                               int bit, int* b) {
  const int d = R.packed ? s : e / R.per_rank;
  *b = d;
  if (unsigned(d) >= unsigned(R.k)) {
    atomicOr(R.status, bit);
    return -1;
  }
  const long long row = R.packed ? (long long)pos : base[s * R.k + d] + pos;
  if (row < 0 || (unsigned long long)row >= R.cap_rows[d]) {
    atomicOr(R.status, bit);
    return -1;
  }
  return row;
}

// Dispatch: every token row of every source, read once, stored to each of its
// valid pairs' rows in the destination ranks' buffers.  Vector path: a work
// item is (source, token, 2 KiB chunk of the row); a lane loads its
// kDispVecs 16-byte vectors of the chunk up front, resolves the pairs'
// destinations once, and stores the vectors to each.  Byte path: a warp per
// (source, token).
constexpr int kDispVecs = 4;                      // 16-byte vectors per lane per item
constexpr int kDispChunk = 32 * kDispVecs * 16;   // bytes of a row per item
__global__ void ep_dispatch_fused_kernel(const __grid_constant__ EpRoute R, int vec) {
  pdl_enter();
  __shared__ long long base[kMaxRanks * kMaxRanks];
  route_bases(R, base);
  const int lane = threadIdx.x & 31;
  const int hb = R.hidden * 2;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long first = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nv = hb / 16;
  const int chunks = vec ? (hb + kDispChunk - 1) / kDispChunk : 1;
  const long long rows = (long long)R.tokens * R.k;
  const long long items = rows * chunks;
  for (long long it = first; it < items; it += warps) {
    const long long row_it = it / chunks;
    const int c = int(it - row_it * chunks);
    const int s = int(row_it / R.tokens), t = int(row_it - (long long)s * R.tokens);
    const char* src = R.x[s] + size_t(t) * hb;
    uint4 a[kDispVecs];
    const int v0 = c * (kDispChunk / 16) + lane;
    if (vec) {
#pragma unroll
      for (int q = 0; q < kDispVecs; ++q)
        if (v0 + 32 * q < nv) a[q] = __ldg(reinterpret_cast<const uint4*>(src) + v0 + 32 * q);
    }
    for (int j0 = 0; j0 < R.topk; j0 += 32) {
      const size_t pr = size_t(t) * R.topk + j0 + lane;
      const bool in = j0 + lane < R.topk;
      const int pl = in ? R.pos_of[s][pr] : -1;
      const int el = in ? pair_expert(R, s, pr) : 0;
      // each lane resolves its own pair's destination row once
      long long myrow = -1;
      int md = 0;
      if (pl >= 0) myrow = route_row(R, base, s, el, pl, 1, &md);
      const int nj = min(32, R.topk - j0);
      for (int j = 0; j < nj; ++j) {
        const long long row = __shfl_sync(0xFFFFFFFFu, myrow, j);
        const int d = __shfl_sync(0xFFFFFFFFu, md, j);
        if (row < 0) continue;  // dropped pair, or no room: sent nowhere
        char* dst = R.buf[d] + size_t(row) * hb;
        if (vec) {
#pragma unroll
          for (int q = 0; q < kDispVecs; ++q)
            if (v0 + 32 * q < nv) reinterpret_cast<uint4*>(dst)[v0 + 32 * q] = a[q];
        } else {
          for (int i = lane; i < hb; i += 32) dst[i] = src[i];
        }
      }
    }
  }
}

// Dispatch through the tensor-memory accelerator: a CTA of one warp streams
// its share of the (source, token, piece) work items; lane 0 bulk-loads each
// piece (a row, or a part of a long row) into a shared-memory stage, waits for
// it on the stage's mbarrier and issues one bulk store per valid pair to the
// destination row, the stores of one piece forming one bulk group; a stage is
// refilled once the stores before the last have read it, so loads run up to
// kBulkStages pieces ahead.  Every 32 items the warp resolves the next 32
// items' destinations together (one lane per item).  Needs rows and buffers
// aligned to 16 bytes and topk <= kBulkMaxTopk.  Every mbarrier wait is
// bounded; on a timeout the kernel sets status bit 2, waits (bounded) for its
// own loads and returns.
constexpr int kBulkStages = 16;
constexpr int kBulkBatch = 32;
constexpr int kBulkMaxTopk = 16;
constexpr uint32_t kBulkPiece = 4096;  // bytes per stage
constexpr uint64_t kBulkWaitNs = 2000000000ull;

__global__ void __launch_bounds__(32) ep_dispatch_bulk_kernel(const __grid_constant__ EpRoute R) {
  using namespace ptx;
  pdl_enter();
  extern __shared__ __align__(128) unsigned char stage_mem[];  // kBulkStages x kBulkPiece
  __shared__ __align__(8) uint64_t bar[kBulkStages];
  __shared__ long long base[kMaxRanks * kMaxRanks];
  __shared__ char* dst_tab[kBulkBatch][kBulkMaxTopk];
  __shared__ uint32_t len_tab[kBulkBatch];
  const int lane = threadIdx.x;
  route_bases(R, base);
  if (lane == 0) {
    for (int st = 0; st < kBulkStages; ++st) mbar_init(&bar[st], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();
  const uint32_t hb = uint32_t(R.hidden) * 2;
  const uint32_t pieces = (hb + kBulkPiece - 1) / kBulkPiece;
  const uint64_t items = uint64_t(R.k) * uint64_t(R.tokens) * pieces;
  const uint64_t mine = items > blockIdx.x ? (items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  // item i of this CTA: global item blockIdx.x + i * gridDim.x = (row, piece), row = s * tokens + t
  auto locate = [&](uint64_t i, int& s, int& t, uint32_t& off, uint32_t& n) {
    const uint64_t g = blockIdx.x + i * gridDim.x;
    const uint64_t row = g / pieces;
    off = uint32_t(g - row * pieces) * kBulkPiece;
    n = hb - off < kBulkPiece ? hb - off : kBulkPiece;
    s = int(row / uint64_t(R.tokens));
    t = int(row - uint64_t(s) * uint64_t(R.tokens));
  };
  uint64_t nload = 0, nstore = 0;
  auto issue_load = [&]() {
    int s, t;
    uint32_t off, n;
    locate(nload, s, t, off, n);
    uint64_t* b = &bar[nload % kBulkStages];
    mbar_arrive_expect_tx(b, n + R.tx_pad);
    bulk_load(stage_mem + size_t(nload % kBulkStages) * kBulkPiece, R.x[s] + size_t(t) * hb + off, n, b);
    ++nload;
  };
  if (lane == 0)
    while (nload < mine && nload < uint64_t(kBulkStages)) issue_load();
  bool failed = false;
  for (uint64_t b0 = 0; b0 < mine && !failed; b0 += kBulkBatch) {
    const uint64_t i = b0 + lane;
    if (i < mine) {  // this lane's item: the destination of each of its pairs
      int s, t;
      uint32_t off, n;
      locate(i, s, t, off, n);
      len_tab[lane] = n;
      for (int j = 0; j < R.topk; ++j) {
        const size_t pr = size_t(t) * R.topk + j;
        const int p = R.pos_of[s][pr];
        char* d = nullptr;
        if (p >= 0) {
          int rk;
          const long long row = route_row(R, base, s, pair_expert(R, s, pr), p, 1, &rk);
          if (row >= 0) d = R.buf[rk] + size_t(row) * hb + off;
        }
        dst_tab[lane][j] = d;
      }
    }
    __syncwarp();
    if (lane == 0) {
      const uint64_t b1 = mine < b0 + kBulkBatch ? mine : b0 + kBulkBatch;
      for (uint64_t it = b0; it < b1; ++it) {
        const int st = int(it % kBulkStages);
        if (!mbar_wait_bounded(&bar[st], uint32_t(it / kBulkStages) & 1u, global_ns() + R.wait_ns)) {
          failed = true;
          break;
        }
        const unsigned char* piece = stage_mem + size_t(st) * kBulkPiece;
        const int slot = int(it - b0);
        for (int j = 0; j < R.topk; ++j)
          if (dst_tab[slot][j]) bulk_store(dst_tab[slot][j], piece, len_tab[slot]);
        bulk_commit();
        ++nstore;
        if (nstore >= 2) {  // the stage of the item before the last is read: refill it
          bulk_wait_read_1();
          if (nload < mine) issue_load();
        }
      }
    }
    failed = __shfl_sync(0xFFFFFFFFu, failed, 0);
    __syncwarp();
  }
  if (lane == 0) {
    if (failed) {
      atomicOr(R.status, 4);
      const uint64_t deadline = global_ns() + R.wait_ns;
      for (uint64_t b = nstore; b < nload; ++b)
        if (!mbar_wait_bounded(&bar[b % kBulkStages], uint32_t(b / kBulkStages) & 1u, deadline)) break;
    }
    bulk_wait_all();
  }
}

// Combine, reading every row straight from the expert rank's buffer; the same
// fold as the packed-order combine.  A work item is (source, token, 1 KiB
// chunk of the row): the token's pairs are resolved once (lanes < topk load
// their pair, then broadcast source row and weight), and a lane folds two
// 16-byte vectors per row.  TK > 0: all TK x 2 row loads of a lane are issued
// before the ordered fold; TK == 0: any topk, one row at a time.
constexpr int kCombVecs = 2;                      // 16-byte vectors per lane per item
constexpr int kCombChunk = 32 * kCombVecs;        // vectors of a row per item

__device__ __forceinline__ void fold_bf16x8(float* acc, const uint4& x, float w, bool first) {
  const uint32_t q[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __fmul_rn(w, __uint_as_float(q[i] << 16));
    const float hi = __fmul_rn(w, __uint_as_float(q[i] & 0xFFFF0000u));
    acc[2 * i] = first ? lo : __fadd_rn(acc[2 * i], lo);
    acc[2 * i + 1] = first ? hi : __fadd_rn(acc[2 * i + 1], hi);
  }
}

__device__ __forceinline__ uint4 narrow_bf16x8(const float* acc, bool any) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = any ? acc[2 * i] : 0.f, hi = any ? acc[2 * i + 1] : 0.f;
    o[i] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int TK>
__global__ void ep_combine_fused_vec_kernel(const __grid_constant__ EpRoute R) {
  pdl_enter();
  __shared__ long long base[kMaxRanks * kMaxRanks];
  route_bases(R, base);
  const int lane = threadIdx.x & 31;
  const int hv = R.hidden / 8;
  const int chunks = (hv + kCombChunk - 1) / kCombChunk;
  const long long rows = (long long)R.tokens * R.k;
  const long long items = rows * chunks;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const long long row_it = it / chunks;
    const int c = int(it - row_it * chunks);
    const int s = int(row_it / R.tokens), t = int(row_it - (long long)s * R.tokens);
    const int v0 = c * kCombChunk + lane;
    float acc[kCombVecs][8];
    bool any = false;
    if constexpr (TK > 0) {
      // lane j < TK resolves pair j: its source row (or none) and weight
      const size_t pr = size_t(t) * TK + lane;
      const char* mine = nullptr;
      float wl = 0.f;
      if (lane < TK) {
        const int p = R.pos_of[s][pr];
        wl = R.w[s][pr];
        if (p >= 0) {
          int d;
          const long long row = route_row(R, base, s, pair_expert(R, s, pr), p, 2, &d);
          if (row >= 0) mine = R.buf[d] + size_t(row) * R.hidden * 2;
        }
      }
      const char* src[TK];
      float wj[TK];
#pragma unroll
      for (int j = 0; j < TK; ++j) {
        src[j] = reinterpret_cast<const char*>(__shfl_sync(0xFFFFFFFFu, reinterpret_cast<uintptr_t>(mine), j));
        wj[j] = __shfl_sync(0xFFFFFFFFu, wl, j);
      }
      uint4 x[TK][kCombVecs];
#pragma unroll
      for (int j = 0; j < TK; ++j)
#pragma unroll
        for (int q = 0; q < kCombVecs; ++q)
          x[j][q] = src[j] && v0 + 32 * q < hv ? __ldg(reinterpret_cast<const uint4*>(src[j]) + v0 + 32 * q)
                                               : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < TK; ++j) {
        if (!src[j]) continue;
#pragma unroll
        for (int q = 0; q < kCombVecs; ++q) fold_bf16x8(acc[q], x[j][q], wj[j], !any);
        any = true;
      }
    } else {
      for (int j = 0; j < R.topk; ++j) {
        const size_t pr = size_t(t) * R.topk + j;
        const int p = R.pos_of[s][pr];
        if (p < 0) continue;
        int d;
        const long long row = route_row(R, base, s, pair_expert(R, s, pr), p, 2, &d);
        if (row < 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(R.buf[d] + size_t(row) * R.hidden * 2);
        const float wj = R.w[s][pr];
#pragma unroll
        for (int q = 0; q < kCombVecs; ++q)
          if (v0 + 32 * q < hv) fold_bf16x8(acc[q], __ldg(src + v0 + 32 * q), wj, !any);
        any = true;
      }
    }
    uint4* y = reinterpret_cast<uint4*>(R.y[s] + size_t(t) * R.hidden * 2);
#pragma unroll
    for (int q = 0; q < kCombVecs; ++q)
      if (v0 + 32 * q < hv) y[v0 + 32 * q] = narrow_bf16x8(acc[q], any);
  }
}

// Combine fed by the tensor-memory accelerator.  Each warp owns two
// shared-memory stages of topk slices (1-4 KiB, by topk); for its work item
// (source, token, slice of the row) lane 0 bulk-loads the slice of every
// valid pair's row into a stage, completing on the stage's mbarrier, and the
// warp folds from shared memory in slot order while the next item's loads are
// in flight.  So the bytes in flight do not take registers: two stages per
// warp.  The pairs' positions, experts and weights are loaded one item
// earlier still, so resolving where an item's rows are costs no wait (at
// the EP workload's shape the combine went from 0.187 to 0.158 ms).  The
// fold starts each sum at -0 (x + -0 = x for every binary32 x, so the first
// product passes unchanged) and adds two elements per instruction.  Needs
// 16-byte-aligned rows, hidden % 8 == 0 and topk <= kBulkTopk.
// Waits are bounded: on a timeout the warp sets status bit 2, waits (bounded)
// for its own loads and stops.
constexpr int kBulkTopk = 8;
constexpr int kCombWarps = 4;                 // warps per CTA
// Bytes of a row per item: the largest of 4, 2 and 1 KiB whose topk slices
// fit a 6 KiB stage (1 KiB from top-4 on).  A stage of about 4-6 KiB per warp
// is what the measurements favour: at 4 KiB rows, top-6, 1 KiB slices took
// 0.187 ms, 2 KiB 0.216 ms, whole rows 0.289 ms (fewer CTAs fit per SM); at
// top-1 and top-2, 1 KiB slices left too few bytes in flight (0.084 and
// 0.092 ms, against 0.049 ms for 4 KiB and 0.069 ms for 2 KiB slices), and
// at top-2 and top-4 the next size up was slower again (4 KiB: 0.078 ms;
// 2 KiB: 0.115 against 0.112 ms).
constexpr uint32_t kCombSlice = 1024;
constexpr uint32_t kCombStage = 6144;
inline uint32_t comb_slice(int topk) {
  uint32_t slice = 4096;
  while (slice > kCombSlice && uint32_t(topk) * slice > kCombStage) slice /= 2;
  return slice;
}

__global__ void __launch_bounds__(32 * kCombWarps) ep_combine_bulk_kernel(const __grid_constant__ EpRoute R,
                                                                         uint32_t slice) {
  using namespace ptx;
  pdl_enter();
  extern __shared__ __align__(128) unsigned char comb_mem[];  // [warps][2 stages][topk][slice]
  __shared__ __align__(8) uint64_t bar[kCombWarps][2];
  __shared__ long long base[kMaxRanks * kMaxRanks];
  route_bases(R, base);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    mbar_init(&bar[warp][0], 1);
    mbar_init(&bar[warp][1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncwarp();
  const uint32_t stage_bytes = uint32_t(R.topk) * slice;
  unsigned char* stages = comb_mem + size_t(warp) * 2 * stage_bytes;
  const uint32_t hb = uint32_t(R.hidden) * 2;
  const uint32_t chunks = (hb + slice - 1) / slice;
  const uint64_t items = uint64_t(R.k) * uint64_t(R.tokens) * chunks;
  const uint64_t warps = uint64_t(gridDim.x) * kCombWarps;
  const uint64_t first = uint64_t(blockIdx.x) * kCombWarps + warp;
  // lane j < topk: pair j of an item (its packed row, expert and weight)
  struct Pair {
    int p, e;
    float w;
  };
  // what an item needs after its loads land
  struct Item {
    int s, t;
    uint32_t off, n;
    unsigned valid;  // bit j: pair j has a row in the stage
    float w;         // lane j < topk: weight of pair j
  };
  auto locate = [&](uint64_t it, int& s, int& t, uint32_t& off) {
    const uint64_t row_it = it / chunks;
    off = uint32_t(it - row_it * chunks) * slice;
    s = int(row_it / uint64_t(R.tokens));
    t = int(row_it - uint64_t(s) * uint64_t(R.tokens));
  };
  // Load item `it`'s pairs (all lanes; nothing waits on them until they are used).
  auto fetch = [&](uint64_t it, Pair& q) {
    int s, t;
    uint32_t off;
    locate(it, s, t, off);
    q.p = -1;
    q.e = 0;
    q.w = 0.f;
    if (lane < R.topk) {
      const size_t pr = size_t(t) * R.topk + lane;
      q.p = R.pos_of[s][pr];
      q.e = pair_expert(R, s, pr);
      q.w = R.w[s][pr];
    }
  };
  // Resolve item `it` from its pairs and, on lane 0, issue its loads into stage `st`.
  auto start = [&](uint64_t it, const Pair& q, int st, Item& I) {
    locate(it, I.s, I.t, I.off);
    I.n = hb - I.off < slice ? hb - I.off : slice;
    const char* src = nullptr;
    I.w = q.w;
    if (q.p >= 0) {
      int d;
      const long long row = route_row(R, base, I.s, q.e, q.p, 2, &d);
      if (row >= 0) src = R.buf[d] + size_t(row) * hb + I.off;
    }
    I.valid = __ballot_sync(0xFFFFFFFFu, src != nullptr);
    uint64_t* b = &bar[warp][st];
    if (lane == 0) mbar_arrive_expect_tx(b, uint32_t(__popc(I.valid)) * I.n + R.tx_pad);
    __syncwarp();
    if (src) bulk_load(stages + size_t(st) * stage_bytes + size_t(lane) * slice, src, I.n, b);
  };
  uint64_t k_items = first < items ? (items - first + warps - 1) / warps : 0;
  Item cur{}, nxt{};
  Pair ahead{};
  bool failed = false;
  uint64_t issued = 0, done = 0;
  if (k_items) {
    fetch(first, ahead);
    start(first, ahead, 0, cur);
    issued = 1;
    if (k_items > 1) fetch(first + warps, ahead);
  }
  for (uint64_t i = 0; i < k_items && !failed; ++i) {
    const int st = int(i & 1);
    if (i + 1 < k_items) {  // the next item's loads go out before this one is folded
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of that stage come first
      start(first + (i + 1) * warps, ahead, st ^ 1, nxt);
      ++issued;
      if (i + 2 < k_items) fetch(first + (i + 2) * warps, ahead);  // and the pairs of the one after
    }
    // every lane waits for the stage itself before reading what the bulk loads wrote
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[warp][st], uint32_t(i >> 1) & 1u,
                                                              global_ns() + R.wait_ns));
    if (!ok) {
      failed = true;
      break;
    }
    ++done;
    float wj[kBulkTopk];
#pragma unroll
    for (int j = 0; j < kBulkTopk; ++j) wj[j] = __shfl_sync(0xFFFFFFFFu, cur.w, j);
    const unsigned char* stage = stages + size_t(st) * stage_bytes;
    const uint32_t nvec = cur.n / 16;
    const bool any = cur.valid != 0;
    uint4* y = reinterpret_cast<uint4*>(R.y[cur.s] + size_t(cur.t) * hb + cur.off);
    for (uint32_t v = lane; v < nvec; v += 32) {
      unsigned long long acc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = 0x8000000080000000ull;  // -0 in both lanes
#pragma unroll
      for (int j = 0; j < kBulkTopk; ++j) {
        if (j >= R.topk || !(cur.valid >> j & 1u)) continue;
        const uint4 x = *reinterpret_cast<const uint4*>(stage + size_t(j) * slice + size_t(v) * 16);
        const uint32_t q[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc[e] = mul_add_bf16x2(acc[e], wj[j], q[e]);
      }
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = any ? __uint_as_float(uint32_t(acc[e])) : 0.f;
        const float hi = any ? __uint_as_float(uint32_t(acc[e] >> 32)) : 0.f;
        o[e] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
      }
      y[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncwarp();
    cur = nxt;
  }
  if (failed && lane == 0) {
    atomicOr(R.status, 4);
    const uint64_t deadline = global_ns() + R.wait_ns;
    for (uint64_t b = done; b < issued; ++b)  // the loads still in flight: bounded again
      if (!mbar_wait_bounded(&bar[warp][b & 1], uint32_t(b >> 1) & 1u, deadline)) break;
  }
}

// Combine, scalar path (hidden not a multiple of 8 or buffers not 16-byte
// aligned): a warp per (source, token), a lane per element.
__global__ void ep_combine_fused_kernel(const __grid_constant__ EpRoute R) {
  pdl_enter();
  __shared__ long long base[kMaxRanks * kMaxRanks];
  route_bases(R, base);
  const int lane = threadIdx.x & 31;
  const long long items = (long long)R.tokens * R.k;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const int s = int(it / R.tokens), t = int(it % R.tokens);
    uint16_t* yrow = reinterpret_cast<uint16_t*>(R.y[s] + size_t(t) * R.hidden * 2);
    for (int h = lane; h < R.hidden; h += 32) {
      float acc = 0.f;
      bool any = false;
      for (int j = 0; j < R.topk; ++j) {
        const size_t pr = size_t(t) * R.topk + j;
        const int p = R.pos_of[s][pr];
        if (p < 0) continue;
        int d;
        const long long row = route_row(R, base, s, pair_expert(R, s, pr), p, 2, &d);
        if (row < 0) continue;
        const uint16_t* src = reinterpret_cast<const uint16_t*>(R.buf[d] + size_t(row) * R.hidden * 2);
        const float prod = __fmul_rn(R.w[s][pr], __uint_as_float(uint32_t(src[h]) << 16));
        acc = any ? __fadd_rn(acc, prod) : prod;
        any = true;
      }
      yrow[h] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
  }
}

int tiles_of(int n) { return (n + kTileItems - 1) / kTileItems; }

// Launch with programmatic stream serialization (see pdl_enter).
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, int block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// A grid of every CTA the device can hold at once for kernel `fn` (256
// threads, no dynamic shared memory), but no more than `want`.
// Grid of the row-scatter kernels: one work item per warp (8 warps per CTA),
// so the block scheduler hands out work as CTAs finish.  At the EP workload
// (8 x 4096 rows of 4 KiB to 6 destinations each) that ran the scatter at
// 0.139 ms against 0.159 ms for a persistent grid of 4 CTAs per SM, whose
// warps each took a fixed share of 13 or 14 items.  Past 2^20 CTAs the
// kernels' grid-stride loops take the rest.
unsigned scatter_grid(long long warps) {
  const long long ctas = (warps + 7) / 8;
  return unsigned(ctas < 1 ? 1 : (ctas < (1LL << 20) ? ctas : (1LL << 20)));
}

int persistent_grid(const void* fn, long long want) {
  int dev = 0, sms = 1, occ = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 256, 0) != cudaSuccess || occ < 1) {
    cudaGetLastError();
    occ = 1;
  }
  const long long cap = (long long)sms * occ;
  return int(want < 1 ? 1 : (want < cap ? want : cap));
}

using CombineIlpFn = void (*)(const uint16_t*, const int32_t*, const float*, int, int, int, uint16_t*);
const CombineIlpFn kCombineIlp[kCombineTopk] = {
    ep_combine_vec_ilp_kernel<1>, ep_combine_vec_ilp_kernel<2>, ep_combine_vec_ilp_kernel<3>,
    ep_combine_vec_ilp_kernel<4>, ep_combine_vec_ilp_kernel<5>, ep_combine_vec_ilp_kernel<6>,
    ep_combine_vec_ilp_kernel<7>, ep_combine_vec_ilp_kernel<8>};

void launch_combine_ilp(int topk, cudaStream_t s, const uint16_t* rows, const int32_t* pos_of, const float* w,
                        int tokens, int hidden, int n_rows, uint16_t* y) {
  const long long items = (long long)tokens * ((hidden / 8 + 31) / 32);  // one warp per item
  const CombineIlpFn fn = kCombineIlp[topk - 1];
  launch_pdl(fn, persistent_grid(reinterpret_cast<const void*>(fn), (items + 7) / 8), 256, 0, s, rows, pos_of, w, tokens,
             hidden, n_rows, y);
}

int grid_for(int items, int per_cta) {
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int want = (items + per_cta - 1) / per_cta;
  const int cap = sms * 8;
  return want < 1 ? 1 : (want < cap ? want : cap);
}

// Per-source scratch of the sort: tile path [experts] totals, [tiles][experts]
// histograms and one valid-pair count; many-experts path [experts] counts.
size_t sort_ws_ints(int n, int experts) {
  return experts <= kMaxTileExperts ? size_t(experts) * (1 + size_t(tiles_of(n))) + 1 : size_t(experts);
}

// Stable counting sort of the n = tokens * topk pairs of `sources` sources in
// one set of launches: pos_of (and perm where wanted) of every source, and the
// per-destination element counts (row s of P.counts).
cudaError_t sort_pairs(const EpSort& P, int sources, int n, int experts, int nranks, int hidden, cudaStream_t s) {
  if (experts <= kMaxTileExperts) {
    // histograms, one scan per source (which writes every destination count),
    // stable placement (which writes every pos_of and the -1 tail of perm)
    const int tiles = tiles_of(n);
    cudaError_t e = launch_pdl(ep_tile_hist_kernel, dim3(tiles, sources), kEpThreads, sizeof(int) * size_t(experts), s,
                               P, n, experts);
    // few histogram cells: every placement CTA scans them itself (no scan launch)
    const int scan_here = size_t(tiles) * experts <= size_t(kPlaceScanCells);
    const size_t stage_ints = size_t(experts) + size_t(tiles) * experts;
    const int staged = stage_ints <= size_t(kScanSmemInts);
    if (e == cudaSuccess && !scan_here)
      e = launch_pdl(ep_scan_kernel, dim3(sources), kScanThreads, staged ? sizeof(int) * stage_ints : 0, s, P, tiles,
                     experts, nranks, experts / nranks, hidden, staged);
    const size_t place_smem = sizeof(int) * (size_t(kEpWarps) + (scan_here ? 2 : 0)) * experts;
    if (e == cudaSuccess)
      e = launch_pdl(ep_tile_place_kernel, dim3(tiles, sources), kEpThreads, place_smem, s, P, n, experts, tiles,
                     scan_here, nranks, experts / nranks, hidden);
    return e;
  }
  // many experts: one CTA per (expert, source) scanning every pair of its source
  for (int src = 0; src < sources; ++src) {
    if (P.perm[src] && cudaMemsetAsync(P.perm[src], 0xFF, sizeof(int32_t) * size_t(n), s) != cudaSuccess)
      return cudaGetLastError();
    if (cudaMemsetAsync(P.pos_of[src], 0xFF, sizeof(int32_t) * size_t(n), s) != cudaSuccess) return cudaGetLastError();
  }
  if (cudaMemsetAsync(P.counts, 0, sizeof(uint64_t) * size_t(sources) * nranks, s) != cudaSuccess)
    return cudaGetLastError();
  ep_count_kernel<<<dim3(experts, sources), kEpThreads, 0, s>>>(P, n);
  ep_place_kernel<<<dim3(experts, sources), kEpThreads, 0, s>>>(P, n, hidden, experts / nranks, nranks);
  return cudaGetLastError();
}

using CombineFusedFn = void (*)(EpRoute);
const CombineFusedFn kCombineFused[kCombineTopk + 1] = {
    ep_combine_fused_vec_kernel<0>, ep_combine_fused_vec_kernel<1>, ep_combine_fused_vec_kernel<2>,
    ep_combine_fused_vec_kernel<3>, ep_combine_fused_vec_kernel<4>, ep_combine_fused_vec_kernel<5>,
    ep_combine_fused_vec_kernel<6>, ep_combine_fused_vec_kernel<7>, ep_combine_fused_vec_kernel<8>};

}  // namespace

cudaError_t ep_preload() {
  const void* fns[] = {reinterpret_cast<const void*>(&ep_count_kernel),
                       reinterpret_cast<const void*>(&ep_place_kernel),
                       reinterpret_cast<const void*>(&ep_tile_hist_kernel),
                       reinterpret_cast<const void*>(&ep_scan_kernel),
                       reinterpret_cast<const void*>(&ep_tile_place_kernel),
                       reinterpret_cast<const void*>(&ep_scatter_kernel),
                       reinterpret_cast<const void*>(&ep_combine_kernel),
                       reinterpret_cast<const void*>(&ep_combine_vec_kernel),
                       reinterpret_cast<const void*>(kCombineIlp[0]), reinterpret_cast<const void*>(kCombineIlp[1]),
                       reinterpret_cast<const void*>(kCombineIlp[2]), reinterpret_cast<const void*>(kCombineIlp[3]),
                       reinterpret_cast<const void*>(kCombineIlp[4]), reinterpret_cast<const void*>(kCombineIlp[5]),
                       reinterpret_cast<const void*>(kCombineIlp[6]), reinterpret_cast<const void*>(kCombineIlp[7]),
                       reinterpret_cast<const void*>(&ep_dispatch_fused_kernel),
                       reinterpret_cast<const void*>(&ep_dispatch_bulk_kernel),
                       reinterpret_cast<const void*>(&ep_combine_bulk_kernel),
                       reinterpret_cast<const void*>(&ep_combine_fused_kernel),
                       reinterpret_cast<const void*>(kCombineFused[0]), reinterpret_cast<const void*>(kCombineFused[1]),
                       reinterpret_cast<const void*>(kCombineFused[2]), reinterpret_cast<const void*>(kCombineFused[3]),
                       reinterpret_cast<const void*>(kCombineFused[4]), reinterpret_cast<const void*>(kCombineFused[5]),
                       reinterpret_cast<const void*>(kCombineFused[6]), reinterpret_cast<const void*>(kCombineFused[7]),
                       reinterpret_cast<const void*>(kCombineFused[8])};
  for (const void* f : fns) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hoc

extern "C" hocResult_t hoc_ep_pack_workspace(int tokens, int topk, int experts, size_t* ints) {
  using namespace hoc;
  if (tokens < 0 || topk < 1 || experts < 1 || !ints) return HOC_ERR_INVALID_ARG;
  if (size_t(tokens) * topk > size_t(INT32_MAX)) return HOC_ERR_INVALID_ARG;
  *ints = sort_ws_ints(tokens * topk, experts);
  return HOC_SUCCESS;
}

extern "C" hocResult_t hoc_ep_pack(const int32_t* expert_ids, const void* x, int tokens, int topk, int hidden,
                                   int experts, int nranks, void* send, int32_t* perm, int32_t* pos_of,
                                   uint64_t* dst_counts, int32_t* workspace, size_t workspace_ints, void* stream) {
  using namespace hoc;
  if (tokens < 0 || topk < 1 || hidden < 1 || experts < 1 || nranks < 1 || experts % nranks != 0)
    return HOC_ERR_INVALID_ARG;
  if (!dst_counts) return HOC_ERR_INVALID_ARG;
  if (tokens == 0)  // nothing to pack: the rank sends nothing to anyone
    return cudaMemsetAsync(dst_counts, 0, sizeof(uint64_t) * size_t(nranks), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? HOC_SUCCESS
               : HOC_ERR_CUDA;
  if (!expert_ids || !x || !send || !perm || !pos_of || !workspace) return HOC_ERR_INVALID_ARG;
  if (size_t(tokens) * topk > size_t(INT32_MAX)) return HOC_ERR_INVALID_ARG;
  size_t need = 0;
  hoc_ep_pack_workspace(tokens, topk, experts, &need);
  if (workspace_ints < need) {
    set_error_detail("hoc_ep_pack: workspace smaller than hoc_ep_pack_workspace() asks for");
    return HOC_ERR_INVALID_ARG;
  }
  const int n = tokens * topk;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EpSort P{};
  P.ids[0] = expert_ids;
  P.perm[0] = perm;
  P.pos_of[0] = pos_of;
  P.counts = reinterpret_cast<unsigned long long*>(dst_counts);
  P.ws = workspace;
  P.ws_stride = need;
  if (sort_pairs(P, 1, n, experts, nranks, hidden, s) != cudaSuccess) {
    set_error_detail("hoc_ep_pack: launching the sort failed");
    return HOC_ERR_CUDA;
  }
  const int hb = hidden * 2;
  const int vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(send)) & 15u) == 0 && hb % 16 == 0;
  const long long scatter_warps = vec ? (long long)tokens * ((hb / 16 + kScatterSliceVecs - 1) / kScatterSliceVecs)
                                      : tokens;
  launch_pdl(ep_scatter_kernel, scatter_grid(scatter_warps), 256, 0, s,
             static_cast<const char*>(x), static_cast<const int32_t*>(pos_of), tokens, topk, hb,
             static_cast<char*>(send), int(vec));
  return cudaGetLastError() == cudaSuccess ? HOC_SUCCESS : HOC_ERR_CUDA;
}

extern "C" hocResult_t hoc_ep_combine(const void* rows, const int32_t* pos_of, const float* weights, int tokens,
                                      int topk, int hidden, void* y, void* stream) {
  using namespace hoc;
  if (tokens < 0 || topk < 1 || hidden < 1) return HOC_ERR_INVALID_ARG;
  if (tokens == 0) return HOC_SUCCESS;
  if (!rows || !pos_of || !weights || !y) return HOC_ERR_INVALID_ARG;
  if (size_t(tokens) * topk > size_t(INT32_MAX)) return HOC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool vec = hidden % 8 == 0 && ((reinterpret_cast<uintptr_t>(rows) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
  if (vec && topk <= kCombineTopk)
    launch_combine_ilp(topk, s, static_cast<const uint16_t*>(rows), pos_of, weights, tokens, hidden, tokens * topk,
                       static_cast<uint16_t*>(y));
  else if (vec)
    ep_combine_vec_kernel<<<grid_for(tokens, 8), 256, 0, s>>>(static_cast<const uint16_t*>(rows), pos_of, weights,
                                                              tokens, topk, hidden, tokens * topk,
                                                              static_cast<uint16_t*>(y));
  else
    ep_combine_kernel<<<grid_for(tokens, 8), 256, 0, s>>>(static_cast<const uint16_t*>(rows), pos_of, weights, tokens,
                                                          topk, hidden, tokens * topk, static_cast<uint16_t*>(y));
  return cudaGetLastError() == cudaSuccess ? HOC_SUCCESS : HOC_ERR_CUDA;
}

namespace hoc {
namespace {

// Bounded waits of the bulk-copy kernels: 2 s, or with HOC_FAULT=ep_stall
// (host-side fault injection, as for the communicator's TMA moves) 0.1 s with
// every mbarrier expecting 16 bytes more than its loads bring.
void set_bulk_waits(EpRoute& R) {
  const char* fault = getenv("HOC_FAULT");
  const bool stall = fault && !strcmp(fault, "ep_stall");
  R.tx_pad = stall ? 16u : 0u;
  R.wait_ns = stall ? 100000000ull : kBulkWaitNs;
}

// Sort of every source's pairs, then the row scatter: into the destination
// ranks' receive buffers (packed = 0, the dispatch fused with the exchange) or
// into each source's own send buffer in packed order (packed = 1).
hocResult_t dispatch_ranks(const char* who, int packed, int nranks, const int32_t* const* expert_ids,
                           const void* const* x, int tokens, int topk, int hidden, int experts, void* const* out,
                           const size_t* out_capacity, int32_t* const* pos_of, uint64_t* counts, int32_t* workspace,
                           size_t workspace_ints, int32_t* status, cudaStream_t s) {
  char msg[160];
  if (nranks < 1 || nranks > kMaxRanks || tokens < 0 || topk < 1 || hidden < 1 || experts < 1 ||
      experts % nranks != 0) {
    snprintf(msg, sizeof msg, "%s: bad rank count, shape or expert count", who);
    set_error_detail(msg);
    return HOC_ERR_INVALID_ARG;
  }
  if (!expert_ids || !x || !out || !out_capacity || !pos_of || !counts || !status) return HOC_ERR_INVALID_ARG;
  if (size_t(tokens) * topk > size_t(INT32_MAX)) return HOC_ERR_INVALID_ARG;
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return HOC_ERR_CUDA;
  if (tokens == 0)  // nobody sends anything
    return cudaMemsetAsync(counts, 0, sizeof(uint64_t) * size_t(nranks) * nranks, s) == cudaSuccess ? HOC_SUCCESS
                                                                                                     : HOC_ERR_CUDA;
  const int n = tokens * topk;
  const size_t per = sort_ws_ints(n, experts);
  if (!workspace || workspace_ints < per * size_t(nranks)) {
    snprintf(msg, sizeof msg, "%s: workspace smaller than nranks * hoc_ep_pack_workspace()", who);
    set_error_detail(msg);
    return HOC_ERR_INVALID_ARG;
  }
  EpSort P{};
  EpRoute R{};
  bool vec = (size_t(hidden) * 2) % 16 == 0;
  for (int r = 0; r < nranks; ++r) {
    if (!expert_ids[r] || !x[r] || !out[r] || !pos_of[r]) {
      snprintf(msg, sizeof msg, "%s: NULL per-rank pointer", who);
      set_error_detail(msg);
      return HOC_ERR_INVALID_ARG;
    }
    P.ids[r] = expert_ids[r];
    P.pos_of[r] = pos_of[r];
    R.x[r] = static_cast<const char*>(x[r]);
    R.ids[r] = expert_ids[r];
    R.pos_of[r] = pos_of[r];
    R.buf[r] = static_cast<char*>(out[r]);
    R.cap_rows[r] = out_capacity[r] / size_t(hidden);
    vec = vec && ((reinterpret_cast<uintptr_t>(x[r]) | reinterpret_cast<uintptr_t>(out[r])) & 15u) == 0;
  }
  P.counts = reinterpret_cast<unsigned long long*>(counts);
  P.ws = workspace;
  P.ws_stride = per;
  if (sort_pairs(P, nranks, n, experts, nranks, hidden, s) != cudaSuccess) {
    snprintf(msg, sizeof msg, "%s: launching the sort failed", who);
    set_error_detail(msg);
    return HOC_ERR_CUDA;
  }
  R.counts = P.counts;
  R.status = status;
  R.k = nranks;
  R.tokens = tokens;
  R.topk = topk;
  R.hidden = hidden;
  R.per_rank = experts / nranks;
  R.packed = packed;
  set_bulk_waits(R);
  const int hb = hidden * 2;
  // Row scatter: per-thread vector copies; with HOC_EP_DISPATCH=bulk (rows and
  // buffers aligned, topk <= 16) bulk copies through shared memory instead --
  // measured equal on GB300 at the EP workload's shape, kept as the TMA engine.
  const char* eng = getenv("HOC_EP_DISPATCH");
  const bool bulk = vec && topk <= kBulkMaxTopk && eng && !strcmp(eng, "bulk");
  cudaError_t e;
  if (bulk) {
    const void* fn = reinterpret_cast<const void*>(&ep_dispatch_bulk_kernel);
    const size_t smem = size_t(kBulkStages) * kBulkPiece;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    int dev = 0, sms = 1, occ = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 32, smem);
    const long long items = (long long)nranks * tokens * ((hb + kBulkPiece - 1) / kBulkPiece);
    const long long cap = (long long)sms * (occ > 0 ? occ : 1);
    if (e == cudaSuccess)
      e = launch_pdl(ep_dispatch_bulk_kernel, dim3(unsigned(items < cap ? items : cap)), 32, smem, s, R);
  } else {
    const long long warps = (long long)nranks * tokens * (vec ? (hb + kDispChunk - 1) / kDispChunk : 1);
    e = launch_pdl(ep_dispatch_fused_kernel, dim3(scatter_grid(warps)), 256, 0, s, R, int(vec));
  }
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "%s: launching the row scatter failed", who);
    set_error_detail(msg);
    return HOC_ERR_CUDA;
  }
  return HOC_SUCCESS;
}

// The combine of every source: rows read from the expert ranks' buffers
// (packed = 0, fused with the combine exchange) or from each source's own
// buffer of returned rows in packed order (packed = 1; ids and counts unused).
hocResult_t combine_ranks(const char* who, int packed, int nranks, const void* const* rows,
                          const size_t* rows_capacity, const int32_t* const* expert_ids,
                          const int32_t* const* pos_of, const uint64_t* counts, const float* const* weights,
                          int tokens, int topk, int hidden, int experts, void* const* y, int32_t* status,
                          cudaStream_t s) {
  char msg[160];
  if (nranks < 1 || nranks > kMaxRanks || tokens < 0 || topk < 1 || hidden < 1 || experts < 1 ||
      experts % nranks != 0) {
    snprintf(msg, sizeof msg, "%s: bad rank count, shape or expert count", who);
    set_error_detail(msg);
    return HOC_ERR_INVALID_ARG;
  }
  if (tokens == 0) return HOC_SUCCESS;
  if (!rows || !rows_capacity || (!packed && (!expert_ids || !counts)) || !pos_of || !weights || !y || !status)
    return HOC_ERR_INVALID_ARG;
  if (size_t(tokens) * topk > size_t(INT32_MAX)) return HOC_ERR_INVALID_ARG;
  EpRoute R{};
  bool vec = hidden % 8 == 0;
  for (int r = 0; r < nranks; ++r) {
    if (!rows[r] || (!packed && !expert_ids[r]) || !pos_of[r] || !weights[r] || !y[r]) {
      snprintf(msg, sizeof msg, "%s: NULL per-rank pointer", who);
      set_error_detail(msg);
      return HOC_ERR_INVALID_ARG;
    }
    R.buf[r] = static_cast<char*>(const_cast<void*>(rows[r]));
    R.cap_rows[r] = rows_capacity[r] / size_t(hidden);
    R.ids[r] = packed ? nullptr : expert_ids[r];
    R.pos_of[r] = pos_of[r];
    R.w[r] = weights[r];
    R.y[r] = static_cast<char*>(y[r]);
    vec = vec && ((reinterpret_cast<uintptr_t>(rows[r]) | reinterpret_cast<uintptr_t>(y[r])) & 15u) == 0;
  }
  R.counts = packed ? nullptr : reinterpret_cast<const unsigned long long*>(counts);
  R.status = status;
  R.k = nranks;
  R.tokens = tokens;
  R.topk = topk;
  R.hidden = hidden;
  R.per_rank = experts / nranks;
  R.packed = packed;
  set_bulk_waits(R);
  cudaError_t e;
  // Rows through shared memory by TMA bulk copies where shapes allow (the
  // default), else (or with HOC_EP_COMBINE=lsu) per-thread vector loads.
  const char* eng = getenv("HOC_EP_COMBINE");
  if (vec && topk <= kBulkTopk && !(eng && !strcmp(eng, "lsu"))) {
    const void* fn = reinterpret_cast<const void*>(&ep_combine_bulk_kernel);
    const uint32_t slice = comb_slice(topk);
    const size_t smem = size_t(kCombWarps) * 2 * size_t(topk) * slice;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    int dev = 0, sms = 1, occ = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 32 * kCombWarps, smem);
    const long long items = (long long)nranks * tokens * ((size_t(hidden) * 2 + slice - 1) / slice);
    const long long want = (items + kCombWarps - 1) / kCombWarps;
    const long long cap = (long long)sms * (occ > 0 ? occ : 1);
    if (e == cudaSuccess)
      e = launch_pdl(ep_combine_bulk_kernel, dim3(unsigned(want < cap ? want : cap)), 32 * kCombWarps, smem, s, R,
                     slice);
  } else if (vec) {
    const CombineFusedFn fn = kCombineFused[topk <= kCombineTopk ? topk : 0];
    const long long items = (long long)nranks * tokens * ((hidden / 8 + kCombChunk - 1) / kCombChunk);  // warps
    e = launch_pdl(fn, dim3(persistent_grid(reinterpret_cast<const void*>(fn), (items + 7) / 8)), 256, 0, s, R);
  } else {
    const void* fn = reinterpret_cast<const void*>(&ep_combine_fused_kernel);
    e = launch_pdl(ep_combine_fused_kernel, dim3(persistent_grid(fn, ((long long)nranks * tokens + 7) / 8)), 256, 0,
                   s, R);
  }
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "%s: launch failed", who);
    set_error_detail(msg);
    return HOC_ERR_CUDA;
  }
  return HOC_SUCCESS;
}

}  // namespace
}  // namespace hoc

extern "C" hocResult_t hoc_ep_dispatch_fused(int nranks, const int32_t* const* expert_ids, const void* const* x,
                                             int tokens, int topk, int hidden, int experts, void* const* recv,
                                             const size_t* recv_capacity, int32_t* const* pos_of, uint64_t* counts,
                                             int32_t* workspace, size_t workspace_ints, int32_t* status, void* stream) {
  return hoc::dispatch_ranks("hoc_ep_dispatch_fused", 0, nranks, expert_ids, x, tokens, topk, hidden, experts, recv,
                             recv_capacity, pos_of, counts, workspace, workspace_ints, status,
                             static_cast<cudaStream_t>(stream));
}

extern "C" hocResult_t hoc_ep_pack_all(int nranks, const int32_t* const* expert_ids, const void* const* x, int tokens,
                                       int topk, int hidden, int experts, void* const* send,
                                       const size_t* send_capacity, int32_t* const* pos_of, uint64_t* counts,
                                       int32_t* workspace, size_t workspace_ints, int32_t* status, void* stream) {
  return hoc::dispatch_ranks("hoc_ep_pack_all", 1, nranks, expert_ids, x, tokens, topk, hidden, experts, send,
                             send_capacity, pos_of, counts, workspace, workspace_ints, status,
                             static_cast<cudaStream_t>(stream));
}

extern "C" hocResult_t hoc_ep_combine_fused(int nranks, const void* const* rows, const size_t* rows_capacity,
                                            const int32_t* const* expert_ids, const int32_t* const* pos_of,
                                            const uint64_t* counts, const float* const* weights, int tokens, int topk,
                                            int hidden, int experts, void* const* y, int32_t* status, void* stream) {
  return hoc::combine_ranks("hoc_ep_combine_fused", 0, nranks, rows, rows_capacity, expert_ids, pos_of, counts,
                            weights, tokens, topk, hidden, experts, y, status, static_cast<cudaStream_t>(stream));
}

extern "C" hocResult_t hoc_ep_combine_all(int nranks, const void* const* rows, const size_t* rows_capacity,
                                          const int32_t* const* pos_of, const float* const* weights, int tokens,
                                          int topk, int hidden, void* const* y, int32_t* status, void* stream) {
  return hoc::combine_ranks("hoc_ep_combine_all", 1, nranks, rows, rows_capacity, nullptr, pos_of, nullptr, weights,
                            tokens, topk, hidden, nranks, y, status, static_cast<cudaStream_t>(stream));
}
