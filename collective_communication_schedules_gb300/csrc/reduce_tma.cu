// k-way chunk-reduce fed by the tensor-memory accelerator.
//
// Same fold as reduce.cu (ring order: succ(owner), ..., owner; binary32 adds
// with round to nearest even, bf16 rounded once at the end; int32 modulo 2^32)
// and the same segments, but the bytes move by bulk asynchronous copies
// instead of per-thread loads and stores:
//   * one producer warp per CTA streams the k operand tiles of a work tile
//     (tile_bytes each, operand j = ring position j, issued by lane j) into
//     a shared-memory stage with cp.async.bulk, completing on that stage's
//     "full" mbarrier;
//   * eight consumer warps fold the k tiles vector by vector from shared
//     memory, store each folded 16-byte vector straight to the owner's buffer
//     (or to all k buffers: the fused allreduce, with streaming stores), and
//     release the stage on its "empty" mbarrier;
//   * stages cycle, so up to ~190 KiB of operand loads are in flight per SM
//     while the consumers fold -- more than per-thread loads can keep in
//     registers, which is what an SM budget needs.
// One CTA per SM (persistent over tiles).  Only the 16-byte-aligned body of
// each segment moves by bulk copies; the few elements before the first
// aligned element and after the last whole vector go through plain loads.
//
// Every mbarrier wait is bounded by the global timer; on a timeout the CTA
// records a status code, stops issuing work, waits (bounded) for its own
// loads in flight and returns.
#include <cuda_bf16.h>

#include "f32x2.cuh"
#include "hoc_internal.h"
#include "ptx_async.cuh"

namespace hoc {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreadsT = kConsumers + 32;  // + one producer warp

using namespace ptx;

// Barrier over the consumer warps that also ORs a predicate: every consumer
// gets the same answer, so they leave the loop together.
__device__ __forceinline__ bool consumers_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v)), "n"(kConsumers)
      : "memory");
  return r != 0;
}

__host__ __device__ inline int lanes_for(int dtype) { return dtype == HOC_BFLOAT16 ? 8 : 4; }
__host__ __device__ inline int bytes_for(int dtype) { return dtype == HOC_BFLOAT16 ? 2 : 4; }

// Work tiles of a segment: the aligned body cut into tile_bytes pieces (the
// last may be shorter, always a multiple of 16 bytes); at least one tile when
// the segment is not empty, so that its head and tail elements get an owner.
__host__ __device__ inline uint64_t tma_seg_body_vecs(const ReduceSeg& s, int lanes) {
  const uint64_t mis = s.elem_off % lanes;
  uint64_t h = mis ? lanes - mis : 0;
  if (h > s.elems) h = s.elems;
  return (s.elems - h) / lanes;
}
__host__ __device__ inline uint64_t tma_seg_tiles(const ReduceSeg& s, int dtype, uint32_t tile_bytes) {
  if (s.elems == 0) return 0;
  const uint64_t vecs_per_tile = tile_bytes / 16;
  const uint64_t v = tma_seg_body_vecs(s, lanes_for(dtype));
  const uint64_t t = (v + vecs_per_tile - 1) / vecs_per_tile;
  return t ? t : 1;
}

template <class E, class F, class N>
__device__ __forceinline__ void scalar_fold(const ReduceParams& p, const uint8_t* seq, uint32_t owner, uint64_t e,
                                            uint64_t o, F widen_add, N narrow) {
  float acc = 0.f;
  uint32_t iacc = 0;
  for (int j = 0; j < p.k; ++j) {
    const E x = static_cast<const E*>(p.in[seq[j]])[e];
    widen_add(acc, iacc, x, j == 0);
  }
  const E y = narrow(acc, iacc);
  if (p.broadcast) {
    for (int r = 0; r < p.k; ++r) static_cast<E*>(p.out[r])[o] = y;
  } else {
    static_cast<E*>(p.out[owner])[o] = y;
  }
}

__device__ __forceinline__ void scalar_elem(const ReduceParams& p, const uint8_t* seq, uint32_t owner, uint64_t e,
                                            uint64_t o) {
  if (p.dtype == HOC_BFLOAT16) {
    scalar_fold<uint16_t>(
        p, seq, owner, e, o,
        [](float& a, uint32_t&, uint16_t x, bool first) {
          const float v = __uint_as_float(uint32_t(x) << 16);
          a = first ? v : __fadd_rn(a, v);
        },
        [](float a, uint32_t) { return static_cast<uint16_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))); });
  } else if (p.dtype == HOC_FLOAT32) {
    scalar_fold<uint32_t>(
        p, seq, owner, e, o,
        [](float& a, uint32_t&, uint32_t x, bool first) {
          const float v = __uint_as_float(x);
          a = first ? v : __fadd_rn(a, v);
        },
        [](float a, uint32_t) { return __float_as_uint(a); });
  } else {
    scalar_fold<uint32_t>(
        p, seq, owner, e, o, [](float&, uint32_t& a, uint32_t x, bool first) { a = first ? x : a + x; },
        [](float, uint32_t a) { return a; });
  }
}

// Fold one 16-byte vector position of the k tiles in a stage.  K > 0: the
// rank count is a compile-time constant and all K shared-memory loads are
// issued before the adds; K == 0: runtime k.  Floating-point sums run two
// binary32 lanes per instruction (f32x2.cuh), the same bits as scalar adds.

template <int K>
__device__ __forceinline__ uint4 fold_vec(const unsigned char* stage, uint32_t tile_bytes, int k, uint32_t off,
                                          int dtype) {
  const int n = K > 0 ? K : k;
  auto tile = [&](int j) { return *reinterpret_cast<const uint4*>(stage + size_t(j) * tile_bytes + off); };
  if constexpr (K > 0) {
    uint4 v[K];
#pragma unroll
    for (int j = 0; j < K; ++j) v[j] = tile(j);
    if (dtype == HOC_BFLOAT16) {
      unsigned long long a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = bf16_pair((&v[0].x)[i]);
#pragma unroll
      for (int j = 1; j < K; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = add_f32x2(a[i], bf16_pair((&v[j].x)[i]));
      return make_uint4(bf16_narrow_pair(a[0]), bf16_narrow_pair(a[1]), bf16_narrow_pair(a[2]),
                        bf16_narrow_pair(a[3]));
    }
    if (dtype == HOC_FLOAT32) {
      unsigned long long a0 = pack_f32x2(v[0].x, v[0].y), a1 = pack_f32x2(v[0].z, v[0].w);
#pragma unroll
      for (int j = 1; j < K; ++j) {
        a0 = add_f32x2(a0, pack_f32x2(v[j].x, v[j].y));
        a1 = add_f32x2(a1, pack_f32x2(v[j].z, v[j].w));
      }
      return make_uint4(uint32_t(a0), uint32_t(a0 >> 32), uint32_t(a1), uint32_t(a1 >> 32));
    }
    uint4 x = v[0];
#pragma unroll
    for (int j = 1; j < K; ++j) {
      x.x += v[j].x;
      x.y += v[j].y;
      x.z += v[j].z;
      x.w += v[j].w;
    }
    return x;
  }
  uint4 x = tile(0);
  if (dtype == HOC_BFLOAT16) {
    unsigned long long a[4] = {bf16_pair(x.x), bf16_pair(x.y), bf16_pair(x.z), bf16_pair(x.w)};
    for (int j = 1; j < n; ++j) {
      const uint4 y = tile(j);
      a[0] = add_f32x2(a[0], bf16_pair(y.x));
      a[1] = add_f32x2(a[1], bf16_pair(y.y));
      a[2] = add_f32x2(a[2], bf16_pair(y.z));
      a[3] = add_f32x2(a[3], bf16_pair(y.w));
    }
    return make_uint4(bf16_narrow_pair(a[0]), bf16_narrow_pair(a[1]), bf16_narrow_pair(a[2]), bf16_narrow_pair(a[3]));
  }
  if (dtype == HOC_FLOAT32) {
    unsigned long long a0 = pack_f32x2(x.x, x.y), a1 = pack_f32x2(x.z, x.w);
    for (int j = 1; j < n; ++j) {
      const uint4 y = tile(j);
      a0 = add_f32x2(a0, pack_f32x2(y.x, y.y));
      a1 = add_f32x2(a1, pack_f32x2(y.z, y.w));
    }
    return make_uint4(uint32_t(a0), uint32_t(a0 >> 32), uint32_t(a1), uint32_t(a1 >> 32));
  }
  for (int j = 1; j < n; ++j) {
    const uint4 y = tile(j);
    x.x += y.x;
    x.y += y.y;
    x.z += y.z;
    x.w += y.w;
  }
  return x;
}

struct TileRef {
  int seg;
  uint64_t local;
};

__device__ __forceinline__ TileRef tile_of(const ReduceParams& p, uint64_t t) {
  int s = 0;
  while (t >= p.tile_start[s + 1]) ++s;
  return {s, t - p.tile_start[s]};
}

// Byte range [off, off + n) of the segment's aligned body covered by a tile.
__device__ __forceinline__ void tile_body(const ReduceParams& p, const ReduceSeg& sg, uint64_t local,
                                          uint32_t tile_bytes, uint64_t& body_elem0, uint64_t& off_b, uint32_t& n) {
  const int lanes = lanes_for(p.dtype);
  const uint64_t mis = sg.elem_off % lanes;
  uint64_t h = mis ? lanes - mis : 0;
  if (h > sg.elems) h = sg.elems;
  body_elem0 = h;
  const uint64_t body_bytes = tma_seg_body_vecs(sg, lanes) * 16;
  off_b = local * tile_bytes;
  n = off_b >= body_bytes ? 0u : uint32_t(body_bytes - off_b < tile_bytes ? body_bytes - off_b : tile_bytes);
}

template <int K>
__global__ void __launch_bounds__(kThreadsT, 1)
    reduce_tma_kernel(const __grid_constant__ ReduceParams p, uint32_t tile_bytes, int stages, int* status,
                      uint64_t wait_ns, uint32_t tx_pad) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[8];
  __shared__ __align__(8) uint64_t empty[8];
  __shared__ int abort_flag;
  const int k = p.k;
  const int eb = bytes_for(p.dtype);
  const uint32_t stage_bytes = uint32_t(k) * tile_bytes;
  const uint64_t total = p.tile_start[p.nseg];
  const uint64_t mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // The whole warp: every lane waits for the stage to be free, lane 0 sets
    // the stage's expected bytes, and lane j < k issues operand j's bulk load,
    // so the k loads of a stage go out in parallel (one thread issuing them
    // one after another was what bounded this kernel under an SM budget).
    uint64_t issued = 0;
    for (uint64_t it = 0; it < mine; ++it) {
      const int s = int(it % stages);
      bool ok = true;
      if (it >= uint64_t(stages))
        ok = mbar_wait_bounded(&empty[s], uint32_t((it / stages - 1) & 1), global_ns() + wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        if (lane == 0) {
          atomicExch(status, kStatusTimeoutLoad);
          atomicExch(&abort_flag, 1);
        }
        break;
      }
      if (__any_sync(0xFFFFFFFFu, *(volatile int*)&abort_flag != 0)) break;
      const TileRef tr = tile_of(p, blockIdx.x + it * gridDim.x);
      const ReduceSeg& sg = p.seg[tr.seg];
      uint64_t e0, off;
      uint32_t n;
      tile_body(p, sg, tr.local, tile_bytes, e0, off, n);
      if (n == 0) {
        if (lane == 0) mbar_arrive(&full[s]);  // nothing to load (a segment shorter than one vector)
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&full[s], n * uint32_t(k) + tx_pad);  // tx_pad: injected stalls only
        __syncwarp();
        if (lane < k) {
          const uint8_t* seq = p.seq[sg.owner];
          const uint64_t gb = (sg.elem_off + e0) * eb + off;
          bulk_load(smem + size_t(s) * stage_bytes + size_t(lane) * tile_bytes,
                    static_cast<const char*>(p.in[seq[lane]]) + gb, n, &full[s]);
        }
      }
      issued = it + 1;
    }
    // Do not leave while loads still target this CTA's shared memory.
    if (lane == 0) {
      const uint64_t first = issued > uint64_t(stages) ? issued - stages : 0;
      const uint64_t deadline = global_ns() + wait_ns;
      for (uint64_t it = first; it < issued; ++it)
        if (!mbar_wait_bounded(&full[it % stages], uint32_t((it / stages) & 1), deadline)) {
          atomicExch(status, kStatusTimeoutDrain);
          break;
        }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int ct = threadIdx.x - 32;
  for (uint64_t it = 0; it < mine; ++it) {
    const int s = int(it % stages);
    bool bad = !mbar_wait_bounded(&full[s], uint32_t((it / stages) & 1), global_ns() + wait_ns);
    if (bad) atomicExch(status, kStatusTimeoutLoad);
    bad = bad || *(volatile int*)&abort_flag;
    if (consumers_sync_or(bad)) {
      if (lane == 0) atomicExch(&abort_flag, 1);
      break;
    }
    const TileRef tr = tile_of(p, blockIdx.x + it * gridDim.x);
    const ReduceSeg& sg = p.seg[tr.seg];
    const uint8_t* seq = p.seq[sg.owner];
    uint64_t e0, off;
    uint32_t n;
    tile_body(p, sg, tr.local, tile_bytes, e0, off, n);
    const unsigned char* stage = smem + size_t(s) * stage_bytes;
    const uint64_t gb = (sg.out_off + e0) * eb + off;  // byte offset of the tile in the output buffers
    for (uint32_t v = uint32_t(ct) * 16; v < n; v += kConsumers * 16) {
      const uint4 y = fold_vec<K>(stage, tile_bytes, k, v, p.dtype);
      if (p.broadcast) {
        for (int r = 0; r < k; ++r) __stcs(reinterpret_cast<uint4*>(static_cast<char*>(p.out[r]) + gb + v), y);
      } else {
        *reinterpret_cast<uint4*>(static_cast<char*>(p.out[sg.owner]) + gb + v) = y;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    // head and tail elements of the segment (plain loads)
    const uint64_t tiles_here = p.tile_start[tr.seg + 1] - p.tile_start[tr.seg];
    if (tr.local == 0 && uint64_t(ct) < e0) scalar_elem(p, seq, sg.owner, sg.elem_off + ct, sg.out_off + ct);
    if (tr.local == tiles_here - 1) {
      const uint64_t done = e0 + tma_seg_body_vecs(sg, lanes_for(p.dtype)) * lanes_for(p.dtype);
      if (uint64_t(ct) < sg.elems - done) scalar_elem(p, seq, sg.owner, sg.elem_off + done + ct, sg.out_off + done + ct);
    }
  }
}

}  // namespace

// Operand tile per rank: as large as two stages of k tiles allow in ~200 KiB of
// shared memory.  A stage is folded only once all k of its tiles are in, so
// while the consumers fold one stage about one stage of loads is in flight,
// and the time per tile grows with a fixed part (load latency, the stage
// handshake) plus its bytes: at 8 ranks under a 4-SM budget a 25 MiB
// reduce-scatter takes 1.82 / 1.39 / 1.12 / 0.92 ms with 4 / 6 / 8 / 12 KiB
// tiles (register-fed kernel: 0.77 ms).  Across rank counts a stage of about
// 64-96 KiB did best in the fused allreduce of 256 MiB bf16 per rank on all
// SMs: at k = 2, 32 KiB tiles read 0.96 of the measured copy rate against
// 0.80 with 16 KiB; at k = 3, 24 KiB 0.89 against 0.85 (16 KiB) and 0.86
// (32 KiB); at k = 4, 20 KiB 0.90 against 0.88; at k = 12 and 16, 6 KiB 0.94
// and 0.91 against 0.87 and 0.89 with 4 KiB.
uint32_t reduce_tma_tile_bytes(int k) {
  return k <= 2 ? 32768u : (k <= 3 ? 24576u : (k <= 4 ? 20480u : (k <= 8 ? 12288u : 6144u)));
}

int reduce_tma_stages(int k) {
  const uint32_t stage = uint32_t(k) * reduce_tma_tile_bytes(k);
  const uint32_t budget = 200u * 1024u;
  int s = int(budget / stage);
  return s < 2 ? 2 : (s > 8 ? 8 : s);
}

size_t reduce_tma_smem(int k) { return size_t(reduce_tma_stages(k)) * k * reduce_tma_tile_bytes(k); }

uint64_t reduce_tma_seg_tiles(int dtype, const ReduceSeg& s, int k) {
  return tma_seg_tiles(s, dtype, reduce_tma_tile_bytes(k));
}

namespace {
// The kernel for rank count k: compile-time k for 2..8, runtime k otherwise.
const void* reduce_tma_fn(int k) {
  switch (k) {
    case 2: return reinterpret_cast<const void*>(&reduce_tma_kernel<2>);
    case 3: return reinterpret_cast<const void*>(&reduce_tma_kernel<3>);
    case 4: return reinterpret_cast<const void*>(&reduce_tma_kernel<4>);
    case 5: return reinterpret_cast<const void*>(&reduce_tma_kernel<5>);
    case 6: return reinterpret_cast<const void*>(&reduce_tma_kernel<6>);
    case 7: return reinterpret_cast<const void*>(&reduce_tma_kernel<7>);
    case 8: return reinterpret_cast<const void*>(&reduce_tma_kernel<8>);
    default: return reinterpret_cast<const void*>(&reduce_tma_kernel<0>);
  }
}
}  // namespace

cudaError_t reduce_tma_prepare() {
  for (int k = 1; k <= kMaxRanks + 1; ++k) {  // k = 1 and k > 8 select the runtime-k kernel
    const cudaError_t e = cudaFuncSetAttribute(reduce_tma_fn(k), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               int(reduce_tma_smem(k > kMaxRanks ? kMaxRanks : k)));
    if (e != cudaSuccess) return e;
  }
  size_t most = 0;  // the runtime-k kernel serves every k outside 2..8
  for (int k = 1; k <= kMaxRanks; ++k) most = reduce_tma_smem(k) > most ? reduce_tma_smem(k) : most;
  return cudaFuncSetAttribute(reduce_tma_fn(0), cudaFuncAttributeMaxDynamicSharedMemorySize, int(most));
}

cudaError_t tma_preload() {
  for (int k = 0; k <= 8; ++k) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, reduce_tma_fn(k));
    if (e != cudaSuccess) return e;
  }
  return tma_copy_preload();
}

cudaError_t launch_reduce_tma(const ReduceParams& p, int grid, int* status, cudaStream_t stream, uint32_t tx_pad,
                              uint64_t wait_ns) {
  if (grid < 1) return cudaSuccess;
  uint32_t tb = reduce_tma_tile_bytes(p.k);
  int stages = reduce_tma_stages(p.k);
  void* args[] = {const_cast<ReduceParams*>(&p), &tb, &stages, &status, &wait_ns, &tx_pad};
  return cudaLaunchKernel(reduce_tma_fn(p.k), dim3(grid), dim3(kThreadsT), args, reduce_tma_smem(p.k), stream);
}

}  // namespace hoc
