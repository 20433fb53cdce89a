// k-way chunk-reduce kernel: the reduction of ring reduce-scatter with the
// ring's k-1 hops collapsed into one pass over the k rank buffers.
//
// HOCCL (section 5, Limitations) leaves reductions to SM-side execution; the
// fold order here is the textbook ring reduce-scatter hop order: block r
// starts from rank succ(r)'s input and every later hop adds the receiving
// rank's input, ending with r itself.  Because every hop of the ring is
// folded in the same order, the bits equal those of the hop-by-hop ring with
// binary32 partials.
//
// Layout: rank buffers are 1-D arrays in HBM.  A launch covers one element
// range (a chunk) of every block: one segment per block.  Segments are cut into
// tiles of THREADS x VPT 16-byte vectors; CTAs stride over tiles.  Each thread
// issues all k x VPT 16-byte loads before folding.  Two shapes:
//   * whole GPU: 256-thread CTAs, 2 vectors per thread, several CTAs per SM
//     (k * 8 KiB of loads in flight per CTA);
//   * SM budget (one CTA per SM): 1024-thread CTAs, 1 vector per thread, so
//     each of the few SMs keeps k * 16 KiB of loads in flight.
// The whole-GPU grid is 8 waves of the resident CTAs (a finished CTA is
// replaced at once), the fused kernel's k outputs use streaming stores, and
// multi-wave launches use programmatic dependent launch (the next kernel in
// the stream is scheduled into the slots the last wave frees).
//
// Arithmetic: fp32 adds rounded to nearest even, no flush to zero, two lanes per
// instruction (add.rn.f32x2, the same bits as __fadd_rn; scalar __fadd_rn on the
// scalar path); bf16 widens exactly to fp32, adds in fp32 and rounds once
// with __float2bfloat16_rn; int32 adds modulo 2^32 in uint32.
#include <cuda_bf16.h>

#include "f32x2.cuh"
#include "hoc_internal.h"

namespace hoc {
namespace {

constexpr int kThreadsNarrow = 256, kVecNarrow = 2;  // whole GPU
constexpr int kThreadsWide = 1024, kVecWide = 1;     // one CTA per SM under a budget

__host__ __device__ inline int lanes_of(int dtype) { return dtype == HOC_BFLOAT16 ? 8 : 4; }
__host__ __device__ inline uint64_t tile_vecs(bool wide) {
  return wide ? uint64_t(kThreadsWide) * kVecWide : uint64_t(kThreadsNarrow) * kVecNarrow;
}

// Elements before the first 16-byte-aligned element of a vector segment.
__host__ __device__ inline uint64_t seg_head(const ReduceSeg& s, int lanes) {
  const uint64_t mis = s.elem_off % lanes;
  uint64_t h = mis ? uint64_t(lanes) - mis : 0;
  return h > s.elems ? s.elems : h;
}

__host__ __device__ inline uint64_t seg_tiles(const ReduceSeg& s, int lanes, uint64_t tvecs) {
  if (s.elems == 0) return 0;
  if (s.vec) {
    const uint64_t nvec = (s.elems - seg_head(s, lanes)) / lanes;
    const uint64_t t = (nvec + tvecs - 1) / tvecs;
    return t ? t : 1;
  }
  const uint64_t per = tvecs * lanes;
  return (s.elems + per - 1) / per;
}

// ---------------------------------------------------------------- dtype traits
struct TrF32 {
  static constexpr int kLanes = 4;
  static constexpr int kBytes = 4;
  using Elem = uint32_t;
  struct Acc { unsigned long long v[2]; };  // lanes (0, 1) and (2, 3), two binary32 sums per add
  struct Acc1 { float v; };
  __device__ static Acc widen(uint4 x) { return {{pack_f32x2(x.x, x.y), pack_f32x2(x.z, x.w)}}; }
  __device__ static void add(Acc& a, uint4 x) {
    a.v[0] = add_f32x2(a.v[0], pack_f32x2(x.x, x.y));
    a.v[1] = add_f32x2(a.v[1], pack_f32x2(x.z, x.w));
  }
  __device__ static uint4 narrow(const Acc& a) {
    return make_uint4(uint32_t(a.v[0]), uint32_t(a.v[0] >> 32), uint32_t(a.v[1]), uint32_t(a.v[1] >> 32));
  }
  __device__ static Acc1 widen1(Elem e) { return {__uint_as_float(e)}; }
  __device__ static void add1(Acc1& a, Elem e) { a.v = __fadd_rn(a.v, __uint_as_float(e)); }
  __device__ static Elem narrow1(const Acc1& a) { return __float_as_uint(a.v); }
};

struct TrI32 {
  static constexpr int kLanes = 4;
  static constexpr int kBytes = 4;
  using Elem = uint32_t;
  struct Acc { uint32_t v[4]; };
  struct Acc1 { uint32_t v; };
  __device__ static Acc widen(uint4 x) { return {{x.x, x.y, x.z, x.w}}; }
  __device__ static void add(Acc& a, uint4 x) {
    a.v[0] += x.x;
    a.v[1] += x.y;
    a.v[2] += x.z;
    a.v[3] += x.w;
  }
  __device__ static uint4 narrow(const Acc& a) { return make_uint4(a.v[0], a.v[1], a.v[2], a.v[3]); }
  __device__ static Acc1 widen1(Elem e) { return {e}; }
  __device__ static void add1(Acc1& a, Elem e) { a.v += e; }
  __device__ static Elem narrow1(const Acc1& a) { return a.v; }
};

struct TrBF16 {
  static constexpr int kLanes = 8;
  static constexpr int kBytes = 2;
  using Elem = uint16_t;
  // Element 2w is the low half of 32-bit word w (little endian); acc.v[w]
  // holds elements (2w, 2w + 1) widened, two binary32 sums per add.
  struct Acc { unsigned long long v[4]; };
  struct Acc1 { float v; };
  __device__ static Acc widen(uint4 x) { return {{bf16_pair(x.x), bf16_pair(x.y), bf16_pair(x.z), bf16_pair(x.w)}}; }
  __device__ static void add(Acc& a, uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) a.v[i] = add_f32x2(a.v[i], bf16_pair(w[i]));
  }
  __device__ static uint4 narrow(const Acc& a) {
    return make_uint4(bf16_narrow_pair(a.v[0]), bf16_narrow_pair(a.v[1]), bf16_narrow_pair(a.v[2]),
                      bf16_narrow_pair(a.v[3]));
  }
  __device__ static Acc1 widen1(Elem e) { return {__uint_as_float(uint32_t(e) << 16)}; }
  __device__ static void add1(Acc1& a, Elem e) { a.v = __fadd_rn(a.v, __uint_as_float(uint32_t(e) << 16)); }
  __device__ static Elem narrow1(const Acc1& a) { return __bfloat16_as_ushort(__float2bfloat16_rn(a.v)); }
};

__device__ __forceinline__ const void* at(const void* base, uint64_t elem, int bytes) {
  return static_cast<const char*>(base) + elem * uint64_t(bytes);
}
__device__ __forceinline__ void* at(void* base, uint64_t elem, int bytes) {
  return static_cast<char*>(base) + elem * uint64_t(bytes);
}

// Broadcast outputs (the fused allreduce) are not read again soon: streaming
// stores keep them from displacing the inputs' lines in L2.  The owner-only
// output of the copy-engine path is read right away by the all-gather copies,
// so it is stored normally and stays in L2 for them.
template <class Tr>
__device__ __forceinline__ void store_vec(const ReduceParams& p, uint32_t owner, int k, uint64_t o, uint4 y) {
  if (p.broadcast) {
    for (int r = 0; r < k; ++r) __stcs(static_cast<uint4*>(at(p.out[r], o, Tr::kBytes)), y);
  } else {
    *static_cast<uint4*>(at(p.out[owner], o, Tr::kBytes)) = y;
  }
}

// One element through the scalar path (heads, tails, misaligned segments).
template <class Tr>
__device__ __forceinline__ void scalar_elem(const ReduceParams& p, const uint8_t* seq, uint32_t owner, int k,
                                            uint64_t e, uint64_t o) {
  using E = typename Tr::Elem;
  typename Tr::Acc1 acc = Tr::widen1(*static_cast<const E*>(at(p.in[seq[0]], e, Tr::kBytes)));
  for (int j = 1; j < k; ++j) Tr::add1(acc, *static_cast<const E*>(at(p.in[seq[j]], e, Tr::kBytes)));
  const E y = Tr::narrow1(acc);
  if (p.broadcast) {
    for (int r = 0; r < k; ++r) *static_cast<E*>(at(p.out[r], o, Tr::kBytes)) = y;
  } else {
    *static_cast<E*>(at(p.out[owner], o, Tr::kBytes)) = y;
  }
}

// K > 0: compile-time rank count (all loads hoisted); K == 0: runtime p.k.
constexpr int kRuntimeGroup = 4;
template <class Tr, int K, int kThreads, int kVecPerThread>
__global__ void __launch_bounds__(kThreads) reduce_kernel(const __grid_constant__ ReduceParams p) {
  // Programmatic dependent launch (both no-ops for a launch without the
  // attribute): wait until the grid before this one in the stream has
  // completed and its writes are visible, then let the next grid launch.  A
  // multi-wave grid triggers only once its last wave has started, so the next
  // grid's CTAs take the SM slots this one's last wave frees.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int L = Tr::kLanes;
  constexpr uint64_t kTileVecs = uint64_t(kThreads) * kVecPerThread;
  const int k = K > 0 ? K : p.k;
  const uint64_t total = p.tile_start[p.nseg];
  for (uint64_t t = blockIdx.x; t < total; t += gridDim.x) {
    int s = 0;
    while (t >= p.tile_start[s + 1]) ++s;
    const ReduceSeg& sg = p.seg[s];
    const uint64_t lt = t - p.tile_start[s];
    const uint8_t* seq = p.seq[sg.owner];
    if (sg.vec) {
      const uint64_t head = seg_head(sg, L);
      const uint64_t body = sg.elems - head;
      const uint64_t nvec = body / L;
      const uint64_t e0 = sg.elem_off + head;
      const uint64_t o0 = sg.out_off + head;
      const uint64_t vbase = lt * kTileVecs + threadIdx.x;
      if constexpr (K > 0) {
        uint4 x[K][kVecPerThread];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          const uint64_t v = vbase + uint64_t(i) * kThreads;
          if (v < nvec) {
#pragma unroll
            for (int j = 0; j < K; ++j) x[j][i] = __ldcs(static_cast<const uint4*>(at(p.in[seq[j]], e0 + v * L, Tr::kBytes)));
          }
        }
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          const uint64_t v = vbase + uint64_t(i) * kThreads;
          if (v < nvec) {
            typename Tr::Acc acc = Tr::widen(x[0][i]);
#pragma unroll
            for (int j = 1; j < K; ++j) Tr::add(acc, x[j][i]);
            store_vec<Tr>(p, sg.owner, K, o0 + v * L, Tr::narrow(acc));
          }
        }
      } else {
        // Runtime k: the operands after the first come in groups of
        // kRuntimeGroup, every load of a group issued before its adds (which
        // stay in ring order), so that a thread keeps as many loads in flight
        // as the compile-time kernels do.
        typename Tr::Acc acc[kVecPerThread];
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          const uint64_t v = vbase + uint64_t(i) * kThreads;
          if (v < nvec) acc[i] = Tr::widen(__ldcs(static_cast<const uint4*>(at(p.in[seq[0]], e0 + v * L, Tr::kBytes))));
        }
        for (int j0 = 1; j0 < k; j0 += kRuntimeGroup) {
          uint4 x[kRuntimeGroup][kVecPerThread];
#pragma unroll
          for (int g = 0; g < kRuntimeGroup; ++g)
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) {
              const uint64_t v = vbase + uint64_t(i) * kThreads;
              if (j0 + g < k && v < nvec)
                x[g][i] = __ldcs(static_cast<const uint4*>(at(p.in[seq[j0 + g]], e0 + v * L, Tr::kBytes)));
            }
#pragma unroll
          for (int g = 0; g < kRuntimeGroup; ++g)
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) {
              const uint64_t v = vbase + uint64_t(i) * kThreads;
              if (j0 + g < k && v < nvec) Tr::add(acc[i], x[g][i]);
            }
        }
#pragma unroll
        for (int i = 0; i < kVecPerThread; ++i) {
          const uint64_t v = vbase + uint64_t(i) * kThreads;
          if (v < nvec) store_vec<Tr>(p, sg.owner, k, o0 + v * L, Tr::narrow(acc[i]));
        }
      }
      if (lt == 0 && threadIdx.x < head) scalar_elem<Tr>(p, seq, sg.owner, k, sg.elem_off + threadIdx.x, sg.out_off + threadIdx.x);
      const uint64_t tail = body - nvec * L;
      const uint64_t last = p.tile_start[s + 1] - p.tile_start[s] - 1;
      if (lt == last && threadIdx.x < tail)
        scalar_elem<Tr>(p, seq, sg.owner, k, e0 + nvec * L + threadIdx.x, o0 + nvec * L + threadIdx.x);
    } else {
      const uint64_t base = lt * kTileVecs * L;
#pragma unroll 4
      for (int i = 0; i < kVecPerThread * L; ++i) {
        const uint64_t e = base + uint64_t(i) * kThreads + threadIdx.x;
        if (e < sg.elems) scalar_elem<Tr>(p, seq, sg.owner, k, sg.elem_off + e, sg.out_off + e);
      }
    }
  }
}

template <class Tr, int T, int V>
const void* pick_kernel(int k) {
  switch (k) {
    case 2: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 2, T, V>);
    case 3: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 3, T, V>);
    case 4: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 4, T, V>);
    case 5: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 5, T, V>);
    case 6: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 6, T, V>);
    case 7: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 7, T, V>);
    case 8: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 8, T, V>);
    default: return reinterpret_cast<const void*>(&reduce_kernel<Tr, 0, T, V>);
  }
}

template <class Tr>
const void* pick_shape(int k, bool wide) {
  return wide ? pick_kernel<Tr, kThreadsWide, kVecWide>(k) : pick_kernel<Tr, kThreadsNarrow, kVecNarrow>(k);
}

const void* kernel_for(int dtype, int k, bool wide) {
  switch (dtype) {
    case HOC_FLOAT32: return pick_shape<TrF32>(k, wide);
    case HOC_INT32: return pick_shape<TrI32>(k, wide);
    case HOC_BFLOAT16: return pick_shape<TrBF16>(k, wide);
    default: return nullptr;
  }
}

}  // namespace

uint64_t reduce_seg_tiles(int dtype, const ReduceSeg& s, bool wide) {
  return seg_tiles(s, lanes_of(dtype), tile_vecs(wide));
}

int reduce_ctas_per_sm(int dtype, int k, int /*broadcast*/) {
  const void* fn = kernel_for(dtype, k, false);
  if (!fn) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreadsNarrow, 0) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 1;
  }
  return n;
}

cudaError_t reduce_preload() {
  const int dtypes[] = {HOC_FLOAT32, HOC_INT32, HOC_BFLOAT16};
  for (int dt : dtypes)
    for (int k = 1; k <= kMaxRanks + 1; ++k)  // k outside 2..8 selects the generic-k kernel
      for (int wide = 0; wide < 2; ++wide) {
        cudaFuncAttributes a;
        const cudaError_t e = cudaFuncGetAttributes(&a, kernel_for(dt, k, wide != 0));
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

cudaError_t launch_reduce(const ReduceParams& p, int grid, bool wide, cudaStream_t stream, bool overlap_launch) {
  const void* fn = kernel_for(p.dtype, p.k, wide);
  if (!fn) return cudaErrorInvalidValue;
  if (grid < 1) return cudaSuccess;
  void* args[] = {const_cast<ReduceParams*>(&p)};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(wide ? kThreadsWide : kThreadsNarrow);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_launch ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace hoc
