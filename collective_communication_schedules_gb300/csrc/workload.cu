// Kernels that run beside the collectives: the compute-bound FMA probe whose
// slowdown measures SM contention (HOCCL section 2.1, Eq. 1 and Fig. 2b) and
// the XOR transform that stands in for a pipeline stage's compute.
#include "hoc_internal.h"
#include "hoc_workload.h"

namespace hoc {
namespace {

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// CTA 0's thread 0 reports how many SM cycles and nanoseconds it ran, so the
// host can see the SM clock the probe actually got.
__device__ __forceinline__ void report_clock(float* sink, long long c0, uint64_t t0) {
  if (sink != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    sink[0] = float(clock64() - c0);
    sink[1] = float(gtimer() - t0);
  }
}

// Eight independent FMA chains per thread; no memory traffic besides the
// clock report.  The chains' result is stored only if it equals a sentinel
// the chains cannot reach (their values stay in (0, 1]), which keeps the
// compiler from removing the work.
__global__ void probe_kernel(int iters, float* sink, int pdl) {
  if (pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long c0 = clock64();
  const uint64_t t0 = gtimer();
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = 0.5f + 0.0625f * j + 1e-7f * threadIdx.x;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = fmaf(a[j], 0.999f, 0.0005f);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += a[j];
  if (s == -1.0f && sink != nullptr) sink[2] = s;
  report_clock(sink, c0, t0);
}

// Whole-SM variant: 1024 threads, 48 independent chains per thread.  The
// chains need about 64 registers per thread, i.e. the SM's whole register file
// for one CTA, and the launch also reserves most of the shared memory, so no
// other kernel's CTA can share the SM while one of these runs -- the
// footprint of a GEMM tile.
constexpr int kWideChains = 48;
__global__ void __launch_bounds__(1024, 1) probe_wide_kernel(int iters, float* sink, int pdl) {
  if (pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long c0 = clock64();
  const uint64_t t0 = gtimer();
  float a[kWideChains];
#pragma unroll
  for (int j = 0; j < kWideChains; ++j) a[j] = 0.25f + 0.01f * j + 1e-7f * threadIdx.x;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < kWideChains; ++j) a[j] = fmaf(a[j], 0.999f, 0.0005f);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kWideChains; ++j) s += a[j];
  if (s == -1.0f && sink != nullptr) sink[2] = s;
  report_clock(sink, c0, t0);
}

// 16-byte vectors of eight 16-bit words; a scalar loop covers the unaligned
// head and the tail.
__global__ void xor16_kernel(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, size_t n, uint32_t key2,
                             size_t head, size_t nvec) {
  const size_t tid = blockIdx.x * size_t(blockDim.x) + threadIdx.x;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  const uint4* vin = reinterpret_cast<const uint4*>(in + head);
  uint4* vout = reinterpret_cast<uint4*>(out + head);
  for (size_t v = tid; v < nvec; v += stride) {
    uint4 x = __ldcs(vin + v);
    x.x ^= key2;
    x.y ^= key2;
    x.z ^= key2;
    x.w ^= key2;
    __stcs(vout + v, x);
  }
  const uint16_t key = static_cast<uint16_t>(key2 & 0xFFFFu);
  const size_t tail0 = head + nvec * 8;
  for (size_t i = tid; i < head; i += stride) out[i] = in[i] ^ key;
  for (size_t i = tid; i < n - tail0; i += stride) out[tail0 + i] = in[tail0 + i] ^ key;
}

}  // namespace

cudaError_t workload_preload() {
  const void* fns[] = {reinterpret_cast<const void*>(&probe_kernel), reinterpret_cast<const void*>(&probe_wide_kernel),
                       reinterpret_cast<const void*>(&xor16_kernel)};
  for (const void* f : fns) {
    cudaFuncAttributes a;
    const cudaError_t e = cudaFuncGetAttributes(&a, f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hoc

namespace hoc {
namespace {

// Launch with programmatic dependent launch allowed when `pdl`: the probe
// kernel waits (griddepcontrol.wait) for the previous kernel on the stream to
// finish before its FMA work, so only the launch itself overlaps.
template <typename... Args>
cudaError_t probe_start(void (*kernel)(Args...), int ctas, int threads, size_t smem, cudaStream_t s, bool pdl,
                        Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace
}  // namespace hoc

extern "C" hocResult_t hoc_probe_launch(void* stream, int ctas, int threads, int iters, int flags, float* sink) {
  if (ctas < 1 || threads < 32 || threads > 1024 || (threads % 32) != 0 || iters < 0) return HOC_ERR_INVALID_ARG;
  if (flags & ~(HOC_PROBE_WHOLE_SM | HOC_PROBE_PDL)) return HOC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pdl = (flags & HOC_PROBE_PDL) != 0;
  if (!(flags & HOC_PROBE_WHOLE_SM))
    return hoc::probe_start(hoc::probe_kernel, ctas, threads, 0, s, pdl, iters, sink, int(pdl)) == cudaSuccess
               ? HOC_SUCCESS
               : HOC_ERR_CUDA;
  if (threads != 1024) return HOC_ERR_INVALID_ARG;
  int dev = 0, smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return HOC_ERR_CUDA;
  smem -= 1024;  // leave the per-CTA reservation headroom
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&hoc::probe_wide_kernel),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return HOC_ERR_CUDA;
  return hoc::probe_start(hoc::probe_wide_kernel, ctas, 1024, size_t(smem), s, pdl, iters, sink, int(pdl)) ==
                 cudaSuccess
             ? HOC_SUCCESS
             : HOC_ERR_CUDA;
}

extern "C" hocResult_t hoc_xor16_launch(void* stream, const uint16_t* in, uint16_t* out, size_t n, uint16_t key) {
  if (n == 0) return HOC_SUCCESS;
  if (in == nullptr || out == nullptr) return HOC_ERR_INVALID_ARG;
  const uintptr_t ai = reinterpret_cast<uintptr_t>(in), ao = reinterpret_cast<uintptr_t>(out);
  if ((ai & 1u) || (ao & 1u)) return HOC_ERR_INVALID_ARG;
  if (ai != ao && ai < ao + 2 * n && ao < ai + 2 * n) return HOC_ERR_INVALID_ARG;
  size_t head = 0, nvec = 0;
  if (((ai ^ ao) & 15u) == 0) {
    head = ((16 - (ai & 15u)) & 15u) / 2;
    if (head > n) head = n;
    nvec = (n - head) / 8;
  } else {
    head = n;  // no common alignment: every word through the scalar path
  }
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t scalar = head > 8 ? head : 8;
  size_t want = (nvec > scalar ? nvec : scalar) + 255;
  want /= 256;
  const size_t cap = size_t(sms) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  const uint32_t key2 = uint32_t(key) | (uint32_t(key) << 16);
  hoc::xor16_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n, key2, head, nvec);
  return cudaGetLastError() == cudaSuccess ? HOC_SUCCESS : HOC_ERR_CUDA;
}

extern "C" hocResult_t hoc_device_sm_count(int device, int* sms) {
  if (sms == nullptr) return HOC_ERR_INVALID_ARG;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    cudaGetLastError();
    return HOC_ERR_NO_DEVICE;
  }
  if (device < 0 || device >= n) return HOC_ERR_INVALID_ARG;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess ? HOC_SUCCESS
                                                                                             : HOC_ERR_CUDA;
}
