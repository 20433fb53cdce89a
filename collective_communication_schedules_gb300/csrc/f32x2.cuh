// Two binary32 lanes in one 64-bit register: the packed add of sm_100-class
// GPUs (IEEE, round to nearest even, no flush to zero) gives the same bits as
// two scalar __fadd_rn.  Only sums are packed here; a packed multiply feeding
// a packed add is fused by the code generator into one multiply-add (one
// rounding), so products stay scalar wherever their own rounding matters.
#pragma once

#include <cstdint>

namespace hoc {

__device__ __forceinline__ unsigned long long pack_f32x2(uint32_t lo, uint32_t hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  return pack_f32x2(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ unsigned long long add_f32x2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float lo_f32(unsigned long long v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi_f32(unsigned long long v) { return __uint_as_float(uint32_t(v >> 32)); }

}  // namespace hoc
