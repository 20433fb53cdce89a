// Two binary32 lanes in one 64-bit register: the packed add of sm_100-class
// GPUs (IEEE, round to nearest even, no flush to zero) gives the same bits as
// two scalar __fadd_rn.  Only sums are packed here; a packed multiply feeding
// a packed add is fused by the code generator into one multiply-add (one
// rounding), so products stay scalar wherever their own rounding matters.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

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

// The two bf16 values of a 32-bit word (element 2w in the low half), widened
// exactly to binary32 lanes; and back, each lane rounded once to bf16
// (nearest even).
__device__ __forceinline__ unsigned long long bf16_pair(uint32_t w) { return pack_f32x2(w << 16, w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16_narrow_pair(unsigned long long a) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(lo_f32(a)))) |
         (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(hi_f32(a)))) << 16);
}

}  // namespace hoc
