// device_util.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_val(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// float -> bf16 bits, round to nearest even (inputs here are finite).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// Record the first device-side error in the sticky word (later ones are dropped).
__device__ __forceinline__ void record_error(int32_t* err, int code) {
  atomicCAS(err, 0, code);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over aligned groups of `width` lanes (width a power of two <= 32).
__device__ __forceinline__ float group_sum(float v, int width) {
  for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum of the 32 codes of a uint4 chunk (8 codes per word, low nibble first)
// weighted by xs[0..31]:  sum_i q_i * xs[i], fp32 FMA chain.
__device__ __forceinline__ float dot_chunk32(uint4 w, const float* __restrict__ xs) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      acc = fmaf((float)((ws[j] >> (4 * n)) & 0xFu), xs[8 * j + n], acc);
    }
  }
  return acc;
}

// The same for 32 int8 codes: word j of a, then of b, holds codes 4j..4j+3
// (8 bits each, low byte first).
__device__ __forceinline__ float dot_chunk32_q8(uint4 a, uint4 b, const float* __restrict__ xs) {
  const uint32_t ws[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      acc = fmaf((float)((ws[j] >> (8 * n)) & 0xFFu), xs[4 * j + n], acc);
    }
  }
  return acc;
}

// silu(a) = a / (1 + e^-a); the fast division's error (a few ulp of fp32) is
// far below the bf16 or fp32 rounding of what consumes it.
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

}  // namespace moe
