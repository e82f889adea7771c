// Per-token Canalized Rotation and Omni-Token Scaling of one 128-vector held
// by a warp (lane l: elements 4l..4l+3), shared by the rotate kernels and the
// fused prefill ("OScaR: The Occam's Razor for Extreme KV Cache Quantization
// in LLMs and Beyond" reading notes, II. Step One and Step Two; news article
// on arXiv 2605.19660, 三: FHT and scaling in one kernel, hardware rsqrt).
#pragma once

#include "common.cuh"

namespace oscar {

constexpr float kInvSqrtD = 0.088388347648318440550f;  // 1/sqrt(128)

// Unnormalised natural-order Walsh-Hadamard transform of the warp's vector:
// index bits 0-1 butterflied in registers, bits 2-6 across lanes.
__device__ __forceinline__ void fht128(float (&x)[4], int lane) {
  float a = x[0] + x[1], b = x[0] - x[1], c = x[2] + x[3], d = x[2] - x[3];
  x[0] = a + c; x[2] = a - c; x[1] = b + d; x[3] = b - d;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float y = __shfl_xor_sync(0xffffffffu, x[r], m);
      x[r] = upper ? (y - x[r]) : (x[r] + y);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Rotates (unless OSCAR_NO_ROTATE) and scales to unit norm (unless
// OSCAR_NO_SCALE) the key held in x; returns its norm (1 when not scaled,
// 0 for a zero key, whose k_hat is then 0).
__device__ __forceinline__ float rotate_scale_key(float (&x)[4], int lane, unsigned flags) {
  const bool rot = !(flags & OSCAR_NO_ROTATE);
  if (rot) fht128(x, lane);
  if (flags & OSCAR_NO_SCALE) {
    const float f = rot ? kInvSqrtD : 1.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] *= f;
    return 1.0f;
  }
  const float s = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
  if (s > 0.0f) {
    const float rs = rsqrtf(s);
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] *= rs;
    return sqrtf(s) * (rot ? kInvSqrtD : 1.0f);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) x[r] = 0.0f;
  return 0.0f;
}

// The warp's vector as 4 bf16 (round to nearest even), packed in a uint2.
__device__ __forceinline__ uint2 pack_bf16x4(const float (&x)[4]) {
  __nv_bfloat162 p0 = __floats2bfloat162_rn(x[0], x[1]);
  __nv_bfloat162 p1 = __floats2bfloat162_rn(x[2], x[3]);
  uint2 o;
  o.x = *reinterpret_cast<uint32_t*>(&p0);
  o.y = *reinterpret_cast<uint32_t*>(&p1);
  return o;
}

}  // namespace oscar
