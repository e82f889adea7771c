// Per-token Canalized Rotation and Omni-Token Scaling of one 128-vector held
// by a warp (lane l: elements 4l..4l+3), shared by the rotate kernels and the
// fused prefill ("OScaR: The Occam's Razor for Extreme KV Cache Quantization
// in LLMs and Beyond" reading notes, II. Step One and Step Two; news article
// on arXiv 2605.19660, 三: FHT and scaling in one kernel, hardware rsqrt).
#pragma once

#include "common.cuh"
#include "launch.h"

namespace oscar {

constexpr float kInvSqrtD = 0.088388347648318440550f;  // 1/sqrt(128)

// Unnormalised natural-order Walsh-Hadamard transform of the warp's vector:
// index bits 0-1 butterflied in registers, bits 2-6 across lanes.
__device__ __forceinline__ void fht128(float (&x)[4], int lane) {
  float a = x[0] + x[1], b = x[0] - x[1], c = x[2] + x[3], d = x[2] - x[3];
  x[0] = a + c; x[2] = a - c; x[1] = b + d; x[3] = b - d;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    // upper lanes take y - x, lower lanes x + y: one fma with a +-1 factor,
    // the same single rounding as the subtraction or the addition
    const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float y = __shfl_xor_sync(0xffffffffu, x[r], m);
      x[r] = fmaf(sg, x[r], y);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Sum of squares of one token's raw keys over all Hkv heads, for the
// all-heads norm: head h's key (4 elements per lane) at k0 + h * head_stride;
// each head's sum is a warp sum of the lanes' partials, added in head order,
// so every kernel that scales keys forms the same value.  By orthogonality of
// H the rotated keys have 128 times this sum (exact in fp32).
__device__ __forceinline__ float all_heads_sq(const uint16_t* k0, long long head_stride, int Hkv,
                                             int lane) {
  float s = 0.0f;
  for (int h = 0; h < Hkv; ++h) {
    const uint2 raw = reinterpret_cast<const uint2*>(k0 + h * head_stride)[lane];
    const float a = bf16_lo(raw.x), b = bf16_hi(raw.x), c = bf16_lo(raw.y), d = bf16_hi(raw.y);
    s += warp_sum(fmaf(d, d, fmaf(c, c, fmaf(b, b, a * a))));
  }
  return s;
}

// Rotates (unless OSCAR_NO_ROTATE) and scales (unless OSCAR_NO_SCALE) the key
// held in x to the norm ks.target; returns the stored norm n / target, with n
// the key's own norm or, with OSCAR_NORM_ALL_HEADS, the norm of the token's
// keys over all heads, whose raw sum of squares the caller passes in s_all.
// Unscaled keys store 1; a zero key (zero norm) keeps k_hat = 0 and stores 0.
// PLAIN: the method itself (no flags, unit target) fixed at compile time, so
// the per-token tests of the variants fold away.
template <bool PLAIN = false>
__device__ __forceinline__ float rotate_scale_key(float (&x)[4], int lane, KeyScale ks,
                                                  float s_all = 0.0f) {
  if constexpr (PLAIN) {
    ks.flags = 0u;
    ks.target = 1.0f;
  }
  const bool rot = !(ks.flags & OSCAR_NO_ROTATE);
  if (rot) fht128(x, lane);
  if (ks.flags & OSCAR_NO_SCALE) {
    const float f = rot ? kInvSqrtD : 1.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] *= f;
    return 1.0f;
  }
  const float s = (ks.flags & OSCAR_NORM_ALL_HEADS)
                      ? (rot ? 128.0f * s_all : s_all)
                      : warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
  if (s > 0.0f) {
    const bool unit = ks.target == 1.0f;   // the method's target: no extra rounding
    const float f = unit ? rsqrtf(s) : rsqrtf(s) * ks.target;
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] *= f;
    const float n = sqrtf(s) * (rot ? kInvSqrtD : 1.0f);
    return unit ? n : n / ks.target;
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

namespace oscar {
// The method's own scaling (no ablation or scope flag, unit target): the
// kernels that scale keys are instantiated for it separately.
inline bool plain_scale(const KeyScale& ks) { return ks.flags == 0u && ks.target == 1.0f; }
}  // namespace oscar
