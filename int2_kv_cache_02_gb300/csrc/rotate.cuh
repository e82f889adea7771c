// Per-token Canalized Rotation and Omni-Token Scaling of one 128-vector,
// shared by the rotate kernels and the group kernels ("OScaR: The Occam's
// Razor for Extreme KV Cache Quantization in LLMs and Beyond" reading notes,
// II. Step One and Step Two; news article on arXiv 2605.19660, 三: FHT and
// scaling in one kernel, hardware rsqrt).  Two layouts of the vector:
//  * one warp per vector, lane l holding elements 4l..4l+3 (float[4]);
//  * the quarter layout, four lanes per vector (lanes l, l ^ 8, l ^ 16,
//    l ^ 24), lane l holding elements 32Q..32Q+31 with Q = l >> 3, so a warp
//    works 8 vectors at once (float[32]).
// Both apply the same butterflies in the same order and sum the squares in
// the same order, so they give the same bits.
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
    // the same single rounding as the subtraction or the addition (two
    // elements per packed fma)
    const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int r = 0; r < 4; r += 2) {
      const float y0 = __shfl_xor_sync(0xffffffffu, x[r], m);
      const float y1 = __shfl_xor_sync(0xffffffffu, x[r + 1], m);
      const float2 v = fma2(make_float2(sg, sg), make_float2(x[r], x[r + 1]), make_float2(y0, y1));
      x[r] = v.x;
      x[r + 1] = v.y;
    }
  }
}

// The same transform in the quarter layout: index bits 0-4 butterflied in
// registers (a + b and a - b, the roundings of the lane pairs above), bits 5
// and 6 across lanes xor 8 and xor 16.  Elements 2i, 2i + 1 travel as one
// packed pair from bit 1 on: a packed operation rounds each half as the
// scalar one would, so the results are those of the scalar butterflies.
__device__ __forceinline__ void fht128(float (&x)[32], int lane) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float a = x[e], b = x[e + 1];
    x[e] = a + b;
    x[e + 1] = a - b;
  }
#pragma unroll
  for (int h = 2; h < 32; h <<= 1)
#pragma unroll
    for (int e = 0; e < 32; e += 2)
      if (!(e & h)) {
        const float2 a = make_float2(x[e], x[e + 1]), b = make_float2(x[e + h], x[e + h + 1]);
        const float2 s = add2(a, b), d = sub2(a, b);
        x[e] = s.x;
        x[e + 1] = s.y;
        x[e + h] = d.x;
        x[e + h + 1] = d.y;
      }
#pragma unroll
  for (int m = 8; m < 32; m <<= 1) {
    const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float y0 = __shfl_xor_sync(0xffffffffu, x[e], m);
      const float y1 = __shfl_xor_sync(0xffffffffu, x[e + 1], m);
      const float2 r = fma2(make_float2(sg, sg), make_float2(x[e], x[e + 1]), make_float2(y0, y1));
      x[e] = r.x;
      x[e + 1] = r.y;
    }
  }
}

// Sum over the warp's lanes, pairing lanes xor 1 first and xor 16 last: every
// lane ends with the same value, and the quarter layout below forms the same
// sum with the first three pairings in registers.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Sum of squares of four elements, one rounding order for every kernel.
__device__ __forceinline__ float sq4(float a, float b, float c, float d) {
  return fmaf(d, d, fmaf(c, c, fmaf(b, b, a * a)));
}

// Sum of squares of the vector, in either layout: per group of 4 elements
// sq4, then the groups paired as warp_sum pairs the lanes of the one-warp
// layout (groups 8Q..8Q+7 of a quarter in registers, then lanes xor 8, 16).
__device__ __forceinline__ float sum_sq(const float (&x)[4]) {
  return warp_sum(sq4(x[0], x[1], x[2], x[3]));
}
__device__ __forceinline__ float sum_sq(const float (&x)[32]) {
  float p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = sq4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int i = 0; i < 8; i += 2 * h) p[i] += p[i + h];
  float s = p[0];
  s += __shfl_xor_sync(0xffffffffu, s, 8);
  s += __shfl_xor_sync(0xffffffffu, s, 16);
  return s;
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
    s += warp_sum(sq4(a, b, c, d));
  }
  return s;
}
// The same sum in the quarter layout (lane: 32 elements of its quarter of
// each head's key).
__device__ __forceinline__ float all_heads_sq_q(const uint16_t* k0, long long head_stride, int Hkv,
                                               int lane) {
  float s = 0.0f;
  for (int h = 0; h < Hkv; ++h) {
    const uint4* src = reinterpret_cast<const uint4*>(k0 + h * head_stride) + 4 * (lane >> 3);
    float x[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = src[i];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[8 * i + 2 * j] = bf16_lo(w[j]);
        x[8 * i + 2 * j + 1] = bf16_hi(w[j]);
      }
    }
    s += sum_sq(x);
  }
  return s;
}

// x[r] *= f for every element, two at a time (each product rounded as the
// scalar one).
template <int N>
__device__ __forceinline__ void scale_all(float (&x)[N], float f) {
#pragma unroll
  for (int r = 0; r < N; r += 2) {
    const float2 p = mul2(make_float2(x[r], x[r + 1]), make_float2(f, f));
    x[r] = p.x;
    x[r + 1] = p.y;
  }
}

// Rotates (unless OSCAR_NO_ROTATE) and scales (unless OSCAR_NO_SCALE) the key
// held in x to the norm ks.target; returns the stored norm n / target, with n
// the key's own norm or, with OSCAR_NORM_ALL_HEADS, the norm of the token's
// keys over all heads, whose raw sum of squares the caller passes in s_all.
// Unscaled keys store 1; a zero key (zero norm) keeps k_hat = 0 and stores 0.
// PLAIN: the method itself (no flags, unit target) fixed at compile time, so
// the per-token tests of the variants fold away.  N: elements per lane (4:
// one warp per vector; 32: the quarter layout).
template <bool PLAIN = false, int N>
__device__ __forceinline__ float rotate_scale_key(float (&x)[N], int lane, KeyScale ks,
                                                  float s_all = 0.0f) {
  if constexpr (PLAIN) {
    ks.flags = 0u;
    ks.target = 1.0f;
  }
  const bool rot = !(ks.flags & OSCAR_NO_ROTATE);
  if (rot) fht128(x, lane);
  if (ks.flags & OSCAR_NO_SCALE) {
    scale_all(x, rot ? kInvSqrtD : 1.0f);
    return 1.0f;
  }
  const float s = (ks.flags & OSCAR_NORM_ALL_HEADS) ? (rot ? 128.0f * s_all : s_all) : sum_sq(x);
  if (s > 0.0f) {
    const bool unit = ks.target == 1.0f;   // the method's target: no extra rounding
    scale_all(x, unit ? rsqrtf(s) : rsqrtf(s) * ks.target);
    const float n = sqrtf(s) * (rot ? kInvSqrtD : 1.0f);
    return unit ? n : n / ks.target;
  }
#pragma unroll
  for (int r = 0; r < N; ++r) x[r] = 0.0f;
  return 0.0f;
}

// Two floats as bf16 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}
// The warp's vector as 4 bf16, packed in a uint2.
__device__ __forceinline__ uint2 pack_bf16x4(const float (&x)[4]) {
  return make_uint2(bf16x2_bits(x[0], x[1]), bf16x2_bits(x[2], x[3]));
}

}  // namespace oscar

namespace oscar {
// The method's own scaling (no ablation or scope flag, unit target): the
// kernels that scale keys are instantiated for it separately.
inline bool plain_scale(const KeyScale& ks) { return ks.flags == 0u && ks.target == 1.0f; }
}  // namespace oscar
