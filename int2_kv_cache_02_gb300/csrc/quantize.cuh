// INT2 (or INT4) quantisation and packing of one 32-token block of keys and values,
// shared by quantize_kv_kernel and the fused prefill kernel (kernel (2) of the
// news article on arXiv 2605.19660, 三).
//
// Keys: block-wise per-channel asymmetric INT2 -- every channel of every
// group of G consecutive tokens (G = 32 by default; 64 and 128 are the
// larger groups) has its own step and zero, which every 32-token record of
// the group carries; values:
// per-token INT2 ("OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
// 方法步骤详情 (2)(3); 前置知识, step Δ and zero z per block).  Per group:
// z = min, Δ = (max - min)/3, code = round-half-even((x - z)/Δ) clamped to
// [0, 3], every operation one IEEE fp32 rounding; Δ = 0 and codes 0 for a
// constant group; Δ and z stored as fp16 (round to nearest even).
#pragma once

#include "common.cuh"

namespace oscar {

// Largest code of a BITS-bit quantiser (3 for INT2, 15 for INT4).
template <int BITS>
constexpr float kMaxCode = (float)((1 << BITS) - 1);

template <int BITS>
__device__ __forceinline__ uint8_t quant_code(float x, float mn, float step, bool live) {
  if (!live) return 0;
  const float t = __fdiv_rn(__fsub_rn(x, mn), step);
  float r = rintf(t);
  r = fminf(fmaxf(r, 0.0f), kMaxCode<BITS>);
  return (uint8_t)r;
}

// The same code with the quotient formed as a * (1/step): the correctly
// rounded reciprocal times a is within ~2^-21 (relative) of the rounded
// quotient, ~2^-19 absolute for quotients up to 16, so both round to the
// same integer unless the quotient lies within 1e-5 of a half-integer,
// where the exact division decides.
template <int BITS>
__device__ __forceinline__ uint8_t quant_code_fast(float x, float mn, float step, float rstep,
                                                   bool live) {
  if (!live) return 0;
  const float q = __fsub_rn(x, mn) * rstep;
  if (fabsf(q - floorf(q) - 0.5f) < 1e-5f) return quant_code<BITS>(x, mn, step, live);
  return (uint8_t)fminf(fmaxf(rintf(q), 0.0f), kMaxCode<BITS>);
}

// The fast code without a branch: c = round-half-even(q), q = (x - mn) /
// step formed as (x - mn) * (1/step) (0 for a constant group, whose step and
// reciprocal are 0 and x == mn).  dist keeps the largest |q - c| seen; above
// kNearHalf, some quotient may lie within 1e-5 of a half-integer (the case
// quant_code_fast hands to the exact division), and the caller redoes the
// warp's codes with quant_code_fast, so the codes are always those of
// quant_code_fast.  (|q - c| is exact and 0.5 - |q - c| equals
// |q - floor(q) - 0.5| wherever either is below 0.25; the threshold keeps a
// margin of 1e-5 over that test, so a redo may happen needlessly, never be
// missed.)
template <int BITS>
__device__ __forceinline__ uint8_t quant_code_nb(float x, float mn, float rstep, float& dist) {
  const float q = __fsub_rn(x, mn) * rstep;
  const int c = __float2int_rn(q);
  dist = fmaxf(dist, fabsf(q - (float)c));
  return (uint8_t)min(c, (1 << BITS) - 1);
}
constexpr float kNearHalf = 0.5f - 2e-5f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t u) {
  return __uint_as_float(((uint32_t)u) << 16);
}

// Row length of the byte-per-code tiles: 4 bytes of padding put the rows a
// packing warp reads (4 tokens, 128 bytes apart) on different banks.
constexpr int kCodeRow = kD + 4;

// Step and zero of one key channel over a group of N tokens (thread c =
// channel c of the rows of kt, rotated and scaled keys as bf16).
struct KeyParams {
  float mn, step, rstep;
  bool live;
};
template <int N, int BITS>
__device__ __forceinline__ KeyParams key_params(const uint16_t (*kt)[kD]) {
  const int c = threadIdx.x;
  float mn = bf16_bits_to_float(kt[0][c]), mx = mn;
#pragma unroll 8
  for (int t = 1; t < N; ++t) {
    const float x = bf16_bits_to_float(kt[t][c]);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
  KeyParams p;
  p.live = mx > mn;
  p.mn = mn;
  p.step = p.live ? __fdiv_rn(__fsub_rn(mx, mn), kMaxCode<BITS>) : 0.0f;
  p.rstep = p.live ? __frcp_rn(p.step) : 0.0f;
  return p;
}

// Called by all 128 threads of the CTA after a __syncthreads that follows
// the staging of kt (rotated, scaled keys as bf16) and vt (values as bf16)
// for the 32 tokens of one block; kp: this thread's key channel parameters
// over the block's group; norms: the block's 32 key norms (global or shared
// memory).  Writes the block record at rec (layout in oscar.h for BITS).
template <int BITS>
__device__ __forceinline__ void quantize_block(const uint16_t (*kt)[kD],
                                               const uint16_t (&vt)[kG][kD],
                                               uint8_t (&kc)[kG][kCodeRow],
                                               uint8_t (&vc)[kG][kCodeRow],
                                               const __half* norms, uint8_t* rec,
                                               const KeyParams& kp) {
  const int tid = threadIdx.x;
  using RL = Rec<BITS>;
  uint32_t* k_codes = reinterpret_cast<uint32_t*>(rec + RL::KC);
  uint32_t* v_codes = reinterpret_cast<uint32_t*>(rec + RL::VC);
  __half* k_scale = reinterpret_cast<__half*>(rec + RL::KS);
  __half* k_zero = reinterpret_cast<__half*>(rec + RL::KZ);
  __half* k_norm_out = reinterpret_cast<__half*>(rec + RL::KN);
  __half* v_scale = reinterpret_cast<__half*>(rec + RL::VS);
  __half* v_zero = reinterpret_cast<__half*>(rec + RL::VZ);

  // Keys: thread = channel, with its group's parameters.  Codes without a
  // branch; the rare quotients near a half-integer are redone exactly.
  {
    const int c = tid;
    float dist = 0.0f;
#pragma unroll 8
    for (int t = 0; t < kG; ++t)
      kc[t][c] = quant_code_nb<BITS>(bf16_bits_to_float(kt[t][c]), kp.mn, kp.rstep, dist);
    if (__any_sync(0xffffffffu, dist > kNearHalf)) {
      for (int t = 0; t < kG; ++t)
        kc[t][c] = quant_code_fast<BITS>(bf16_bits_to_float(kt[t][c]), kp.mn, kp.step, kp.rstep,
                                         kp.live);
    }
    k_scale[c] = __float2half_rn(kp.step);
    k_zero[c] = __float2half_rn(kp.mn);
  }

  // Values: warp w handles tokens 8w..8w+7, lane holds channels 4l..4l+3.
  {
    const int w = tid >> 5, lane = tid & 31;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int t = 8 * w + i;
      // the lane's 4 channels in one 8-byte load (the warp reads 256
      // contiguous bytes)
      const uint2 raw = reinterpret_cast<const uint2*>(&vt[t][0])[lane];
      const float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                          __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
      float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, m));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      }
      const bool live = mx > mn;
      const float step = live ? __fdiv_rn(__fsub_rn(mx, mn), kMaxCode<BITS>) : 0.0f;
      const float rstep = live ? __frcp_rn(step) : 0.0f;
      float dist = 0.0f;
      uint8_t cv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) cv[j] = quant_code_nb<BITS>(x[j], mn, rstep, dist);
      if (__any_sync(0xffffffffu, dist > kNearHalf)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) cv[j] = quant_code_fast<BITS>(x[j], mn, step, rstep, live);
      }
      // the lane's 4 codes as one 32-bit store (channels 4 lane .. 4 lane + 3)
      *reinterpret_cast<uint32_t*>(&vc[t][4 * lane]) =
          (uint32_t)cv[0] | ((uint32_t)cv[1] << 8) | ((uint32_t)cv[2] << 16) |
          ((uint32_t)cv[3] << 24);
      if (lane == 0) {
        v_scale[tok_slot(t)] = __float2half_rn(step);
        v_zero[tok_slot(t)] = __float2half_rn(mn);
      }
    }
  }
  if (tid < kG) k_norm_out[tok_slot(tid)] = norms[tid];
  __syncthreads();

  if constexpr (BITS == 2) {
    // Pack keys: word (t, w) = channels 16w..16w+15 of token t; channel 16w+j
    // at bit 2*(j/2) + 16*(j%2).
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int wi = tid + 128 * r;
      const int t = wi >> 3, w = wi & 7;
      const uint8_t* src = &kc[t][16 * w];
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) word |= (uint32_t)src[j] << (2 * (j >> 1) + 16 * (j & 1));
      k_codes[t * 8 + w] = word;
    }
    // Pack values: word 128*kh + 4*lane + 2p + hh, lane = 4g + t4; low half
    // token 16kh + 2*t4 + 8p, high half the next token; slot k = channel
    // g + 8*(8hh+k).
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int wi = tid + 128 * r;
      const int kh = wi >> 7, lane = (wi >> 2) & 31, p = (wi >> 1) & 1, hh = wi & 1;
      const int g = lane >> 2, t4 = lane & 3;
      const int tok = 16 * kh + 2 * t4 + 8 * p;
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int ch = g + 8 * (8 * hh + k);
        word |= (uint32_t)vc[tok][ch] << (2 * k);
        word |= (uint32_t)vc[tok + 1][ch] << (16 + 2 * k);
      }
      v_codes[wi] = word;
    }
  } else {
    // INT4 keys: word (t, w) = channels 8w..8w+7 of token t; channel 8w+j at
    // bit 4*(j/2) + 16*(j%2).
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int wi = tid + 128 * r;
      const int t = wi >> 4, w = wi & 15;
      const uint8_t* src = &kc[t][8 * w];
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) word |= (uint32_t)src[j] << (4 * (j >> 1) + 16 * (j & 1));
      k_codes[t * 16 + w] = word;
    }
    // INT4 values: word 256*kh + 128p + 4*lane + hh, lane = 4g + t4; low
    // half token 16kh + 2*t4 + 8p, high half the next token; slot k (4 bits)
    // = channel g + 8*(4hh+k).
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int wi = tid + 128 * r;
      const int kh = wi >> 8, p = (wi >> 7) & 1, lane = (wi >> 2) & 31, hh = wi & 3;
      const int g = lane >> 2, t4 = lane & 3;
      const int tok = 16 * kh + 2 * t4 + 8 * p;
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int ch = g + 8 * (4 * hh + k);
        word |= (uint32_t)vc[tok][ch] << (4 * k);
        word |= (uint32_t)vc[tok + 1][ch] << (16 + 4 * k);
      }
      v_codes[wi] = word;
    }
  }
}

}  // namespace oscar
