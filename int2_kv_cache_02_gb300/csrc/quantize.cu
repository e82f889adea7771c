// INT2 quantisation and packing of keys and values (kernel (2) of the news
// article on arXiv 2605.19660, 三).
//
// Keys: block-wise per-channel asymmetric INT2 -- every channel of every
// block of G = 32 consecutive tokens has its own step and zero; values:
// per-token INT2 ("OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
// 方法步骤详情 (2)(3); 前置知识, step Δ and zero z per block).  Per group:
// z = min, Δ = (max - min)/3, code = round-half-even((x - z)/Δ) clamped to
// [0, 3], every operation one IEEE fp32 rounding; Δ = 0 and codes 0 for a
// constant group; Δ and z stored as fp16 (round to nearest even).
//
// One CTA of 128 threads per (b, h, block of 32 tokens): the 32x128 key and
// value tiles are staged in shared memory, codes computed one byte each, then
// packed 16 per word into the block record declared in oscar.h.
#include "common.cuh"
#include "launch.h"

namespace oscar {

__device__ __forceinline__ uint8_t quant_code(float x, float mn, float step, bool live) {
  if (!live) return 0;
  const float t = __fdiv_rn(__fsub_rn(x, mn), step);
  float r = rintf(t);
  r = fminf(fmaxf(r, 0.0f), 3.0f);
  return (uint8_t)r;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t u) {
  return __uint_as_float(((uint32_t)u) << 16);
}

__global__ void __launch_bounds__(128) quantize_kv_kernel(
    const uint16_t* __restrict__ k_hat, const __half* __restrict__ k_norm,
    const uint16_t* __restrict__ v, int src_T, int Hkv, int T_cap, int p0,
    uint8_t* __restrict__ packed) {
  __shared__ __align__(16) uint16_t kt[kG][kD];
  __shared__ __align__(16) uint16_t vt[kG][kD];
  __shared__ __align__(16) uint8_t kc[kG][kD];
  __shared__ __align__(16) uint8_t vc[kG][kD];

  const int tid = threadIdx.x;
  const int blk = blockIdx.x;
  const long long row = (long long)blockIdx.z * Hkv + blockIdx.y;
  const long long src_tok = row * src_T + (long long)blk * kG;

  // Stage both tiles: 32 tokens x 256 B each, 16 B per thread per step.
  {
    const uint4* ks = reinterpret_cast<const uint4*>(k_hat + src_tok * kD);
    const uint4* vs = reinterpret_cast<const uint4*>(v + src_tok * kD);
    uint4* kd = reinterpret_cast<uint4*>(&kt[0][0]);
    uint4* vd = reinterpret_cast<uint4*>(&vt[0][0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kd[tid + 128 * i] = ks[tid + 128 * i];
      vd[tid + 128 * i] = vs[tid + 128 * i];
    }
  }
  __syncthreads();

  const long long pblk = (long long)p0 / kG + blk;   // packed block index in the row
  uint8_t* rec = packed + (row * (T_cap / kG) + pblk) * kBlkBytes;
  uint32_t* k_codes = reinterpret_cast<uint32_t*>(rec + kRecKC);
  uint32_t* v_codes = reinterpret_cast<uint32_t*>(rec + kRecVC);
  __half* k_scale = reinterpret_cast<__half*>(rec + kRecKS);
  __half* k_zero = reinterpret_cast<__half*>(rec + kRecKZ);
  __half* k_norm_out = reinterpret_cast<__half*>(rec + kRecKN);
  __half* v_scale = reinterpret_cast<__half*>(rec + kRecVS);
  __half* v_zero = reinterpret_cast<__half*>(rec + kRecVZ);

  // Keys: thread = channel, group = the 32 tokens of the block.
  {
    const int c = tid;
    float mn = bf16_bits_to_float(kt[0][c]), mx = mn;
#pragma unroll 8
    for (int t = 1; t < kG; ++t) {
      const float x = bf16_bits_to_float(kt[t][c]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    const bool live = mx > mn;
    const float step = live ? __fdiv_rn(__fsub_rn(mx, mn), 3.0f) : 0.0f;
#pragma unroll 8
    for (int t = 0; t < kG; ++t) kc[t][c] = quant_code(bf16_bits_to_float(kt[t][c]), mn, step, live);
    k_scale[c] = __float2half_rn(step);
    k_zero[c] = __float2half_rn(mn);
  }

  // Values: warp w handles tokens 8w..8w+7, lane holds channels 4l..4l+3.
  {
    const int w = tid >> 5, lane = tid & 31;
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int t = 8 * w + i;
      float x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = bf16_bits_to_float(vt[t][4 * lane + j]);
      float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, m));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      }
      const bool live = mx > mn;
      const float step = live ? __fdiv_rn(__fsub_rn(mx, mn), 3.0f) : 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) vc[t][4 * lane + j] = quant_code(x[j], mn, step, live);
      if (lane == 0) {
        v_scale[tok_slot(t)] = __float2half_rn(step);
        v_zero[tok_slot(t)] = __float2half_rn(mn);
      }
    }
  }
  if (tid < kG) k_norm_out[tok_slot(tid)] = k_norm[src_tok + tid];
  __syncthreads();

  // Pack keys: word (t, w) = channels 16w..16w+15 of token t; channel 16w+j at
  // bit 2*(j/2) + 16*(j%2).
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
  // Pack values: word 128*kh + 4*lane + 2p + hh, lane = 4g + t4; low half token
  // 16kh + 2*t4 + 8p, high half the next token; slot k = channel g + 8*(8hh+k).
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
}

cudaError_t launch_quantize_kv(const uint16_t* k_hat, const __half* k_norm, const uint16_t* v,
                               int src_T, int n_tok, int B, int Hkv, int T_cap, int p0,
                               uint8_t* packed, cudaStream_t s) {
  dim3 grid(n_tok / kG, Hkv, B);
  quantize_kv_kernel<<<grid, 128, 0, s>>>(k_hat, k_norm, v, src_T, Hkv, T_cap, p0, packed);
  return cudaGetLastError();
}

}  // namespace oscar
