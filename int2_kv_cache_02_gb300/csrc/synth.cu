// Seeded synthetic inputs on the GPU (see include/oscar_synth.h for the
// definition).  Not part of the method: it only draws numbers, bit for bit
// the same as int2_kv_cache_02_gb300/synth.py.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/oscar_synth.h"

namespace {

__device__ __forceinline__ uint64_t splitmix_at(uint64_t seed, uint64_t n) {
  uint64_t z = seed + (n + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float normal_at(uint64_t seed, uint64_t e) {
  long long acc = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t r = splitmix_at(seed, 3ull * e + j);
    acc += (long long)(r & 0xFFFF) + (long long)((r >> 16) & 0xFFFF) +
           (long long)((r >> 32) & 0xFFFF) + (long long)(r >> 48);
  }
  acc -= 6 * 65536;
  return __fmul_rn((float)acc, 1.52587890625e-05f);  // exact: |acc| < 2^20, times 2^-16
}

__global__ void synth_kernel(uint16_t* __restrict__ out, int nB, int H, int b0, int out_T, int t0,
                             int n_t, uint64_t seed, const float* __restrict__ chan,
                             const float* __restrict__ tok) {
  const long long n_pairs = (long long)nB * H * n_t * 64;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_pairs;
       i += (long long)gridDim.x * blockDim.x) {
    const int c2 = (int)(i & 63);
    const long long r = i >> 6;                 // (b*H + h)*n_t + t
    const int t = (int)(r % n_t);
    const long long bh = r / n_t;
    const int h = (int)(bh % H);
    const int b = (int)(bh / H);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = 2 * c2 + e;
      const uint64_t ctr =
          ((((uint64_t)(b0 + b)) * (uint64_t)H + (uint64_t)h) * (1ull << 32) + (uint64_t)(t0 + t)) *
              128ull + (uint64_t)c;
      float x = normal_at(seed, ctr);
      if (chan) x = __fmul_rn(x, chan[c]);
      if (tok) x = __fmul_rn(x, tok[(long long)b * n_t + t]);
      const __nv_bfloat16 v = __float2bfloat16_rn(x);
      packed |= (uint32_t)(*reinterpret_cast<const uint16_t*>(&v)) << (16 * e);
    }
    reinterpret_cast<uint32_t*>(out + (bh * out_T + t) * 128)[c2] = packed;
  }
}

}  // namespace

extern "C" int oscar_synth_bf16(uint16_t* out, int nB, int H, int b0, int out_T, int t0, int n_t,
                                unsigned long long seed, const float* chan_factor,
                                const float* tok_factor, void* stream) {
  if (!out || nB <= 0 || H <= 0 || b0 < 0 || n_t <= 0 || out_T < n_t || t0 < 0) return 1;
  if (reinterpret_cast<uintptr_t>(out) & 15u) return 1;
  const long long n_pairs = (long long)nB * H * n_t * 64;
  long long blocks = (n_pairs + 255) / 256;
  if (blocks > 152LL * 64) blocks = 152LL * 64;
  synth_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      out, nB, H, b0, out_T, t0, n_t, seed, chan_factor, tok_factor);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
