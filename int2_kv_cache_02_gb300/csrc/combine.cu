// Log-sum-exp combine of split-K partials (flash-decoding): for every
// (sequence, query head), m* = max_s m_s, out = sum_s 2^(m_s - m*) o_s /
// sum_s 2^(m_s - m*) l_s (scores are kept in the log2 domain).  Splits that
// saw no token carry m = -inf and drop out; an all-empty row gives zeros.
#include "common.cuh"
#include "launch.h"

namespace oscar {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws,
                                                      float* __restrict__ out, int n_rows,
                                                      int n_parts) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const float* r0 = ws + row * n_parts * kRecFloats;
  float M = -INFINITY;
  for (int s = lane; s < n_parts; s += 32) M = fmaxf(M, r0[(long long)s * kRecFloats]);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  float L = 0.0f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int s = 0; s < n_parts; ++s) {
      const float* r = r0 + (long long)s * kRecFloats;
      const float ms = r[0];
      if (ms == -INFINITY) continue;
      const float a = fast_exp2(ms - M);
      L += a * r[1];
      const float4 x = reinterpret_cast<const float4*>(r + 4)[lane];
      o.x += a * x.x; o.y += a * x.y; o.z += a * x.z; o.w += a * x.w;
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  reinterpret_cast<float4*>(out + row * kD)[lane] =
      make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
}

cudaError_t launch_combine(const float* ws, float* out, int n_rows, int n_parts, cudaStream_t s) {
  combine_kernel<<<(n_rows + 7) / 8, 256, 0, s>>>(ws, out, n_rows, n_parts);
  return cudaGetLastError();
}

}  // namespace oscar
