// Log-sum-exp combine of split-K partials (flash-decoding): for every
// (sequence, query head), m* = max_s m_s, out = sum_s 2^(m_s - m*) o_s /
// sum_s 2^(m_s - m*) l_s (scores are kept in the log2 domain).  Splits that
// saw no token carry m = -inf and drop out; an all-empty row gives zeros.
//
// One CTA of kCW warps per (sequence, query head).  Warp w folds partials
// w, w + kCW, w + 2 kCW, ...: each lane first takes the weight of one of
// them, then the warp walks them with the weights broadcast by shuffles, so
// the loads of successive partials do not wait on one another.  Lane l holds
// channels 4 l .. 4 l + 3; shared memory adds the warps' results.
#include "common.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int kCW = 4;  // warps per CTA

__global__ void __launch_bounds__(kCW * 32) combine_kernel(const float* __restrict__ ws,
                                                           float* __restrict__ out, int n_parts) {
  __shared__ float sm_m[kCW], sm_l[kCW];
  __shared__ __align__(16) float sm_o[kCW][kD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = blockIdx.x;
  const float* r0 = ws + row * n_parts * kRecFloats;

  float M = -INFINITY;
  for (int s = threadIdx.x; s < n_parts; s += kCW * 32) M = fmaxf(M, r0[(long long)s * kRecFloats]);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  if (lane == 0) sm_m[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kCW; ++w) M = fmaxf(M, sm_m[w]);

  float L = 0.0f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    // this warp's partials: s_j = warp + kCW j, taken 32 at a time
    const int nj = (n_parts - warp + kCW - 1) / kCW;
    for (int j0 = 0; j0 < nj; j0 += 32) {
      float a = 0.0f;
      if (j0 + lane < nj) {
        const float* r = r0 + (long long)(warp + kCW * (j0 + lane)) * kRecFloats;
        const float ms = r[0];
        a = (ms == -INFINITY) ? 0.0f : fast_exp2(ms - M);
        L = fmaf(a, r[1], L);
      }
      const int cnt = min(32, nj - j0);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j) {
        const float aj = __shfl_sync(0xffffffffu, a, j);
        const float4 x = reinterpret_cast<const float4*>(
            r0 + (long long)(warp + kCW * (j0 + j)) * kRecFloats + 4)[lane];
        o.x = fmaf(aj, x.x, o.x); o.y = fmaf(aj, x.y, o.y);
        o.z = fmaf(aj, x.z, o.z); o.w = fmaf(aj, x.w, o.w);
      }
    }
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) L += __shfl_xor_sync(0xffffffffu, L, m);
  if (lane == 0) sm_l[warp] = L;
  reinterpret_cast<float4*>(sm_o[warp])[lane] = o;
  __syncthreads();
  const int c = threadIdx.x;   // kCW * 32 == kD channels, one per thread
  float Lt = 0.0f, oc = 0.0f;
#pragma unroll
  for (int w = 0; w < kCW; ++w) {
    Lt += sm_l[w];
    oc += sm_o[w][c];
  }
  out[row * kD + c] = Lt > 0.0f ? oc / Lt : 0.0f;
}
static_assert(kCW * 32 == kD, "one combine thread per channel");

}  // namespace

// Self-test of the bounded waits: the same wait loop as the decode rings, on
// a barrier whose phase never completes.
__global__ void wait_timeout_selftest_kernel(unsigned* status, unsigned iterations) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const bool landed = mbar_wait_bounded(&bar, 0u, iterations);
  if (!landed && threadIdx.x == 0) record_error(status, kDevErrWaitTimeout);
}

cudaError_t launch_wait_timeout_selftest(unsigned* status, unsigned iterations, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(status, iterations);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* ws, float* out, int n_rows, int n_parts, cudaStream_t s) {
  combine_kernel<<<n_rows, kCW * 32, 0, s>>>(ws, out, n_parts);
  return cudaGetLastError();
}

}  // namespace oscar
