// Merge of per-warp online-softmax states into one split-K partial record.
//
// Each warp w leaves, per query head j of the CTA's group, its running max m
// (log2 domain), running sum l, a per-head additive term z (added to every
// channel) and the unnormalised output o[128].  The CTA folds them with the
// log-sum-exp rule and writes record (m, l, -, -, o[0..127]) of its split.
#pragma once
#include "common.cuh"
#include "launch.h"

namespace oscar {

template <int GQ, int NW>
struct MergeSmem {
  float m[NW][GQ];
  float l[NW][GQ];
  float z[NW][GQ];
  float o[NW][GQ][kD];
};

// Called by all NW*32 threads of the CTA (NW*32 >= 128) after a __syncthreads
// that follows the per-warp writes into `s`; heads 0 .. nh - 1 (nh <= GQ) are
// written, the rest are padding.
template <int GQ, int NW>
__device__ __forceinline__ void cta_merge_write(const MergeSmem<GQ, NW>& s, float* rec_base,
                                                long long rec_stride, int nh = GQ) {
  const int c = threadIdx.x;
  if (c >= kD) return;
#pragma unroll 1
  for (int j = 0; j < nh; ++j) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s.m[w][j]);
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float a = fast_exp2(s.m[w][j] - M);
        L += a * s.l[w][j];
        o += a * (s.o[w][j][c] + s.z[w][j]);
      }
    }
    float* rec = rec_base + (long long)j * rec_stride;
    if (c == 0) {
      rec[0] = M;
      rec[1] = L;
    }
    rec[4 + c] = o;
  }
}

}  // namespace oscar
