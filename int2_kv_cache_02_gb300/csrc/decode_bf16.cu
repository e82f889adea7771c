// Unquantised bf16 split-K decode attention: the comparison kernel (the
// "BF16 FlashDecoding-v2" baseline of "OScaR: The Occam's Razor for Extreme
// KV Cache Quantization in LLMs and Beyond", III. Experiments, Efficiency).
// Same grid, split and combine scheme as the INT2 kernel, no rotation or
// scaling, fp32 arithmetic on the CUDA cores.
//
// Grid (num_splits, Hkv, B), 4 warps; warps take chunks of CT = 64/GV tokens
// of the split round-robin, GV = max(GQ, 4) "virtual" heads (a group smaller
// than 4 is repeated so that a chunk always holds 64 (token, head) pairs).
// Lane l owns channels 4l..4l+3: the 64 partial q.k sums are reduced with a
// 5-step butterfly that leaves pairs 2l, 2l+1 in lane l; probabilities go
// through shared memory to the P.V loop, where every lane accumulates its 4
// channels for all heads.
#include "common.cuh"
#include "cta_merge.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int NW = 4;

template <int GQ>
__global__ void __launch_bounds__(NW * 32) decode_bf16_kernel(const Bf16DecodeArgs a) {
  constexpr int GV = GQ < 4 ? 4 : GQ;  // virtual heads: head j computes query head j % GQ
  constexpr int CT = 64 / GV;          // tokens per chunk: CT * GV = 64 partial dot products
  __shared__ MergeSmem<GQ, NW> E;
  __shared__ __align__(16) float pbuf[NW][64];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // blockIdx.y = slice sl of KV head h's query group (heads GQ sl ..), as in
  // the INT2 kernel: nh of its GQ heads are active, the rest padding
  const int split = blockIdx.x, b = blockIdx.z;
  const int slices = decode_slices(a.Hq / a.Hkv);
  const int h = blockIdx.y / slices, sl = blockIdx.y - h * slices;
  const int g = a.Hq / a.Hkv, nh = min(GQ, g - GQ * sl);
  const long long row = (long long)b * a.Hkv + h;
  const long long qrow0 = (long long)b * a.Hq + (long long)h * g + GQ * sl;
  const int t_begin = (int)((long long)a.T * split / a.num_splits);
  const int t_end = (int)((long long)a.T * (split + 1) / a.num_splits);

  float qv[GV][4];
#pragma unroll
  for (int j = 0; j < GV; ++j) {
    const uint2 r = reinterpret_cast<const uint2*>(a.q + (qrow0 + min(j % GQ, nh - 1)) * kD)[lane];
    qv[j][0] = bf16_lo(r.x); qv[j][1] = bf16_hi(r.x);
    qv[j][2] = bf16_lo(r.y); qv[j][3] = bf16_hi(r.y);
  }
  float o[GV][4], m_run[GV];
#pragma unroll
  for (int j = 0; j < GV; ++j) {
    m_run[j] = -INFINITY;
    o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
  }
  float l_part[2] = {0.0f, 0.0f};
  // heads of this lane's two (token, head) slots after the butterfly
  const int slot_head0 = (2 * lane) % GV;
  const int slot_head1 = (2 * lane + 1) % GV;
  const int slot_tok0 = (2 * lane) / GV;
  const int slot_tok1 = (2 * lane + 1) / GV;

  const uint2* Kr = reinterpret_cast<const uint2*>(a.K + row * (long long)a.T_stride * kD);
  const uint2* Vr = reinterpret_cast<const uint2*>(a.V + row * (long long)a.T_stride * kD);

  for (int t0 = t_begin + warp * CT; t0 < t_end; t0 += NW * CT) {
    uint2 kr[CT], vr[CT];
#pragma unroll
    for (int t = 0; t < CT; ++t) {
      const bool valid = t0 + t < t_end;
      kr[t] = valid ? Kr[(long long)(t0 + t) * 32 + lane] : make_uint2(0u, 0u);
      vr[t] = valid ? Vr[(long long)(t0 + t) * 32 + lane] : make_uint2(0u, 0u);
    }
    float P[64];
#pragma unroll
    for (int t = 0; t < CT; ++t) {
      const float k0 = bf16_lo(kr[t].x), k1 = bf16_hi(kr[t].x);
      const float k2 = bf16_lo(kr[t].y), k3 = bf16_hi(kr[t].y);
#pragma unroll
      for (int j = 0; j < GV; ++j)
        P[t * GV + j] = qv[j][0] * k0 + qv[j][1] * k1 + qv[j][2] * k2 + qv[j][3] * k3;
    }
    // Butterfly reduce-scatter: after the step with mask m a lane keeps the
    // half selected by its bit m; in the end lane l holds pairs 2l and 2l+1.
#pragma unroll
    for (int half = 32, m = 16; m > 0; half >>= 1, m >>= 1) {
      const bool up = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float keep = up ? P[i + half] : P[i];
        const float send = up ? P[i] : P[i + half];
        P[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
    }
    float sc0 = (t0 + slot_tok0 < t_end) ? P[0] * a.scale_log2 : -INFINITY;
    float sc1 = (t0 + slot_tok1 < t_end) ? P[1] * a.scale_log2 : -INFINITY;
    // chunk max per head over the lanes that hold that head
    float mx0 = sc0, mx1 = sc1;
#pragma unroll
    for (int m = GV / 2; m < 32; m <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, m));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, m));
    }
    float alpha[GV];
#pragma unroll
    for (int j = 0; j < GV; ++j) {
      // head j sits in slot (j % 2) of lane j / 2
      const float Mj = __shfl_sync(0xffffffffu, (j & 1) ? mx1 : mx0, j >> 1);
      const float mn = fmaxf(m_run[j], Mj);
      alpha[j] = fast_exp2(m_run[j] - mn);
      m_run[j] = mn;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[j][i] *= alpha[j];
    }
    float ms0 = m_run[0], ms1 = m_run[0], al0 = alpha[0], al1 = alpha[0];
#pragma unroll
    for (int j = 1; j < GV; ++j) {
      if (slot_head0 == j) { ms0 = m_run[j]; al0 = alpha[j]; }
      if (slot_head1 == j) { ms1 = m_run[j]; al1 = alpha[j]; }
    }
    const float p0 = fast_exp2(sc0 - ms0), p1 = fast_exp2(sc1 - ms1);
    l_part[0] = l_part[0] * al0 + p0;
    l_part[1] = l_part[1] * al1 + p1;
    pbuf[warp][2 * lane] = p0;
    pbuf[warp][2 * lane + 1] = p1;
    __syncwarp();
#pragma unroll
    for (int t = 0; t < CT; ++t) {
      const float v0 = bf16_lo(vr[t].x), v1 = bf16_hi(vr[t].x);
      const float v2 = bf16_lo(vr[t].y), v3 = bf16_hi(vr[t].y);
#pragma unroll
      for (int j = 0; j < GV; ++j) {
        const float p = pbuf[warp][t * GV + j];
        o[j][0] = fmaf(p, v0, o[j][0]);
        o[j][1] = fmaf(p, v1, o[j][1]);
        o[j][2] = fmaf(p, v2, o[j][2]);
        o[j][3] = fmaf(p, v3, o[j][3]);
      }
    }
    __syncwarp();
  }

  // l per head: sum the slots that carry it (over lanes with equal head).
  float lh0 = l_part[0], lh1 = l_part[1];
#pragma unroll
  for (int m = GV / 2; m < 32; m <<= 1) {
    lh0 += __shfl_xor_sync(0xffffffffu, lh0, m);
    lh1 += __shfl_xor_sync(0xffffffffu, lh1, m);
  }
#pragma unroll
  for (int j = 0; j < GQ; ++j) {
    const float lj = __shfl_sync(0xffffffffu, (j & 1) ? lh1 : lh0, j >> 1);
    if (lane == 0) {
      E.m[warp][j] = m_run[j];
      E.l[warp][j] = lj;
      E.z[warp][j] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) E.o[warp][j][4 * lane + i] = o[j][i];
  }
  __syncthreads();
  cta_merge_write<GQ, NW>(E, a.ws + (qrow0 * a.num_splits + split) * kRecFloats,
                          (long long)a.num_splits * kRecFloats, nh);
}

template <int GQ>
cudaError_t launch_g(const Bf16DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.num_splits, a.Hkv * decode_slices(a.Hq / a.Hkv), a.B);
  decode_bf16_kernel<GQ><<<grid, NW * 32, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(a.ws, a.out, a.B * a.Hq, a.num_splits, s);
}

template <int GQ>
int occupancy_g() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_bf16_kernel<GQ>, NW * 32, 0) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace

cudaError_t launch_decode_bf16(const Bf16DecodeArgs& a, cudaStream_t s) {
  switch (decode_group_width(a.Hq / a.Hkv)) {
    case 1: return launch_g<1>(a, s);
    case 2: return launch_g<2>(a, s);
    case 4: return launch_g<4>(a, s);
    case 8: return launch_g<8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_bf16_ctas_per_sm(int g) {
  switch (decode_group_width(g)) {
    case 1: return occupancy_g<1>();
    case 2: return occupancy_g<2>();
    case 4: return occupancy_g<4>();
    case 8: return occupancy_g<8>();
    default: return 0;
  }
}

}  // namespace oscar
