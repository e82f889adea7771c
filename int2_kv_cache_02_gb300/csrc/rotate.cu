// Canalized Rotation (online fast Walsh-Hadamard transform over head_dim)
// and Omni-Token Scaling, with its norm-scope and target-norm variants.
//
// "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs and
// Beyond" (reading notes), II. Method, Step One (K' = K.H, H orthogonal with
// entries +-1/sqrt(d), computed as an O(d log d) FHT; the same rotation is
// applied to Q) and Step Two (divide each token by its own L2 norm, keep the
// norm).  News article on arXiv 2605.19660, 三: one fused kernel does the FHT
// and the scaling for K and only the FHT for Q, with the hardware rsqrt.
//
// One warp per 128-vector: lane l holds elements 4l..4l+3.  Index bits 0-1
// are butterflied in registers, bits 2-6 across lanes with shuffles.
#include "launch.h"
#include "rotate.cuh"

namespace oscar {

__global__ void __launch_bounds__(256) rotate_q_kernel(const uint16_t* __restrict__ q,
                                                       float* __restrict__ out, int n_vec,
                                                       unsigned flags) {
  const int lane = threadIdx.x & 31;
  const long long v = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (v >= n_vec) return;
  const uint2 raw = reinterpret_cast<const uint2*>(q + v * kD)[lane];
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  if (!(flags & OSCAR_NO_ROTATE)) {
    fht128(x, lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] *= kInvSqrtD;
  }
  reinterpret_cast<float4*>(out + v * kD)[lane] = make_float4(x[0], x[1], x[2], x[3]);
}

// Rotates and scales n_tok keys per (b,h) row; optionally copies the value of
// the same token (the decode append).
__global__ void __launch_bounds__(256) rotate_scale_k_kernel(
    const uint16_t* __restrict__ k, int in_T, uint16_t* __restrict__ k_hat,
    __half* __restrict__ norm_out, int out_T, int out_t0, int n_rows, int Hkv, int n_tok,
    const uint16_t* __restrict__ v_in, uint16_t* __restrict__ v_out, KeyScale ks) {
  const int lane = threadIdx.x & 31;
  const long long v = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (v >= (long long)n_rows * n_tok) return;
  const long long row = v / n_tok;
  const int t = (int)(v - row * n_tok);
  const long long src = (row * in_T + t) * kD;
  const long long dst_tok = row * out_T + out_t0 + t;

  float s_all = 0.0f;
  if (ks.flags & OSCAR_NORM_ALL_HEADS) {
    const long long row0 = row - row % Hkv;   // head 0 of this sequence
    s_all = all_heads_sq(k + (row0 * in_T + t) * kD, (long long)in_T * kD, Hkv, lane);
  }
  const uint2 raw = reinterpret_cast<const uint2*>(k + src)[lane];
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  const float norm = rotate_scale_key(x, lane, ks, s_all);
  reinterpret_cast<uint2*>(k_hat + dst_tok * kD)[lane] = pack_bf16x4(x);
  if (lane == 0) norm_out[dst_tok] = __float2half_rn(norm);
  if (v_in != nullptr) {
    reinterpret_cast<uint2*>(v_out + dst_tok * kD)[lane] =
        reinterpret_cast<const uint2*>(v_in + src)[lane];
  }
}

// Paged residual append: one warp per (b, h) of an active sequence writes
// its new token at residual slot n_res[b] (slot 0 after a flush of a full
// window, which paged_flush_kernel has done before this launch).
__global__ void __launch_bounds__(256) paged_append_kernel(PagedArgs p,
                                                           const uint16_t* __restrict__ k_new,
                                                           const uint16_t* __restrict__ v_new,
                                                           const int32_t* active) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= (long long)p.B * p.Hkv) return;
  const int b = (int)(row / p.Hkv);
  if (active && active[b] == 0) return;
  const int r = p.seq_res[b];
  if (r < 0 || r > kR) {
    if (lane == 0) record_error(p.status, kDevErrBadPaged);
    return;
  }
  const int slot = (r == kR) ? 0 : r;
  const long long dst = row * kR + slot;
  float s_all = 0.0f;
  if (p.ks.flags & OSCAR_NORM_ALL_HEADS)
    s_all = all_heads_sq(k_new + (long long)b * p.Hkv * kD, kD, p.Hkv, lane);
  const uint2 raw = reinterpret_cast<const uint2*>(k_new + row * kD)[lane];
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  const float norm = rotate_scale_key(x, lane, p.ks, s_all);
  reinterpret_cast<uint2*>(p.k_res + dst * kD)[lane] = pack_bf16x4(x);
  if (lane == 0) p.k_res_norm[dst] = __float2half_rn(norm);
  reinterpret_cast<uint2*>(p.v_res + dst * kD)[lane] =
      reinterpret_cast<const uint2*>(v_new + row * kD)[lane];
}

cudaError_t launch_paged_flush(const PagedArgs& p, const int32_t* active, cudaStream_t s);
cudaError_t launch_paged_lengths(const PagedArgs& p, const int32_t* active, cudaStream_t s);

cudaError_t launch_paged_append(const PagedArgs& p, const uint16_t* k_new, const uint16_t* v_new,
                                const int32_t* active, cudaStream_t s) {
  cudaError_t e = launch_paged_flush(p, active, s);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.Hkv;
  paged_append_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p, k_new, v_new, active);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_paged_lengths(p, active, s);
}

cudaError_t launch_rotate_q(const uint16_t* q, float* out, int n_vec, unsigned flags,
                            cudaStream_t s) {
  const int grid = (n_vec + 7) / 8;
  rotate_q_kernel<<<grid, 256, 0, s>>>(q, out, n_vec, flags);
  return cudaGetLastError();
}

cudaError_t launch_rotate_scale_k(const uint16_t* k, int in_T, uint16_t* k_hat, __half* norm,
                                  int out_T, int out_t0, int n_rows, int Hkv, int n_tok,
                                  const uint16_t* v_in, uint16_t* v_out, KeyScale ks,
                                  cudaStream_t s) {
  const long long n = (long long)n_rows * n_tok;
  const long long grid = (n + 7) / 8;
  rotate_scale_k_kernel<<<(unsigned)grid, 256, 0, s>>>(k, in_T, k_hat, norm, out_T, out_t0,
                                                       n_rows, Hkv, n_tok, v_in, v_out, ks);
  return cudaGetLastError();
}

}  // namespace oscar
