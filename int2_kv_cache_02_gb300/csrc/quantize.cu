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
// packed 16 per word into the block record declared in oscar.h.  The fused
// prefill kernel rotates and scales the raw keys straight into the key tile
// (no k_hat round trip through global memory).
#include "launch.h"
#include "quantize.cuh"
#include "rotate.cuh"

namespace oscar {

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
  quantize_block(kt, vt, kc, vc, k_norm + src_tok, packed + (row * (T_cap / kG) + pblk) * kBlkBytes);
}

// Fused prefill: raw keys and values of n_tok tokens -> block records.  Warp w
// rotates and scales tokens 8w..8w+7 of the block (one token per warp step,
// as rotate_scale_k_kernel does), rounds k_hat to bf16 into the tile, keeps
// the norms in shared memory; the values are staged as in quantize_kv_kernel.
__global__ void __launch_bounds__(128) prefill_kv_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int in_T, int Hkv,
    int T_cap, int p0, KeyScale ks, uint8_t* __restrict__ packed) {
  __shared__ __align__(16) uint16_t kt[kG][kD];
  __shared__ __align__(16) uint16_t vt[kG][kD];
  __shared__ __align__(16) uint8_t kc[kG][kD];
  __shared__ __align__(16) uint8_t vc[kG][kD];
  __shared__ __half ns[kG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x;
  const long long row = (long long)blockIdx.z * Hkv + blockIdx.y;
  const long long src_tok = row * in_T + (long long)blk * kG;
  {
    const uint4* vs = reinterpret_cast<const uint4*>(v + src_tok * kD);
    uint4* vd = reinterpret_cast<uint4*>(&vt[0][0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) vd[tid + 128 * i] = vs[tid + 128 * i];
  }
  // with the all-heads norm, head 0 of this sequence's token src_tok
  const long long head0_tok = src_tok - (long long)blockIdx.y * in_T;
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int t = 8 * warp + i;
    float s_all = 0.0f;
    if (ks.flags & OSCAR_NORM_ALL_HEADS)
      s_all = all_heads_sq(k + (head0_tok + t) * kD, (long long)in_T * kD, Hkv, lane);
    const uint2 raw = reinterpret_cast<const uint2*>(k + (src_tok + t) * kD)[lane];
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    const float norm = rotate_scale_key(x, lane, ks, s_all);
    reinterpret_cast<uint2*>(&kt[t][0])[lane] = pack_bf16x4(x);
    if (lane == 0) ns[t] = __float2half_rn(norm);
  }
  __syncthreads();
  const long long pblk = (long long)p0 / kG + blk;
  quantize_block(kt, vt, kc, vc, ns, packed + (row * (T_cap / kG) + pblk) * kBlkBytes);
}

// ------------------------------------------------------------------ paged
// Record of logical block lb of sequence b, head h, in the page pool; an
// unmapped block (or a page id out of range) is reported and yields nullptr.
__device__ __forceinline__ uint8_t* paged_record(const PagedArgs& p, int b, int lb, int h) {
  if (lb < 0 || lb >= p.max_blocks) return nullptr;
  const int page = p.block_table[(long long)b * p.max_blocks + lb];
  if (page < 0 || page >= p.n_pages) return nullptr;
  return p.pages + ((long long)page * p.Hkv + h) * kBlkBytes;
}

// Fused prefill into pages: CTA (j, h, b) handles tokens 32j..32j+31 of
// sequence b when 32j < n_tok[b]; they become logical block
// seq_packed[b]/32 + j.  Lengths are updated by paged_lengths_kernel after.
__global__ void __launch_bounds__(128) paged_prefill_kernel(PagedArgs p,
                                                            const uint16_t* __restrict__ k,
                                                            const uint16_t* __restrict__ v,
                                                            int in_T, const int32_t* n_tok,
                                                            int max_tok) {
  __shared__ __align__(16) uint16_t kt[kG][kD];
  __shared__ __align__(16) uint16_t vt[kG][kD];
  __shared__ __align__(16) uint8_t kc[kG][kD];
  __shared__ __align__(16) uint8_t vc[kG][kD];
  __shared__ __half ns[kG];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n = n_tok[b], p0 = p.seq_packed[b];
  if (n == 0) return;
  if (n < 0 || n % kG != 0 || n > max_tok || p0 < 0 || p0 % kG != 0 || p.seq_res[b] != 0) {
    if (j == 0 && h == 0 && tid == 0) record_error(p.status, kDevErrBadPaged);
    return;
  }
  if (kG * j >= n) return;
  uint8_t* rec = paged_record(p, b, p0 / kG + j, h);
  if (rec == nullptr) {
    if (tid == 0) record_error(p.status, kDevErrBadPaged);
    return;
  }
  const long long src_tok = ((long long)b * p.Hkv + h) * in_T + (long long)j * kG;
  {
    const uint4* vs = reinterpret_cast<const uint4*>(v + src_tok * kD);
    uint4* vd = reinterpret_cast<uint4*>(&vt[0][0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) vd[tid + 128 * i] = vs[tid + 128 * i];
  }
  const long long head0_tok = src_tok - (long long)h * in_T;
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int t = 8 * warp + i;
    float s_all = 0.0f;
    if (p.ks.flags & OSCAR_NORM_ALL_HEADS)
      s_all = all_heads_sq(k + (head0_tok + t) * kD, (long long)in_T * kD, p.Hkv, lane);
    const uint2 raw = reinterpret_cast<const uint2*>(k + (src_tok + t) * kD)[lane];
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    const float norm = rotate_scale_key(x, lane, p.ks, s_all);
    reinterpret_cast<uint2*>(&kt[t][0])[lane] = pack_bf16x4(x);
    if (lane == 0) ns[t] = __float2half_rn(norm);
  }
  __syncthreads();
  quantize_block(kt, vt, kc, vc, ns, rec);
}

// Flush of full residual windows: CTA (j, h, b) quantises residual tokens
// 32j..32j+31 of (b, h) into logical block seq_packed[b]/32 + j when sequence
// b is active and its window is full.
__global__ void __launch_bounds__(128) paged_flush_kernel(PagedArgs p, const int32_t* active) {
  __shared__ __align__(16) uint16_t kt[kG][kD];
  __shared__ __align__(16) uint16_t vt[kG][kD];
  __shared__ __align__(16) uint8_t kc[kG][kD];
  __shared__ __align__(16) uint8_t vc[kG][kD];
  const int tid = threadIdx.x;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (active && active[b] == 0) return;
  if (p.seq_res[b] != kR) return;
  const int p0 = p.seq_packed[b];
  uint8_t* rec = (p0 >= 0 && p0 % kG == 0) ? paged_record(p, b, p0 / kG + j, h) : nullptr;
  if (rec == nullptr) {
    if (tid == 0) record_error(p.status, kDevErrBadPaged);
    return;
  }
  const long long row = (long long)b * p.Hkv + h;
  const long long src_tok = row * kR + (long long)j * kG;
  {
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_res + src_tok * kD);
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_res + src_tok * kD);
    uint4* kd = reinterpret_cast<uint4*>(&kt[0][0]);
    uint4* vd = reinterpret_cast<uint4*>(&vt[0][0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kd[tid + 128 * i] = ks[tid + 128 * i];
      vd[tid + 128 * i] = vs[tid + 128 * i];
    }
  }
  __syncthreads();
  quantize_block(kt, vt, kc, vc, p.k_res_norm + src_tok, rec);
}

// Length updates after a paged prefill (n_tok != nullptr) or append.
__global__ void paged_lengths_kernel(PagedArgs p, const int32_t* n_tok, int max_tok,
                                     const int32_t* active) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  if (n_tok) {
    const int n = n_tok[b];
    if (n > 0 && n % kG == 0 && n <= max_tok && p.seq_res[b] == 0) p.seq_packed[b] += n;
    return;
  }
  if (active && active[b] == 0) return;
  if (p.seq_res[b] == kR) {
    p.seq_packed[b] += kR;
    p.seq_res[b] = 1;
  } else {
    p.seq_res[b] += 1;
  }
}

cudaError_t launch_paged_prefill(const PagedArgs& p, const uint16_t* k, const uint16_t* v,
                                 int in_T, const int32_t* n_tok, int max_tok, cudaStream_t s) {
  dim3 grid(max_tok / kG, p.Hkv, p.B);
  paged_prefill_kernel<<<grid, 128, 0, s>>>(p, k, v, in_T, n_tok, max_tok);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  paged_lengths_kernel<<<(p.B + 127) / 128, 128, 0, s>>>(p, n_tok, max_tok, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_paged_flush(const PagedArgs& p, const int32_t* active, cudaStream_t s) {
  dim3 grid(kR / kG, p.Hkv, p.B);
  paged_flush_kernel<<<grid, 128, 0, s>>>(p, active);
  return cudaGetLastError();
}

cudaError_t launch_paged_lengths(const PagedArgs& p, const int32_t* active, cudaStream_t s) {
  paged_lengths_kernel<<<(p.B + 127) / 128, 128, 0, s>>>(p, nullptr, 0, active);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv(const uint16_t* k_hat, const __half* k_norm, const uint16_t* v,
                               int src_T, int n_tok, int B, int Hkv, int T_cap, int p0,
                               uint8_t* packed, cudaStream_t s) {
  dim3 grid(n_tok / kG, Hkv, B);
  quantize_kv_kernel<<<grid, 128, 0, s>>>(k_hat, k_norm, v, src_T, Hkv, T_cap, p0, packed);
  return cudaGetLastError();
}

cudaError_t launch_prefill_kv(const uint16_t* k, const uint16_t* v, int in_T, int n_tok, int B,
                              int Hkv, int T_cap, int p0, KeyScale ks, uint8_t* packed,
                              cudaStream_t s) {
  dim3 grid(n_tok / kG, Hkv, B);
  prefill_kv_kernel<<<grid, 128, 0, s>>>(k, v, in_T, Hkv, T_cap, p0, ks, packed);
  return cudaGetLastError();
}

}  // namespace oscar
