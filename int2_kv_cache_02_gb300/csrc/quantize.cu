// INT2 (or INT4) quantisation and packing of keys and values (kernel (2) of
// the news article on arXiv 2605.19660, 三).
//
// Keys: block-wise per-channel asymmetric INT2 -- every channel of every
// group of G consecutive tokens (32, or 64 / 128) has its own step and zero; values:
// per-token INT2 ("OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
// 方法步骤详情 (2)(3); 前置知识, step Δ and zero z per block).  Per group:
// z = min, Δ = (max - min)/3, code = round-half-even((x - z)/Δ) clamped to
// [0, 3], every operation one IEEE fp32 rounding; Δ = 0 and codes 0 for a
// constant group; Δ and z stored as fp16 (round to nearest even).
//
// One CTA of 128 threads per (b, h, key group): the group's key tile and one
// 32-token value tile at a time are staged in shared memory, codes computed
// one byte each, then packed into the block records declared in oscar.h.  The fused
// prefill kernel rotates and scales the raw keys straight into the key tile
// (no k_hat round trip through global memory).
#include "launch.h"
#include "quantize.cuh"
#include "rotate.cuh"

namespace oscar {

// Shared memory of the group kernels: the GS keys of one group (rotated,
// scaled, bf16) and their norms stay for the whole group; values and codes
// are staged one 32-token block at a time.
template <int GS>
struct GroupSmem {
  uint16_t kt[GS][kD];
  uint16_t vt[kG][kD];
  uint8_t kc[kG][kCodeRow];
  uint8_t vc[kG][kCodeRow];
  __half ns[GS];
};

// Copies 32 value rows (bf16, 256 B each) into vt: 16 B per thread per step.
__device__ __forceinline__ void stage_values(uint16_t (&vt)[kG][kD], const uint16_t* v) {
  const uint4* vs = reinterpret_cast<const uint4*>(v);
  uint4* vd = reinterpret_cast<uint4*>(&vt[0][0]);
#pragma unroll
  for (int i = 0; i < 4; ++i) vd[threadIdx.x + 128 * i] = vs[threadIdx.x + 128 * i];
}

// The group's GS/32 records, one block at a time, with the group's key
// parameters.  On entry kt and the norms for GS tokens and the values of
// block 0 (staged first, so that their loads overlap the key work) are in
// place and synced.  rec_of(s) gives block s's record; values of block s at
// v_src + 32 s rows.
template <int GS, int BITS, class RecOf>
__device__ __forceinline__ void quantize_group(GroupSmem<GS>& S, const __half* norms,
                                               const uint16_t* v_src, RecOf rec_of) {
  const KeyParams kp = key_params<GS, BITS>(S.kt);
  quantize_block<BITS>(&S.kt[0], S.vt, S.kc, S.vc, norms, rec_of(0), kp);
  if constexpr (GS > kG) {
#pragma unroll 1
    for (int sb = 1; sb < GS / kG; ++sb) {
      stage_values(S.vt, v_src + (long long)sb * kG * kD);
      __syncthreads();   // also: every thread is done packing the previous block
      quantize_block<BITS>(&S.kt[kG * sb], S.vt, S.kc, S.vc, norms + kG * sb, rec_of(sb), kp);
    }
  }
}

// Quantises tokens [0, n_tok) of each source row (rotated, scaled keys k_hat
// with their norms, and values) into the records of packed positions
// [p0, p0 + n_tok): CTA (j, h, b) handles group j.
template <int GS, int BITS>
__global__ void __launch_bounds__(128) quantize_kv_kernel(
    const uint16_t* __restrict__ k_hat, const __half* __restrict__ k_norm,
    const uint16_t* __restrict__ v, int src_T, int Hkv, int T_cap, int p0,
    uint8_t* __restrict__ packed) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<GroupSmem<GS>*>(smem_raw);
  const int tid = threadIdx.x;
  const int j = blockIdx.x;
  const long long row = (long long)blockIdx.z * Hkv + blockIdx.y;
  const long long src_tok = row * src_T + (long long)j * GS;
  stage_values(S.vt, v + src_tok * kD);
  {
    const uint4* ks = reinterpret_cast<const uint4*>(k_hat + src_tok * kD);
    uint4* kd = reinterpret_cast<uint4*>(&S.kt[0][0]);
#pragma unroll
    for (int i = 0; i < GS / 8; ++i) kd[tid + 128 * i] = ks[tid + 128 * i];
  }
  __syncthreads();
  constexpr int RB = Rec<BITS>::BYTES;
  uint8_t* row_rec = packed + (row * (T_cap / kG) + p0 / kG + (long long)j * (GS / kG)) * RB;
  quantize_group<GS, BITS>(S, k_norm + src_tok, v + src_tok * kD,
                           [&](int sb) { return row_rec + (long long)sb * RB; });
}

// Fused prefill: raw keys and values of n_tok tokens -> block records.  CTA
// (j, h, b) handles group j: warp w rotates and scales tokens w, w + 4, ...
// of the group (one token per warp step, as rotate_scale_k_kernel does),
// rounds k_hat to bf16 into the key tile and keeps the norms in shared
// memory; then the group's records are quantised block by block.
template <int GS, int BITS, bool PLAIN>
__global__ void __launch_bounds__(128) prefill_kv_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int in_T, int Hkv,
    int T_cap, int p0, KeyScale ks, uint8_t* __restrict__ packed) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<GroupSmem<GS>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.x;
  const long long row = (long long)blockIdx.z * Hkv + blockIdx.y;
  const long long src_tok = row * in_T + (long long)j * GS;
  stage_values(S.vt, v + src_tok * kD);
  // with the all-heads norm, head 0 of this sequence's token src_tok
  const long long head0_tok = src_tok - (long long)blockIdx.y * in_T;
  // 8 tokens' raw keys are loaded before any is transformed, so their loads
  // overlap one another rather than each FHT waiting on its own
#pragma unroll 1
  for (int i0 = 0; i0 < GS / 4; i0 += 8) {
    uint2 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      raw[i] = reinterpret_cast<const uint2*>(k + (src_tok + (GS / 4) * warp + i0 + i) * kD)[lane];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = (GS / 4) * warp + i0 + i;
      float s_all = 0.0f;
      if (!PLAIN && (ks.flags & OSCAR_NORM_ALL_HEADS))
        s_all = all_heads_sq(k + (head0_tok + t) * kD, (long long)in_T * kD, Hkv, lane);
      float x[4] = {bf16_lo(raw[i].x), bf16_hi(raw[i].x), bf16_lo(raw[i].y), bf16_hi(raw[i].y)};
      const float norm = rotate_scale_key<PLAIN>(x, lane, ks, s_all);
      reinterpret_cast<uint2*>(&S.kt[t][0])[lane] = pack_bf16x4(x);
      if (lane == 0) S.ns[t] = __float2half_rn(norm);
    }
  }
  __syncthreads();
  constexpr int RB = Rec<BITS>::BYTES;
  uint8_t* row_rec = packed + (row * (T_cap / kG) + p0 / kG + (long long)j * (GS / kG)) * RB;
  quantize_group<GS, BITS>(S, S.ns, v + src_tok * kD,
                           [&](int sb) { return row_rec + (long long)sb * RB; });
}

// ------------------------------------------------------------------ paged
// Record of logical block lb of sequence b, head h, in the page pool; an
// unmapped block (or a page id out of range) is reported and yields nullptr.
template <int BITS>
__device__ __forceinline__ uint8_t* paged_record(const PagedArgs& p, int b, int lb, int h) {
  if (lb < 0 || lb >= p.max_blocks) return nullptr;
  const int page = p.block_table[(long long)b * p.max_blocks + lb];
  if (page < 0 || page >= p.n_pages) return nullptr;
  return p.pages + ((long long)page * p.Hkv + h) * Rec<BITS>::BYTES;
}

// Fused prefill into pages: CTA (j, h, b) handles group j (tokens
// GS j .. GS j + GS - 1) of sequence b when GS j < n_tok[b]; its blocks become
// logical blocks seq_packed[b]/32 + (GS/32) j + s.  Lengths are updated by
// paged_lengths_kernel after.
template <int GS, int BITS, bool PLAIN>
__global__ void __launch_bounds__(128) paged_prefill_kernel(PagedArgs p,
                                                            const uint16_t* __restrict__ k,
                                                            const uint16_t* __restrict__ v,
                                                            int in_T, const int32_t* n_tok,
                                                            int max_tok) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<GroupSmem<GS>*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n = n_tok[b], p0 = p.seq_packed[b];
  if (n == 0) return;
  if (n < 0 || n % GS != 0 || n > max_tok || p0 < 0 || p0 % GS != 0 || p.seq_res[b] != 0) {
    if (j == 0 && h == 0 && tid == 0) record_error(p.status, kDevErrBadPaged);
    return;
  }
  if (GS * j >= n) return;
  const int lb0 = p0 / kG + j * (GS / kG);
  for (int sb = 0; sb < GS / kG; ++sb) {   // every block of the group mapped
    if (paged_record<BITS>(p, b, lb0 + sb, h) == nullptr) {
      if (tid == 0) record_error(p.status, kDevErrBadPaged);
      return;
    }
  }
  const long long src_tok = ((long long)b * p.Hkv + h) * in_T + (long long)j * GS;
  stage_values(S.vt, v + src_tok * kD);
  const long long head0_tok = src_tok - (long long)h * in_T;
#pragma unroll 1
  for (int i0 = 0; i0 < GS / 4; i0 += 8) {
    uint2 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      raw[i] = reinterpret_cast<const uint2*>(k + (src_tok + (GS / 4) * warp + i0 + i) * kD)[lane];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = (GS / 4) * warp + i0 + i;
      float s_all = 0.0f;
      if (!PLAIN && (p.ks.flags & OSCAR_NORM_ALL_HEADS))
        s_all = all_heads_sq(k + (head0_tok + t) * kD, (long long)in_T * kD, p.Hkv, lane);
      float x[4] = {bf16_lo(raw[i].x), bf16_hi(raw[i].x), bf16_lo(raw[i].y), bf16_hi(raw[i].y)};
      const float norm = rotate_scale_key<PLAIN>(x, lane, p.ks, s_all);
      reinterpret_cast<uint2*>(&S.kt[t][0])[lane] = pack_bf16x4(x);
      if (lane == 0) S.ns[t] = __float2half_rn(norm);
    }
  }
  __syncthreads();
  quantize_group<GS, BITS>(S, S.ns, v + src_tok * kD,
                           [&](int sb) { return paged_record<BITS>(p, b, lb0 + sb, h); });
}

// Flush of full residual windows: CTA (j, h, b) quantises residual group j
// (tokens GS j .. GS j + GS - 1) of (b, h) into logical blocks
// seq_packed[b]/32 + (GS/32) j + s when sequence b is active and its window
// is full.
template <int GS, int BITS>
__global__ void __launch_bounds__(128) paged_flush_kernel(PagedArgs p, const int32_t* active) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<GroupSmem<GS>*>(smem_raw);
  const int tid = threadIdx.x;
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (active && active[b] == 0) return;
  if (p.seq_res[b] != kR) return;
  const int p0 = p.seq_packed[b];
  const int lb0 = p0 / kG + j * (GS / kG);
  bool ok = p0 >= 0 && p0 % GS == 0;
  for (int sb = 0; ok && sb < GS / kG; ++sb) ok = paged_record<BITS>(p, b, lb0 + sb, h) != nullptr;
  if (!ok) {
    if (tid == 0) record_error(p.status, kDevErrBadPaged);
    return;
  }
  const long long row = (long long)b * p.Hkv + h;
  const long long src_tok = row * kR + (long long)j * GS;
  stage_values(S.vt, p.v_res + src_tok * kD);
  {
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_res + src_tok * kD);
    uint4* kd = reinterpret_cast<uint4*>(&S.kt[0][0]);
#pragma unroll
    for (int i = 0; i < GS / 8; ++i) kd[tid + 128 * i] = ks[tid + 128 * i];
  }
  __syncthreads();
  quantize_group<GS, BITS>(S, p.k_res_norm + src_tok, p.v_res + src_tok * kD,
                           [&](int sb) { return paged_record<BITS>(p, b, lb0 + sb, h); });
}

// Length updates after a paged prefill (n_tok != nullptr) or append.
__global__ void paged_lengths_kernel(PagedArgs p, const int32_t* n_tok, int max_tok,
                                     const int32_t* active) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  if (n_tok) {
    const int n = n_tok[b];
    if (n > 0 && n % p.group == 0 && n <= max_tok && p.seq_res[b] == 0) p.seq_packed[b] += n;
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

// Dynamic shared memory of the group kernels: opted in once per kernel and
// device when above the 48 KB default (GS = 128).
template <class K>
cudaError_t allow_group_smem(K kernel, size_t bytes, int (&done)[128]) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 128 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 128) done[dev] = 1;
  return e;
}

template <int GS, int BITS, bool PLAIN>
cudaError_t paged_prefill_gp(const PagedArgs& p, const uint16_t* k, const uint16_t* v, int in_T,
                             const int32_t* n_tok, int max_tok, cudaStream_t s) {
  static int done[128] = {};
  const size_t bytes = sizeof(GroupSmem<GS>);
  cudaError_t e = allow_group_smem(paged_prefill_kernel<GS, BITS, PLAIN>, bytes, done);
  if (e != cudaSuccess) return e;
  dim3 grid(max_tok / GS, p.Hkv, p.B);
  paged_prefill_kernel<GS, BITS, PLAIN><<<grid, 128, bytes, s>>>(p, k, v, in_T, n_tok, max_tok);
  return cudaGetLastError();
}
template <int GS, int BITS>
cudaError_t paged_prefill_g(const PagedArgs& p, const uint16_t* k, const uint16_t* v, int in_T,
                            const int32_t* n_tok, int max_tok, cudaStream_t s) {
  return plain_scale(p.ks) ? paged_prefill_gp<GS, BITS, true>(p, k, v, in_T, n_tok, max_tok, s)
                           : paged_prefill_gp<GS, BITS, false>(p, k, v, in_T, n_tok, max_tok, s);
}

template <int GS, int BITS>
cudaError_t paged_flush_g(const PagedArgs& p, const int32_t* active, cudaStream_t s) {
  static int done[128] = {};
  const size_t bytes = sizeof(GroupSmem<GS>);
  cudaError_t e = allow_group_smem(paged_flush_kernel<GS, BITS>, bytes, done);
  if (e != cudaSuccess) return e;
  dim3 grid(kR / GS, p.Hkv, p.B);
  paged_flush_kernel<GS, BITS><<<grid, 128, bytes, s>>>(p, active);
  return cudaGetLastError();
}

template <int GS, int BITS>
cudaError_t quantize_kv_g(const uint16_t* k_hat, const __half* k_norm, const uint16_t* v,
                          int src_T, int n_tok, int B, int Hkv, int T_cap, int p0,
                          uint8_t* packed, cudaStream_t s) {
  static int done[128] = {};
  const size_t bytes = sizeof(GroupSmem<GS>);
  cudaError_t e = allow_group_smem(quantize_kv_kernel<GS, BITS>, bytes, done);
  if (e != cudaSuccess) return e;
  dim3 grid(n_tok / GS, Hkv, B);
  quantize_kv_kernel<GS, BITS><<<grid, 128, bytes, s>>>(k_hat, k_norm, v, src_T, Hkv, T_cap, p0,
                                                        packed);
  return cudaGetLastError();
}

template <int GS, int BITS, bool PLAIN>
cudaError_t prefill_kv_gp(const uint16_t* k, const uint16_t* v, int in_T, int n_tok, int B,
                          int Hkv, int T_cap, int p0, KeyScale ks, uint8_t* packed,
                          cudaStream_t s) {
  static int done[128] = {};
  const size_t bytes = sizeof(GroupSmem<GS>);
  cudaError_t e = allow_group_smem(prefill_kv_kernel<GS, BITS, PLAIN>, bytes, done);
  if (e != cudaSuccess) return e;
  dim3 grid(n_tok / GS, Hkv, B);
  prefill_kv_kernel<GS, BITS, PLAIN><<<grid, 128, bytes, s>>>(k, v, in_T, Hkv, T_cap, p0, ks,
                                                              packed);
  return cudaGetLastError();
}
template <int GS, int BITS>
cudaError_t prefill_kv_g(const uint16_t* k, const uint16_t* v, int in_T, int n_tok, int B,
                         int Hkv, int T_cap, int p0, KeyScale ks, uint8_t* packed,
                         cudaStream_t s) {
  return plain_scale(ks)
             ? prefill_kv_gp<GS, BITS, true>(k, v, in_T, n_tok, B, Hkv, T_cap, p0, ks, packed, s)
             : prefill_kv_gp<GS, BITS, false>(k, v, in_T, n_tok, B, Hkv, T_cap, p0, ks, packed, s);
}

// Calls F::run<GS, BITS>(args...) for a (group, bits) pair the cache format
// allows (group 32, 64, 128; bits 2, 4).
template <class F, class... A>
cudaError_t dispatch_gb(int group, int bits, A&&... args) {
  if (bits == 2) {
    switch (group) {
      case 32: return F::template run<32, 2>(args...);
      case 64: return F::template run<64, 2>(args...);
      case 128: return F::template run<128, 2>(args...);
    }
  } else if (bits == 4) {
    switch (group) {
      case 32: return F::template run<32, 4>(args...);
      case 64: return F::template run<64, 4>(args...);
      case 128: return F::template run<128, 4>(args...);
    }
  }
  return cudaErrorInvalidValue;
}
struct PagedPrefillF {
  template <int GS, int BITS, class... A>
  static cudaError_t run(A... a) { return paged_prefill_g<GS, BITS>(a...); }
};
struct PagedFlushF {
  template <int GS, int BITS, class... A>
  static cudaError_t run(A... a) { return paged_flush_g<GS, BITS>(a...); }
};
struct QuantizeF {
  template <int GS, int BITS, class... A>
  static cudaError_t run(A... a) { return quantize_kv_g<GS, BITS>(a...); }
};
struct PrefillF {
  template <int GS, int BITS, class... A>
  static cudaError_t run(A... a) { return prefill_kv_g<GS, BITS>(a...); }
};

cudaError_t launch_paged_prefill(const PagedArgs& p, const uint16_t* k, const uint16_t* v,
                                 int in_T, const int32_t* n_tok, int max_tok, cudaStream_t s) {
  cudaError_t e = dispatch_gb<PagedPrefillF>(p.group, p.bits, p, k, v, in_T, n_tok, max_tok, s);
  if (e != cudaSuccess) return e;
  paged_lengths_kernel<<<(p.B + 127) / 128, 128, 0, s>>>(p, n_tok, max_tok, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_paged_flush(const PagedArgs& p, const int32_t* active, cudaStream_t s) {
  return dispatch_gb<PagedFlushF>(p.group, p.bits, p, active, s);
}

cudaError_t launch_paged_lengths(const PagedArgs& p, const int32_t* active, cudaStream_t s) {
  paged_lengths_kernel<<<(p.B + 127) / 128, 128, 0, s>>>(p, nullptr, 0, active);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv(const uint16_t* k_hat, const __half* k_norm, const uint16_t* v,
                               int src_T, int n_tok, int B, int Hkv, int T_cap, int p0, int group,
                               int bits, uint8_t* packed, cudaStream_t s) {
  return dispatch_gb<QuantizeF>(group, bits, k_hat, k_norm, v, src_T, n_tok, B, Hkv, T_cap, p0,
                                packed, s);
}

cudaError_t launch_prefill_kv(const uint16_t* k, const uint16_t* v, int in_T, int n_tok, int B,
                              int Hkv, int T_cap, int p0, int group, int bits, KeyScale ks,
                              uint8_t* packed, cudaStream_t s) {
  return dispatch_gb<PrefillF>(group, bits, k, v, in_T, n_tok, B, Hkv, T_cap, p0, ks, packed, s);
}

}  // namespace oscar
