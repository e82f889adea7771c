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
// 32-token value tile at a time are staged in shared memory; the key
// parameters are formed per channel, then every thread quantises a quarter
// of one token's keys and values and stores whole words of the block
// records declared in oscar.h (quantize.cuh).  The fused prefill kernel
// rotates and scales the raw keys straight into the key tile (no k_hat round
// trip through global memory).
#include "launch.h"
#include "quantize.cuh"
#include "rotate.cuh"

namespace oscar {

// Shared memory of the group kernels: the GS keys of one group (rotated,
// scaled, bf16, padded rows), their norms and the group's key parameters
// stay for the whole group; values are staged one 32-token block at a time,
// the next block's copies in flight while the current one is worked (two
// buffers when the group has more than one block).
template <int GS>
struct GroupSmem {
  static constexpr int NVB = GS > kG ? 2 : 1;
  alignas(16) uint16_t kt[GS][kTileRow];
  alignas(16) uint16_t vt[NVB][kG][kTileRow];
  KeyParamSmem P;
  KeyMinMax mm[128];
  __half ns[GS];
};

// Rotates and scales one token's quarter of raw keys (raw: its 32 bf16 as
// four 16-byte words) into row t of kt and the token's norm into ns, in the
// quarter layout (lane l holds quarter l >> 3).  With the all-heads norm,
// head0 is the token's key of head 0 and head_stride the distance between
// heads.
template <int GS, bool PLAIN>
__device__ __forceinline__ void rotate_token(GroupSmem<GS>& S, const uint4 (&raw)[4], int t,
                                             const uint16_t* head0, long long head_stride,
                                             int Hkv, KeyScale ks) {
  const int lane = threadIdx.x & 31, Q = lane >> 3;
  float x[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[8 * j + 2 * q] = bf16_lo(u[q]);
      x[8 * j + 2 * q + 1] = bf16_hi(u[q]);
    }
  }
  float s_all = 0.0f;
  if (!PLAIN && (ks.flags & OSCAR_NORM_ALL_HEADS))
    s_all = all_heads_sq_q(head0, head_stride, Hkv, lane);
  const float norm = rotate_scale_key<PLAIN>(x, lane, ks, s_all);
  uint4* dst = reinterpret_cast<uint4*>(&S.kt[t][32 * Q]);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 o;
    o.x = bf16x2_bits(x[8 * j], x[8 * j + 1]);
    o.y = bf16x2_bits(x[8 * j + 2], x[8 * j + 3]);
    o.z = bf16x2_bits(x[8 * j + 4], x[8 * j + 5]);
    o.w = bf16x2_bits(x[8 * j + 6], x[8 * j + 7]);
    dst[j] = o;
  }
  if (Q == 0) S.ns[t] = __float2half_rn(norm);
}

// Rotates and scales the GS raw keys of a group (rows k[t], t < GS) into kt
// and their norms into ns, in the quarter layout: at step i, warp w and lane
// l take token 32 i + 8 w + (l & 7).  With the all-heads norm, head0 + t * 128
// is the token's key of head 0 and head_stride the distance between heads.
// The next step's raw keys are loaded before the current step is worked.
template <int GS, bool PLAIN>
__device__ __forceinline__ void rotate_group(GroupSmem<GS>& S, const uint16_t* k,
                                             const uint16_t* head0, long long head_stride,
                                             int Hkv, KeyScale ks) {
  const int lane = threadIdx.x & 31, Q = lane >> 3;
  const int tw = 8 * (threadIdx.x >> 5) + (lane & 7);
  uint4 raw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    raw[j] = reinterpret_cast<const uint4*>(k + (long long)tw * kD)[4 * Q + j];
#pragma unroll 1
  for (int i = 0; i < GS / kG; ++i) {
    const int t = kG * i + tw;
    uint4 cur[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cur[j] = raw[j];
    if (i + 1 < GS / kG) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        raw[j] = reinterpret_cast<const uint4*>(k + (long long)(t + kG) * kD)[4 * Q + j];
    }
    rotate_token<GS, PLAIN>(S, cur, t, head0 + (long long)t * kD, head_stride, Hkv, ks);
  }
}

// The group's GS/32 records, one block at a time, with the group's key
// parameters.  On entry kt and the norms for GS tokens, the values of block
// 0 in vt[0] (copied first, so that their loads overlap the key work) and a
// cleared P.tiny are in place and synced.  rec_of(s) gives block s's record;
// values of block s at v_src + 32 s rows.
template <int GS, int BITS, class RecOf>
__device__ __forceinline__ void quantize_group(GroupSmem<GS>& S, const __half* norms,
                                               const uint16_t* v_src, RecOf rec_of) {
  constexpr int NB = GS / kG;
  // block 0's values need no key parameter: they are worked between the
  // two halves of the key parameters, so no warp idles at the barriers
  key_minmax_half<GS>(S.kt, S.mm);
  value_block<BITS>(S.vt[0], norms, rec_of(0));
  __syncthreads();
  key_params<GS, BITS>(S.mm, S.P, rec_of);
  __syncthreads();
#pragma unroll 1
  for (int sb = 0; sb < NB; ++sb) {
    // the buffer of block sb + 1 was last read by block sb - 1's values,
    // before the barrier that preceded this block's keys
    if (sb + 1 < NB) stage_rows<kG>(S.vt[(sb + 1) % S.NVB], v_src + (long long)(sb + 1) * kG * kD);
    key_block<BITS>(&S.kt[kG * sb], S.P, rec_of(sb));
    if (sb + 1 < NB) {
      async_wait_all();
      __syncthreads();
      value_block<BITS>(S.vt[(sb + 1) % S.NVB], norms + kG * (sb + 1), rec_of(sb + 1));
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
  const int j = blockIdx.x;
  const long long row = (long long)blockIdx.z * Hkv + blockIdx.y;
  const long long src_tok = row * src_T + (long long)j * GS;
  stage_rows<kG>(S.vt[0], v + src_tok * kD);
  stage_rows<GS>(S.kt, k_hat + src_tok * kD);
  if (threadIdx.x == 0) S.P.tiny = 0;
  async_wait_all();
  __syncthreads();
  constexpr int RB = Rec<BITS>::BYTES;
  uint8_t* row_rec = packed + (row * (T_cap / kG) + p0 / kG + (long long)j * (GS / kG)) * RB;
  quantize_group<GS, BITS>(S, k_norm + src_tok, v + src_tok * kD,
                           [&](int sb) { return row_rec + (long long)sb * RB; });
}

// Fused prefill: raw keys and values of n_tok tokens -> block records.  CTA
// (j, h, b) handles group j: the group's keys are rotated and scaled in the
// quarter layout and rounded to bf16 into the key tile, the norms kept in
// shared memory; then the group's records are quantised block by block.
template <int GS, int BITS, bool PLAIN>
__global__ void __launch_bounds__(128) prefill_kv_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int in_T, int Hkv,
    int T_cap, int p0, KeyScale ks, uint8_t* __restrict__ packed) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<GroupSmem<GS>*>(smem_raw);
  const int j = blockIdx.x;
  const long long row = (long long)blockIdx.z * Hkv + blockIdx.y;
  const long long src_tok = row * in_T + (long long)j * GS;
  stage_rows<kG>(S.vt[0], v + src_tok * kD);
  if (threadIdx.x == 0) S.P.tiny = 0;
  // with the all-heads norm, head 0 of this sequence's token src_tok
  const long long head0_tok = src_tok - (long long)blockIdx.y * in_T;
  rotate_group<GS, PLAIN>(S, k + src_tok * kD, k + head0_tok * kD, (long long)in_T * kD, Hkv,
                          ks);
  async_wait_all();
  __syncthreads();
  constexpr int RB = Rec<BITS>::BYTES;
  uint8_t* row_rec = packed + (row * (T_cap / kG) + p0 / kG + (long long)j * (GS / kG)) * RB;
  quantize_group<GS, BITS>(S, S.ns, v + src_tok * kD,
                           [&](int sb) { return row_rec + (long long)sb * RB; });
}

// The fused prefill for groups of 32 tokens as a persistent kernel: CTA c
// works the units c, c + gridDim.x, ... (unit u: group u % n_groups of row
// u / n_groups, row = b Hkv + h), and the raw keys and values of its next
// unit are copied into shared memory (cp.async) while the current one is
// quantised, so a CTA waits for its loads once, not once per group.  Same
// arithmetic and records as prefill_kv_kernel.
struct PrefillSmem {
  GroupSmem<kG> G;
  alignas(16) uint16_t kraw[kG][kTileRow];   // raw keys of the unit to rotate next
};
template <int BITS, bool PLAIN>
__global__ void __launch_bounds__(128, 7) prefill_kv_persistent(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int in_T, int Hkv,
    int n_groups, long long n_units, int T_cap, int p0, KeyScale ks,
    uint8_t* __restrict__ packed) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& PS = *reinterpret_cast<PrefillSmem*>(smem_raw);
  auto& S = PS.G;
  constexpr int RB = Rec<BITS>::BYTES;
  const int tid = threadIdx.x, lane = tid & 31, Q = lane >> 3;
  const int tw = 8 * (tid >> 5) + (lane & 7);
  auto src_tok_of = [&](long long u) {
    const long long row = u / n_groups;
    return row * in_T + (u - row * n_groups) * kG;
  };
  long long u = blockIdx.x;
  if (u >= n_units) return;
  stage_rows<kG>(PS.kraw, k + src_tok_of(u) * kD);
  stage_rows<kG>(S.vt[0], v + src_tok_of(u) * kD);
#pragma unroll 1
  for (; u < n_units; u += gridDim.x) {
    const long long row = u / n_groups, j = u - row * n_groups;
    const long long src_tok = row * in_T + j * kG;
    const long long un = u + gridDim.x;
    // this unit's raw keys (its values may still be in flight); the
    // barrier also ends the previous unit's reads of kt, P and ns
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    if (tid == 0) S.P.tiny = 0;
    uint4 raw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) raw[q] = reinterpret_cast<const uint4*>(&PS.kraw[tw][32 * Q])[q];
    const long long head0_tok = src_tok - (row % Hkv) * (long long)in_T + tw;
    rotate_token<kG, PLAIN>(S, raw, tw, k + head0_tok * kD, (long long)in_T * kD, Hkv, ks);
    async_wait_all();
    __syncthreads();
    if (un < n_units) stage_rows<kG>(PS.kraw, k + src_tok_of(un) * kD);
    uint8_t* rec = packed + (row * (T_cap / kG) + p0 / kG + j) * RB;
    key_minmax_half<kG>(S.kt, S.mm);
    value_block<BITS>(S.vt[0], S.ns, rec);
    __syncthreads();
    key_params<kG, BITS>(S.mm, S.P, [&](int) { return rec; });
    __syncthreads();
    if (un < n_units) stage_rows<kG>(S.vt[0], v + src_tok_of(un) * kD);
    key_block<BITS>(S.kt, S.P, rec);
  }
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
  const int tid = threadIdx.x;
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
  stage_rows<kG>(S.vt[0], v + src_tok * kD);
  if (tid == 0) S.P.tiny = 0;
  const long long head0_tok = src_tok - (long long)h * in_T;
  rotate_group<GS, PLAIN>(S, k + src_tok * kD, k + head0_tok * kD, (long long)in_T * kD, p.Hkv,
                          p.ks);
  async_wait_all();
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
  stage_rows<kG>(S.vt[0], p.v_res + src_tok * kD);
  stage_rows<GS>(S.kt, p.k_res + src_tok * kD);
  if (tid == 0) S.P.tiny = 0;
  async_wait_all();
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
  if constexpr (GS == kG) {
    // persistent: as many CTAs as fit on the GPU at once (the count per
    // device is found once), none more than the units
    static int ctas[128] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    const size_t bytes = sizeof(PrefillSmem);
    if (!ctas[dev]) {
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_kv_persistent<BITS, PLAIN>,
                                                        128, bytes);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      ctas[dev] = std::max(1, per_sm) * std::max(1, sms);
    }
    const long long units = (long long)(n_tok / kG) * Hkv * B;
    const int grid = (int)std::min<long long>(units, ctas[dev]);
    if (grid <= 0) return cudaSuccess;
    prefill_kv_persistent<BITS, PLAIN><<<grid, 128, bytes, s>>>(k, v, in_T, Hkv, n_tok / kG, units,
                                                                T_cap, p0, ks, packed);
    return cudaGetLastError();
  } else {
    const size_t bytes = sizeof(GroupSmem<GS>);
    cudaError_t e = allow_group_smem(prefill_kv_kernel<GS, BITS, PLAIN>, bytes, done);
    if (e != cudaSuccess) return e;
    dim3 grid(n_tok / GS, Hkv, B);
    prefill_kv_kernel<GS, BITS, PLAIN><<<grid, 128, bytes, s>>>(k, v, in_T, Hkv, T_cap, p0, ks,
                                                                packed);
    return cudaGetLastError();
  }
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
