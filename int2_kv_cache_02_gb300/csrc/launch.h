// Host-side launchers of the liboscar kernels (internal; the public ABI is
// include/oscar.h).  Each returns the cudaGetLastError() after its launches.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/oscar.h"

namespace oscar {

// How keys are scaled (Omni-Token Scaling and its variants): the ablation
// and norm-scope flags of oscar.h and the target norm (1 = unit norm).
struct KeyScale {
  unsigned flags;
  float target;
};

constexpr unsigned kAllFlags = OSCAR_NO_ROTATE | OSCAR_NO_SCALE | OSCAR_NORM_ALL_HEADS;

// Target norm of the scaled keys as the ABI takes it: 0 means 1; otherwise
// within [2^-8, 2^8].
inline bool target_ok(float t) {
  return t == 0.0f || (t >= 0.00390625f && t <= 256.0f);   // false for NaN
}
// Key group size as the ABI takes it: 0 means 32; otherwise 32, 64 or 128.
inline bool key_group_ok(int g) { return g == 0 || g == 32 || g == 64 || g == 128; }
inline int key_group(int g) { return g == 0 ? 32 : g; }
// Code width as the ABI takes it: 0 means 2; otherwise 2 or 4.
inline bool code_bits_ok(int b) { return b == 0 || b == 2 || b == 4; }
inline int code_bits(int b) { return b == 0 ? 2 : b; }
inline KeyScale key_scale(unsigned flags, float target) {
  return KeyScale{flags, target == 0.0f ? 1.0f : target};
}
// Query exponent of the decode kernel: keys scaled to norm t have elements,
// hence steps, below t, so the query's largest element goes to about
// 2^(14 - ceil(log2 t)); unscaled keys are as large as the data (2^1).
inline int query_exponent(const KeyScale& ks) {
  if (ks.flags & OSCAR_NO_SCALE) return 1;
  int e = 0;
  const float m = frexpf(ks.target, &e);   // t = m * 2^e, m in [0.5, 1)
  return 14 - (m > 0.5f ? e : e - 1);
}

cudaError_t launch_rotate_q(const uint16_t* q, float* out, int n_vec, unsigned flags,
                            cudaStream_t s);

// Rows are (b, h) with h fastest over Hkv heads (the all-heads norm reads a
// token's keys in every head of its sequence).
cudaError_t launch_rotate_scale_k(const uint16_t* k, int in_T, uint16_t* k_hat, __half* norm,
                                  int out_T, int out_t0, int n_rows, int Hkv, int n_tok,
                                  const uint16_t* v_in, uint16_t* v_out, KeyScale ks,
                                  cudaStream_t s);

// Quantises tokens [0, n_tok) of each source row into the block records of
// packed positions [p0, p0 + n_tok).
// Keys are grouped by `group` tokens (32, 64 or 128; n_tok and p0 multiples
// of it): every channel of a group shares one step and zero.
cudaError_t launch_quantize_kv(const uint16_t* k_hat, const __half* k_norm, const uint16_t* v,
                               int src_T, int n_tok, int B, int Hkv, int T_cap, int p0, int group,
                               int bits, uint8_t* packed, cudaStream_t s);

struct DecodeArgs {
  const uint8_t* packed;   // block records [B][Hkv][T_cap/32]
  const uint16_t* k_res;
  const uint16_t* v_res;
  const __half* k_res_norm;
  const float* q_rot;
  float* ws;          // partial records [B*Hq][num_splits + 1][kRecFloats]
  unsigned* row_count;  // arrival counters [B*Hkv], zero between calls
  float* out;         // [B][Hq][128]
  unsigned* status;
  int B, Hkv, Hq, T_cap, n_packed, n_res, num_splits;
  // slices of each query group: decode_slices(Hq / Hkv)
  int slices = 1;
  unsigned flags;
  float scale_log2;   // softmax_scale * log2(e)
  // the query is scaled by 2^(q_exp - e), e the exponent of its largest
  // element, so that q'*step stays in fp16 range for the cache's key scale
  int q_exp = 14;
  int bits = 2;   // code width of the records (2 or 4)
  // paged cache (block_table != nullptr): records at packed + (page*Hkv + h)
  // * block bytes, page = block_table[b*max_blocks + block]; per-sequence
  // lengths seq_packed[b], seq_res[b] replace n_packed, n_res; n_packed
  // then holds the host bound on the seq_packed[b], which sizes the splits
  const int32_t* block_table = nullptr;
  const int32_t* seq_packed = nullptr;
  const int32_t* seq_res = nullptr;
  int max_blocks = 0, n_pages = 0;
  // fused decode step (contiguous cache): q_raw (bf16 [B][Hq][128]) replaces
  // q_rot and is rotated in the kernel; k_new, v_new (bf16 [B][Hkv][128]) are
  // the new token, which the residual CTA of each row rotates, scales and
  // writes at residual slot n_res - 1 before it reads the window (n_res then
  // counts the new token); norm_target is the cache's key-scaling target
  const uint16_t* q_raw = nullptr;
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
  float norm_target = 1.0f;
};

// Floats per split-K partial record: m, l, 2 pad, o[128].
constexpr int kRecFloats = 132;

// Decode workspace: a header of kMaxDecodeRows arrival counters (u32, one per
// (b, h) row, zero between calls), then the partial records
// [B*Hq][parts][kRecFloats].  The header has the same size and place for
// every shape and split count, so no call's partials overlap any call's
// counters.
constexpr long long kMaxDecodeRows = 1 << 16;
constexpr size_t kDecodeWsHeader = kMaxDecodeRows * sizeof(unsigned);
inline size_t decode_ws_bytes(long long B, long long /*Hkv*/, long long Hq, long long parts) {
  return kDecodeWsHeader + (size_t)(B * Hq * parts) * kRecFloats * sizeof(float);
}
inline unsigned* decode_row_counters(void* ws) { return static_cast<unsigned*>(ws); }
inline float* decode_partials(void* ws) {
  return reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kDecodeWsHeader);
}

// Query heads per KV head, g = Hq / Hkv, from 1 to kMaxGroup.  The decode
// kernels are instantiated for groups of 1, 2, 4 and 8 heads per CTA
// (decode_group_width); a group of another size takes the next width, with
// padding heads that are worked but neither merged nor written, and a group
// above 8 is cut into slices of 8 (decode_slices), each of which reads the
// KV head's cache on its own.
constexpr int kMaxGroup = 16;
__host__ __device__ constexpr int decode_group_width(int g) {
  return g <= 1 ? 1 : g == 2 ? 2 : g <= 4 ? 4 : 8;
}
__host__ __device__ constexpr int decode_slices(int g) {
  return (g + decode_group_width(g) - 1) / decode_group_width(g);
}
// Rows of a decode launch, one per (sequence, KV head, slice), or 0 when Hq
// is not a multiple of Hkv with a group of 1..kMaxGroup heads.
inline long long decode_rows(long long B, int Hkv, int Hq) {
  if (B <= 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || Hq / Hkv > kMaxGroup) return 0;
  return B * Hkv * decode_slices(Hq / Hkv);
}

// Fused INT2 decode attention with the split-K combine in its last CTA per
// row (one launch).
cudaError_t launch_decode_int2(const DecodeArgs& a, cudaStream_t s);
// The same for query groups that are not a whole kernel group (1, 2, 4, 8
// heads): decode_int2_pad.cu.
cudaError_t launch_decode_int2_padded(const DecodeArgs& a, cudaStream_t s);
// Blocks per SM the INT2 decode kernel reaches for query group size g.
int decode_int2_ctas_per_sm(int g);

struct Bf16DecodeArgs {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;
  float* ws;
  float* out;
  int B, Hq, Hkv, T, T_stride, num_splits;
  float scale_log2;
};

cudaError_t launch_decode_bf16(const Bf16DecodeArgs& a, cudaStream_t s);
int decode_bf16_ctas_per_sm(int g);

// Device address of the current device's status word (nullptr if unavailable),
// and the host launch counter behind oscar_kernel_launches().
unsigned* device_status_word();
void count_launches(int n);
// The argument checks every contiguous-cache call applies to an oscar_cache.
oscar_status validate_cache(const oscar_cache* c);

// Paged cache: fused prefill of n_tok[b] tokens per sequence (then n_packed
// += n_tok), flush of full residual windows, residual append of one token,
// and the length updates of an append.
struct PagedArgs {
  uint8_t* pages;
  int32_t* block_table;
  int32_t* seq_packed;
  int32_t* seq_res;
  uint16_t* k_res;
  uint16_t* v_res;
  __half* k_res_norm;
  unsigned* status;
  int B, Hkv, max_blocks, n_pages;
  int group;   // key group size: 32, 64 or 128 tokens
  int bits;    // code width: 2 or 4
  KeyScale ks;
};
cudaError_t launch_paged_prefill(const PagedArgs& p, const uint16_t* k, const uint16_t* v,
                                 int in_T, const int32_t* n_tok, int max_tok, cudaStream_t s);
cudaError_t launch_paged_append(const PagedArgs& p, const uint16_t* k_new, const uint16_t* v_new,
                                const int32_t* active, cudaStream_t s);

// Fused rotate + scale + quantise of n_tok tokens of raw keys and values.
cudaError_t launch_prefill_kv(const uint16_t* k, const uint16_t* v, int in_T, int n_tok, int B,
                              int Hkv, int T_cap, int p0, int group, int bits, KeyScale ks,
                              uint8_t* packed, cudaStream_t s);

// One CTA polls an mbarrier nothing arrives at, `iterations` times, then
// records kDevErrWaitTimeout in *status (self-test of the bounded waits).
cudaError_t launch_wait_timeout_selftest(unsigned* status, unsigned iterations, cudaStream_t s);

// Log-sum-exp combine of n_parts partial records per (b, q-head).
cudaError_t launch_combine(const float* ws, float* out, int n_rows, int n_parts, cudaStream_t s);

}  // namespace oscar
