// INT2 (or INT4) quantisation and packing of 32-token blocks of keys and
// values, shared by the group kernels (kernel (2) of the news article on
// arXiv 2605.19660, 三).
//
// Keys: block-wise per-channel asymmetric INT2 -- every channel of every
// group of G consecutive tokens (G = 32 by default; 64 and 128 are the
// larger groups) has its own step and zero, which every 32-token record of
// the group carries; values:
// per-token INT2 ("OScaR：面向大模型及多模态LLM极限KV缓存量化的奥卡姆剃刀",
// 方法步骤详情 (2)(3); 前置知识, step Δ and zero z per block).  Per group:
// z = min, Δ = (max - min)/3, code = round-half-even((x - z)/Δ) clamped to
// [0, 3], every operation one IEEE fp32 rounding; Δ = 0 and codes 0 for a
// constant group; Δ and z stored as fp16 (round to nearest even).
//
// Thread layout: the CTA's 128 threads work a block as 32 tokens x 4
// quarters.  Warp w, lane l: token 8w + (l & 7), quarter Q = l >> 3 (the
// quarter layout of rotate.cuh).  For keys a quarter is channels 32Q..32Q+31,
// which are exactly the key words 2Q, 2Q+1 (INT2) or 4Q..4Q+3 (INT4) of the
// token; for values it is the channels 2Q, 2Q+1 + 8m (m = 0..15), which fill
// whole half-words of the value words.  Each thread forms its words in
// registers and stores them; the two tokens of a value word swap halves
// through one shuffle.
#pragma once

#include "common.cuh"

namespace oscar {

// Largest code of a BITS-bit quantiser (3 for INT2, 15 for INT4).
template <int BITS>
constexpr float kMaxCode = (float)((1 << BITS) - 1);

// The code by the exact quotient (the definition).
template <int BITS>
__device__ __forceinline__ uint8_t quant_code(float x, float mn, float step, bool live) {
  if (!live) return 0;
  const float t = __fdiv_rn(__fsub_rn(x, mn), step);
  float r = rintf(t);
  r = fminf(fmaxf(r, 0.0f), kMaxCode<BITS>);
  return (uint8_t)r;
}

// The INT4 code with the quotient formed as q = (x - mn) * (1/step), as an
// exact small integer in float: q + 1.5 * 2^23 has a unit in the last place of 1
// for 0 <= q < 2^22, so adding and removing that constant rounds q to the
// nearest integer, ties to even.  The correctly rounded reciprocal times
// (x - mn) is within ~2^-21 (relative) of the rounded quotient, ~2^-19
// absolute for quotients up to 16, so both give the same integer unless the
// quotient lies within 1e-5 of a half-integer.  d keeps the largest |q - c|
// of a half-word's codes; above kNearHalf the caller redoes that half-word
// by the exact quotient (0.5 - |q - c| is the distance to the half-integer;
// the threshold keeps a margin of 1e-5 over the bound above, so a redo may
// happen needlessly, never be missed).  With bf16 inputs about one code in
// a thousand is an exact tie, so redoing only the half-word concerned keeps
// the redo cheap.  For a constant group step and reciprocal are 0 and
// x == mn, so q = 0.  q <= (2^BITS - 1)(1 + 2^-22) for every x of the group,
// so the code needs no clamp.
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23
constexpr float kNearHalf = 0.5f - 2e-5f;
__device__ __forceinline__ float code_rn(float x, float mn, float rs, float& d) {
  const float q = __fmul_rn(__fsub_rn(x, mn), rs);
  const float c = __fsub_rn(__fadd_rn(q, kRoundMagic), kRoundMagic);
  d = fmaxf(d, fabsf(__fsub_rn(q, c)));
  return c;
}
template <int BITS>
__device__ __forceinline__ float code_exact(float x, float mn, float step) {
  return (float)quant_code<BITS>(x, mn, step, step > 0.0f);
}

// A reciprocal step that overflowed (steps below 2^-128) leaves only the
// exact quotient.
__device__ __forceinline__ bool recip_ok(float rs) { return rs <= 3.0e38f; }

// INT2 codes by thresholds.  The code of a = fl(x - mn) is rint(t) with
// t = fl(a / step), non-decreasing in a, so it is at least j + 1 exactly
// when a >= A_j, the smallest fp32 a for which it is; a code is then three
// comparisons, exact for every input.  A_j follows from the rounding rules:
// h = j + 1/2 has a last mantissa bit of 0, so under round-half-even the
// quotients that round to h form [h - u-/2, h + u+/2] with both ends (u-,
// u+ the fp32 spacings below and above h).  rint(h) = j + 1 when j + 1 is
// even, so then code >= j + 1 iff a / step >= h - u-/2; otherwise iff
// a / step > h + u+/2.  The bound m step is exact in fp64 (m has at most 28
// significant bits, step 24), and A_j is that product rounded up to fp32
// (for the strict case, the next fp32 when the product is itself an fp32);
// the kernels form it in fp32 (code_threshold below).
// fp32 spacing just above (below = false) or just below h = j + 1/2 < 16:
// 2^(e - 23) with e = floor(log2 h), halved below h = 1/2 (a power of two).
__host__ __device__ constexpr double fp32_spacing(int j, bool below) {
  return j == 0 ? (below ? 0x1p-25 : 0x1p-24)
       : j < 2  ? 0x1p-23
       : j < 4  ? 0x1p-22
       : j < 8  ? 0x1p-21
                : 0x1p-20;
}
__host__ __device__ constexpr double threshold_factor(int j) {
  return ((j + 1) % 2 == 0) ? (j + 0.5) - 0.5 * fp32_spacing(j, true)
                            : (j + 0.5) + 0.5 * fp32_spacing(j, false);
}
// In fp32: m_j = h + d with h = j + 1/2 and d = m_j - h = +-2^-k, so
// m_j step = fma(h, step, d step); d step is exact (a power-of-two scaling
// of a normal number) and the fused multiply-add forms h step + d step
// exactly before its one directed rounding, so __fmaf_ru gives the product
// rounded up and __fmaf_rd rounded down.  A step below 2^-100 is first
// scaled by 2^64 (exact), so that d step stays normal, and the two results
// are scaled back with the same directed rounding (a second rounding in the
// same direction onto a coarser grid changes nothing).  The product of a
// non-finite step (never formed from finite bf16 data) takes the fp64 form.
__device__ __forceinline__ float code_threshold(float step, int j) {
  if (!(step <= 3.4028234663852886e38f)) {
    const double b = threshold_factor(j) * (double)step;
    const float up = __double2float_ru(b);
    if ((j + 1) % 2 == 0) return up;
    return __double2float_rd(b) == up ? __uint_as_float(__float_as_uint(up) + 1u) : up;
  }
  const float h = (float)j + 0.5f;
  const float d = (float)(threshold_factor(j) - ((double)j + 0.5));
  const bool tiny = step < 0x1p-100f;
  const float s = tiny ? step * 0x1p64f : step;
  const float c = d * s;
  float up = __fmaf_ru(h, s, c);
  if (tiny) up = __fmul_ru(up, 0x1p-64f);
  if ((j + 1) % 2 == 0) return up;
  float dn = __fmaf_rd(h, s, c);
  if (tiny) dn = __fmul_rd(dn, 0x1p-64f);
  return dn == up ? __uint_as_float(__float_as_uint(up) + 1u) : up;
}
// Number of thresholds at or below a = fl(x - mn): the code, as a float
// (three compares that set 1.0 or 0.0, two adds), for two inputs at once
// (packed fp32: each half rounded as the scalar operation).
__device__ __forceinline__ float2 codes_by_thresholds2(float2 x, float2 mn, float2 A0, float2 A1,
                                                       float2 A2) {
  const float2 a = sub2(x, mn);
  const float2 f0 = make_float2(a.x >= A0.x ? 1.0f : 0.0f, a.y >= A0.y ? 1.0f : 0.0f);
  const float2 f1 = make_float2(a.x >= A1.x ? 1.0f : 0.0f, a.y >= A1.y ? 1.0f : 0.0f);
  const float2 f2 = make_float2(a.x >= A2.x ? 1.0f : 0.0f, a.y >= A2.y ? 1.0f : 0.0f);
  return add2(add2(f0, f1), f2);
}

// Weight of slot k of a half-word (2 or 4 bits per slot): the half-word is
// the exact fp32 sum of c * 2^(BITS k), an integer below 2^16.
template <int BITS>
__host__ __device__ constexpr float slot_weight(int k) {
  return (float)(1u << (BITS * k));
}
// Half-word value h (an integer below 2^16 held in a float) as bits: the
// low 16 bits of the result.
__device__ __forceinline__ uint32_t half_word_bits(float h) {
  return __float_as_uint(__fadd_rn(h, 8388608.0f));   // 2^23 + h
}

// Rows of the bf16 tiles: 128 channels + 8 of padding (272 bytes), so that
// the 16-byte accesses of 8 consecutive rows at one column, and the 4-byte
// accesses of the value layout, fall on different banks.
constexpr int kTileRow = kD + 8;
// Per-channel key parameters in shared memory, 4 floats of padding after
// every 32 channels: the four quarters' 16-byte reads fall on different banks.
constexpr int kParamN = kD + 16;
__host__ __device__ constexpr int param_slot(int c) { return c + 4 * (c >> 5); }

// Per-channel key parameters: the zero mn and, for INT2, the code thresholds
// A_0..A_2 of a = x - mn in p; for INT4 the reciprocal step in p[0] and the
// step in p[1].
struct KeyParamSmem {
  alignas(16) float mn[kParamN];
  alignas(16) float p[3][kParamN];
  int tiny;   // INT4: some channel's reciprocal step overflowed
};

// Exact half-words for the redo of near-half INT4 codes: n codes of x0[2k]
// (keys: parameters mn0[2k], st0[2k]) or of x0[8k] (values: one mn, step),
// slot k weighted 16^k.  Kept out of line: it runs for about one half-word
// in a hundred.
__device__ __noinline__ float exact_key_half_word4(const uint16_t* x0, const float* mn0,
                                                   const float* st0, int n) {
  float h = 0.0f;
  for (int k = 0; k < n; ++k) {
    const float x = __uint_as_float((uint32_t)x0[2 * k] << 16);
    h = fmaf(code_exact<4>(x, mn0[2 * k], st0[2 * k]), slot_weight<4>(k), h);
  }
  return h;
}
__device__ __noinline__ float exact_value_half_word4(const uint16_t* x0, float mn, float step,
                                                     int n) {
  float h = 0.0f;
  for (int k = 0; k < n; ++k) {
    const float x = __uint_as_float((uint32_t)x0[8 * k] << 16);
    h = fmaf(code_exact<4>(x, mn, step), slot_weight<4>(k), h);
  }
  return h;
}

// Copies N rows of 128 bf16 (contiguous in global memory, 256 B each) into
// padded tile rows, 16 B per thread per step, as asynchronous copies that
// bypass the registers (one commit group); async_wait_all() before the
// barrier that publishes them.
template <int N>
__device__ __forceinline__ void stage_rows(uint16_t (*dst)[kTileRow], const uint16_t* src) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < N / 8; ++i) {
    const int c = threadIdx.x + 128 * i;   // 16-byte chunk of the source
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(&dst[c >> 4][8 * (c & 15)])),
                 "l"(s + c)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Step and zero of key channel c from its group's min and max: thresholds
// (INT2) or reciprocal step and step (INT4) into P; returns the fp16 step
// and zero the records carry.
template <int BITS>
__device__ __forceinline__ __half2 channel_params(int c, float mn, float mx, KeyParamSmem& P) {
  const bool live = mx > mn;
  const float step = live ? __fdiv_rn(__fsub_rn(mx, mn), kMaxCode<BITS>) : 0.0f;
  P.mn[param_slot(c)] = mn;
  if constexpr (BITS == 2) {
#pragma unroll
    for (int j = 0; j < 3; ++j) P.p[j][param_slot(c)] = live ? code_threshold(step, j) : INFINITY;
  } else {
    const float rs = live ? __frcp_rn(step) : 0.0f;
    P.p[0][param_slot(c)] = rs;
    P.p[1][param_slot(c)] = step;
    if (!recip_ok(rs)) P.tiny = 1;
  }
  return __halves2half2(__float2half_rn(step), __float2half_rn(mn));
}

// Per-channel min and max of the N tokens of kt, in two halves: thread t
// scans rows N/2 (t >> 6) .. N/2 (t >> 6) + N/2 - 1 of channel pair t & 63
// on packed bf16 and leaves its partial min and max in part[t].
struct KeyMinMax {
  __nv_bfloat162 mn, mx;
};
template <int N>
__device__ __forceinline__ void key_minmax_half(const uint16_t (*kt)[kTileRow], KeyMinMax* part) {
  const int t = threadIdx.x, c2 = 2 * (t & 63), r0 = (N / 2) * (t >> 6);
  __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162*>(&kt[r0][c2]), mx2 = mn2;
#pragma unroll 8
  for (int r = 1; r < N / 2; ++r) {
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&kt[r0 + r][c2]);
    mn2 = __hmin2(mn2, x);
    mx2 = __hmax2(mx2, x);
  }
  part[t] = KeyMinMax{mn2, mx2};
}

// Step and zero of key channel 2 (t & 63) + (t >> 6) (one channel per
// thread) from the two halves' partials of key_minmax_half: its parameters
// into P and its fp16 step and zero into the records rec_of(0 .. N/32 - 1).
// P.tiny must have been cleared before the barrier that precedes the call.
template <int N, int BITS, class RecOf>
__device__ __forceinline__ void key_params(const KeyMinMax* part, KeyParamSmem& P, RecOf rec_of) {
  const int t = threadIdx.x, pr = t & 63, hi = t >> 6, c = 2 * pr + hi;
  const KeyMinMax a = part[pr], b = part[pr + 64];
  const __nv_bfloat162 mn2 = __hmin2(a.mn, b.mn), mx2 = __hmax2(a.mx, b.mx);
  const float mn = hi ? __high2float(mn2) : __low2float(mn2);
  const float mx = hi ? __high2float(mx2) : __low2float(mx2);
  const __half2 sz = channel_params<BITS>(c, mn, mx, P);
  using RL = Rec<BITS>;
#pragma unroll 1
  for (int sb = 0; sb < N / kG; ++sb) {
    uint8_t* rec = rec_of(sb);
    reinterpret_cast<__half*>(rec + RL::KS)[c] = __low2half(sz);
    reinterpret_cast<__half*>(rec + RL::KZ)[c] = __high2half(sz);
  }
}

// Key words of this thread's token (row of kt) and quarter: INT2 words 2Q,
// 2Q+1 (16 channels each; channel 16w + j at bit 2(j/2) + 16(j%2)), INT4
// words 4Q..4Q+3 (8 channels each; channel 8w + j at bit 4(j/2) + 16(j%2)).
// Half-word h = 2 (e / CW) + (e & 1) of the quarter holds its channels e of
// word e / CW with the parity of h, at slot (e % CW) / 2.
template <int BITS>
__device__ __forceinline__ void key_words(const uint16_t* row, int Q, const KeyParamSmem& P,
                                          uint32_t (&w)[BITS == 2 ? 2 : 4]) {
  constexpr int NW = BITS == 2 ? 2 : 4;   // words of the quarter
  constexpr int CW = 32 / NW;             // channels per word
  uint32_t xr[16];                        // the quarter's 32 bf16, packed
  {
    const uint4* src = reinterpret_cast<const uint4*>(row + 32 * Q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = src[i];
      xr[4 * i] = u.x;
      xr[4 * i + 1] = u.y;
      xr[4 * i + 2] = u.z;
      xr[4 * i + 3] = u.w;
    }
  }
  const int q0 = param_slot(32 * Q);
  if constexpr (BITS == 2) {
    // channels e, e + 1 (e even) are one packed bf16 pair and land in the
    // same slot of half-words 2k, 2k + 1 of word k = e / CW: one packed pair
    // of accumulators per word
    float2 hw[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) hw[k] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 m = reinterpret_cast<const float4*>(P.mn + q0)[i];
      const float4 t0 = reinterpret_cast<const float4*>(P.p[0] + q0)[i];
      const float4 t1 = reinterpret_cast<const float4*>(P.p[1] + q0)[i];
      const float4 t2 = reinterpret_cast<const float4*>(P.p[2] + q0)[i];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int e = 4 * i + 2 * jj, k = e / CW;
        const float wgt = slot_weight<BITS>((e % CW) >> 1);
        const float2 mn = jj ? make_float2(m.z, m.w) : make_float2(m.x, m.y);
        const float2 a0 = jj ? make_float2(t0.z, t0.w) : make_float2(t0.x, t0.y);
        const float2 a1 = jj ? make_float2(t1.z, t1.w) : make_float2(t1.x, t1.y);
        const float2 a2 = jj ? make_float2(t2.z, t2.w) : make_float2(t2.x, t2.y);
        hw[k] = fma2(codes_by_thresholds2(bf16_pair(xr[e >> 1]), mn, a0, a1, a2),
                     make_float2(wgt, wgt), hw[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < NW; ++k)
      w[k] = __byte_perm(half_word_bits(hw[k].x), half_word_bits(hw[k].y), 0x5410);
  } else {
    float hw[2 * NW], d[2 * NW];
#pragma unroll
    for (int i = 0; i < 2 * NW; ++i) hw[i] = 0.0f;
    const float d0 = P.tiny ? 1.0f : 0.0f;
#pragma unroll
    for (int i = 0; i < 2 * NW; ++i) d[i] = d0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 m = reinterpret_cast<const float4*>(P.mn + q0)[i];
      const float4 r = reinterpret_cast<const float4*>(P.p[0] + q0)[i];
      const float mv[4] = {m.x, m.y, m.z, m.w}, rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 4 * i + j, jw = e % CW, h = 2 * (e / CW) + (jw & 1);
        const float x = (e & 1) ? bf16_hi(xr[e >> 1]) : bf16_lo(xr[e >> 1]);
        hw[h] = fmaf(code_rn(x, mv[j], rv[j], d[h]), slot_weight<BITS>(jw >> 1), hw[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < 2 * NW; ++h) {
      if (d[h] > kNearHalf) {
        const int e0 = (h >> 1) * CW + (h & 1);
        hw[h] = exact_key_half_word4(row + 32 * Q + e0, P.mn + q0 + e0, P.p[1] + q0 + e0, CW / 2);
      }
    }
#pragma unroll
    for (int k = 0; k < NW; ++k)
      w[k] = __byte_perm(half_word_bits(hw[2 * k]), half_word_bits(hw[2 * k + 1]), 0x5410);
  }
}

// Value words of this thread's token (row of vt) with the token's step and
// zero.  The thread quantises channels g + 8m of its token for g = 2Q, 2Q+1
// (m = 0..15), i.e. whole half-words (g, hh): INT2 slot k = channel
// g + 8(8hh + k) (hh = 0, 1), INT4 slot k = channel g + 8(4hh + k) (hh =
// 0..3).  A value word holds one half-word of each token of a pair (t, t+1),
// t even, in its low and high halves.  The even token stores the words of
// channel group g = 2Q, the odd token those of g = 2Q + 1; each passes the
// other group's half-words to its partner (lane ^ 1).  par = t & 1.
template <int BITS>
__device__ __forceinline__ void value_words(const uint16_t* row, int Q, int par,
                                            uint32_t (&w)[BITS == 2 ? 2 : 4], float& step_out,
                                            float& mn_out) {
  constexpr int NH = BITS == 2 ? 2 : 4;   // half-words per channel group g
  constexpr int PS = 16 / NH;             // slots per half-word
  uint32_t u[16];   // channel pairs (2Q + 8m, 2Q + 1 + 8m), packed bf16
#pragma unroll
  for (int m = 0; m < 16; ++m) u[m] = *reinterpret_cast<const uint32_t*>(row + 8 * m + 2 * Q);
  auto xv = [&](int g, int m) { return g ? bf16_hi(u[m]) : bf16_lo(u[m]); };
  auto b2 = [&](int m) { return *reinterpret_cast<const __nv_bfloat162*>(&u[m]); };
  __nv_bfloat162 mn2 = b2(0), mx2 = b2(0);
#pragma unroll
  for (int m = 1; m < 16; ++m) {
    mn2 = __hmin2(mn2, b2(m));
    mx2 = __hmax2(mx2, b2(m));
  }
  float mn = fminf(__low2float(mn2), __high2float(mn2));
  float mx = fmaxf(__low2float(mx2), __high2float(mx2));
#pragma unroll
  for (int s = 8; s < 32; s <<= 1) {   // the token's other quarters
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, s));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
  }
  const bool live = mx > mn;
  const float step = live ? __fdiv_rn(__fsub_rn(mx, mn), kMaxCode<BITS>) : 0.0f;
  uint32_t Hb[2][NH];   // half-words as bits
  if constexpr (BITS == 2) {
    // the token's thresholds A_0..A_2, one per quarter thread
    const int lane = threadIdx.x & 31;
    const float mine = (live && Q < 3) ? code_threshold(step, Q) : INFINITY;
    const float A0 = __shfl_sync(0xffffffffu, mine, lane & 7);
    const float A1 = __shfl_sync(0xffffffffu, mine, (lane & 7) + 8);
    const float A2 = __shfl_sync(0xffffffffu, mine, (lane & 7) + 16);
    // the pair u[m] holds channel 2Q + 8m (group 0) low and 2Q + 1 + 8m
    // (group 1) high, at the same slot of half-words (0, hh) and (1, hh)
    float2 H[NH];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) H[hh] = make_float2(0.0f, 0.0f);
    const float2 mn2 = make_float2(mn, mn), A02 = make_float2(A0, A0), A12 = make_float2(A1, A1),
                 A22 = make_float2(A2, A2);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float wgt = slot_weight<BITS>(m % PS);
      H[m / PS] = fma2(codes_by_thresholds2(bf16_pair(u[m]), mn2, A02, A12, A22),
                       make_float2(wgt, wgt), H[m / PS]);
    }
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      Hb[0][hh] = half_word_bits(H[hh].x);
      Hb[1][hh] = half_word_bits(H[hh].y);
    }
  } else {
    const float rs = live ? __frcp_rn(step) : 0.0f;
    float H[2][NH], d[2][NH];
    const float d0 = recip_ok(rs) ? 0.0f : 1.0f;
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        H[g][hh] = 0.0f;
        d[g][hh] = d0;
      }
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int m = 0; m < 16; ++m)
        H[g][m / PS] = fmaf(code_rn(xv(g, m), mn, rs, d[g][m / PS]), slot_weight<BITS>(m % PS),
                            H[g][m / PS]);
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int hh = 0; hh < NH; ++hh)
        if (d[g][hh] > kNearHalf)
          H[g][hh] = exact_value_half_word4(row + 2 * Q + g + 8 * PS * hh, mn, step, PS);
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) Hb[g][hh] = half_word_bits(H[g][hh]);
  }
  // keep: this token's half-words of the group it stores; send: the other
  // group's, two per register (hh 2i low, 2i + 1 high)
  uint32_t keep[NH], send[NH / 2];
#pragma unroll
  for (int hh = 0; hh < NH; ++hh) keep[hh] = par ? Hb[1][hh] : Hb[0][hh];
#pragma unroll
  for (int i = 0; i < NH / 2; ++i)
    send[i] = __byte_perm(par ? Hb[0][2 * i] : Hb[1][2 * i],
                          par ? Hb[0][2 * i + 1] : Hb[1][2 * i + 1], 0x5410);
#pragma unroll
  for (int i = 0; i < NH / 2; ++i) {
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send[i], 1);
    // even token: own half-word low, the partner's high; odd token: reversed
    w[2 * i] = __byte_perm(keep[2 * i], recv, par ? 0x1054u : 0x5410u);
    w[2 * i + 1] = __byte_perm(keep[2 * i + 1], recv, par ? 0x1076u : 0x7610u);
  }
  step_out = step;
  mn_out = mn;
}

// One 32-token block of values (vt: 32 rows) and the tokens' norms: its
// value codes, steps and zeros and its norms into the record (layout in
// oscar.h for BITS).  Called by all 128 threads once vt and the norms are
// staged and synced; needs no key parameter.
template <int BITS>
__device__ __forceinline__ void value_block(const uint16_t (*vt)[kTileRow], const __half* norms,
                                            uint8_t* rec) {
  using RL = Rec<BITS>;
  constexpr int NW = BITS == 2 ? 2 : 4;
  const int lane = threadIdx.x & 31, Q = lane >> 3;
  const int t = 8 * (threadIdx.x >> 5) + (lane & 7);
  uint32_t w[NW];
  float step, mn;
  value_words<BITS>(vt[t], Q, t & 1, w, step, mn);
  // word of (token pair, channel group g, hh = 0): INT2 128 kh + 4 (4g +
  // t4) + 2p, INT4 256 kh + 128 p + 4 (4g + t4), the pair's first token
  // being 16 kh + 2 t4 + 8 p
  const int g = 2 * Q + (t & 1), kh = t >> 4, p = (t >> 3) & 1, t4 = (t >> 1) & 3;
  uint32_t* vc = reinterpret_cast<uint32_t*>(rec + RL::VC);
  if constexpr (BITS == 2) {
    *reinterpret_cast<uint2*>(vc + 128 * kh + 4 * (4 * g + t4) + 2 * p) = make_uint2(w[0], w[1]);
  } else {
    *reinterpret_cast<uint4*>(vc + 256 * kh + 128 * p + 4 * (4 * g + t4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (Q == 0) reinterpret_cast<__half*>(rec + RL::VS)[tok_slot(t)] = __float2half_rn(step);
  if (Q == 1) reinterpret_cast<__half*>(rec + RL::VZ)[tok_slot(t)] = __float2half_rn(mn);
  if (Q == 2) reinterpret_cast<__half*>(rec + RL::KN)[tok_slot(t)] = norms[t];
}

// One 32-token block of keys (kt: 32 rotated, scaled bf16 rows) with the
// group's key parameters in P: its key codes into the record (key_params
// writes the key steps and zeros).  Called by all 128 threads once P is
// formed and synced.
template <int BITS>
__device__ __forceinline__ void key_block(const uint16_t (*kt)[kTileRow], const KeyParamSmem& P,
                                          uint8_t* rec) {
  using RL = Rec<BITS>;
  constexpr int NW = BITS == 2 ? 2 : 4;
  const int lane = threadIdx.x & 31, Q = lane >> 3;
  const int t = 8 * (threadIdx.x >> 5) + (lane & 7);
  uint32_t w[NW];
  key_words<BITS>(kt[t], Q, P, w);
  uint32_t* kc = reinterpret_cast<uint32_t*>(rec + RL::KC) + t * 4 * NW + NW * Q;
  if constexpr (BITS == 2) {
    *reinterpret_cast<uint2*>(kc) = make_uint2(w[0], w[1]);
  } else {
    *reinterpret_cast<uint4*>(kc) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace oscar
