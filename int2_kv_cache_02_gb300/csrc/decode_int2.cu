// Fused INT2 dequantisation + inverse token scaling + split-K decode attention
// over the packed cache and the bf16 residual window (kernel (3) of the news
// article on arXiv 2605.19660, 三; "OScaR: The Occam's Razor for Extreme KV
// Cache Quantization in LLMs and Beyond", II. End-to-End Flow and III.
// Efficiency: "Q.K^T and dequantization fused into a single kernel").
//
// One-dimensional grid of B * Hkv * (num_splits + 1) CTAs: the first B * Hkv
// handle the residual windows of rows (b, h), so they all start in the first
// wave; the others, row by row, each stream an equal share of the 32-token
// blocks of their row.  Each CTA writes one log-sum-exp partial per query head
// and counts itself in the row's arrival counter; the row's last CTA to
// arrive folds the row's partials into the output (row_combine) and resets
// the counter, so no second kernel is launched.
//
// Packed path, per 32-token block and warp (all on mma.sync m16n8k16 f16):
//  * no per-element dequantisation: the key step s_c of the block is folded
//    into the query (q~_c = q'_c s_c, split into fp16 hi + lo parts so the
//    product keeps ~22 bits), the key zero z_c becomes one dot product
//    Z = q'.z per block (itself an MMA), and the norm multiplies the score:
//      score_t = tau * n_t * (sum_c q~_c code_tc + Z);
//  * key codes enter Q.K as exact fp16 subnormals (a masked code is
//    c * 4^p * 2^-24; 4^-p goes into the step, 2^24 into the score);
//  * values: p~_t = p_t s_t (hi + lo fp16) multiplies the centred codes
//    code - 1.5 on the tensor cores; the per-token constant z_t + 1.5 s_t is
//    accumulated as sum_t p_t (z_t + 1.5 s_t) and added per channel at the end;
//    a masked value code pair is an fp16 subnormal like the keys, and one
//    exact fp16 FMA turns it into (c - 1.5) times a per-row power of two;
//  * groups of up to 4 query heads ("column" layout): Q.K runs with 16 tokens
//    as the M rows and the (head, limb) pairs of q~ as the 8 N columns, so no
//    row is wasted; each lane then holds whole scores of one head, and the
//    8x8 tiles of (hi, lo) probabilities become the P.V operand with one
//    movmatrix transpose each;
//  * groups of 8 ("row" layout): Q.K runs with the 16 (head, limb) rows of q~
//    as M and 8 tokens as N; its accumulator layout is already the P.V
//    operand layout.
// Each warp streams its own contiguous range of blocks through its own
// NSTAGE-deep shared-memory ring: one 1-D bulk copy (TMA, cp.async.bulk) of
// the block's record per block (2752 bytes; 4800 for the INT4 option, two in
// flight), completing on the warp's mbarrier.  Waits are bounded and record
// kDevErrWaitTimeout instead of hanging; no CTA-wide barrier runs inside the
// main loop.  Instantiations: query group g, contiguous or paged records
// (through the block table), a per-block step scale for caches with the
// all-heads norm, the code width, and whether the CTA's group is padded (a
// group of another size than 1, 2, 4 or 8, or one slice of a group above 8).
#include "common.cuh"
#include "cta_merge.cuh"
#include "launch.h"
#include "rotate.cuh"

namespace oscar {
namespace {

constexpr int NW = 4;       // warps per CTA

// Per code width: the record (key codes, value codes, key step, key zero,
// norms, value step, value zero; oscar.h) and the ring depth per warp.  The
// INT4 record is 1.74x the INT2 one, so two of them in flight per warp hold
// about as many bytes as four INT2 records, and the CTA keeps 4 per SM.
template <int BITS>
struct Layout {
  using RL = Rec<BITS>;
  static constexpr int NSTAGE = BITS == 2 ? 4 : 2;
  static constexpr int SMEM = NW * NSTAGE * RL::BYTES + NW * NSTAGE * 8;
  static constexpr float CENTER = BITS == 2 ? 1.5f : 7.5f;   // mid code (2^BITS - 1) / 2
};

constexpr float kLazyLog2 = 8.0f;         // lazy softmax rescale threshold (log2 units)
constexpr int kQStage = 8 * 32 * 16;   // row layout: staged query fragments (bytes)
constexpr int kQRotStage = 16 * kD * 4;   // fused step: the rotated queries (bytes)
// Dynamic shared memory of an instantiation: the rings and barriers and the
// staged query fragments of the row layout; a fused-step launch adds the
// rotated queries (kQRotStage) after them.
template <int GQ, int BITS>
constexpr int smem_bytes() { return Layout<BITS>::SMEM + (GQ == 8 ? kQStage : 0); }
// The kernel's dynamic shared memory (every extern declaration names the
// same address).
__device__ __forceinline__ uint8_t* dyn_smem() {
  extern __shared__ __align__(128) uint8_t dyn_smem_base[];
  return dyn_smem_base;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t x, uint32_t s, uint32_t b) {
  return half2_as_u32(__hfma2(u32_as_half2(x), u32_as_half2(s), u32_as_half2(b)));
}
__device__ __forceinline__ uint32_t neg2_u(uint32_t x) {
  return half2_as_u32(__hneg2(u32_as_half2(x)));
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t x, uint32_t y) {
  return half2_as_u32(__hmul2(u32_as_half2(x), u32_as_half2(y)));
}

// Key code pair at slot k (low/high half-word) as fp16x2 subnormals: masking
// a code into an otherwise empty half-word gives exactly c * 4^p * 2^-24,
// where p is the code's 2-bit position (slots 0..4 sit at positions 0..4 of
// w, slots 5..7 at positions 0..2 of w10 = w >> 10).  The fp16 MMA
// multiplies subnormals exactly; 4^-p is folded into the query side and 2^24
// into the score, so no per-code arithmetic is left.
template <int K>
__device__ __forceinline__ uint32_t key_pair(uint32_t w, uint32_t w10) {
  if constexpr (K < 5) {
    return w & (0x00030003u << (2 * K));
  } else {
    return w10 & (0x00030003u << (2 * (K - 5)));
  }
}
// 2-bit position of key slot K inside the word it is extracted from.
constexpr int key_pos(int K) { return K < 5 ? K : K - 5; }
// fp16x2 {4^-p, 4^-p}
constexpr uint32_t pow4_inv_h2(int p) {
  return p == 0 ? 0x3C003C00u : p == 1 ? 0x34003400u : p == 2 ? 0x2C002C00u
       : p == 3 ? 0x24002400u : 0x1C001C00u;
}

// Per-block step scale for caches whose keys are not all of unit norm (the
// all-heads norm scope: a head's k_hat may be far below 1).  Returns 2^E as
// fp16x2 with E chosen so that the block's largest key step times 2^E lies in
// [0.5, 1): the query-step products q' sigma s 4^-p then keep both fp16
// limbs in the normal range, as they do for unit-norm keys.  The caller
// divides the Q.K sum by 2^E.  Lane tig holds channels 32 tig .. 32 tig + 31;
// lanes xor 1, 2 hold the rest.  Steps are >= 0, so the max of their fp16
// values picks the largest.
__device__ __forceinline__ int block_step_exp(const uint4* ks4) {
  __half2 m = u32_as_half2(0u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = ks4[i];
    m = __hmax2(m, __hmax2(__hmax2(u32_as_half2(v.x), u32_as_half2(v.y)),
                           __hmax2(u32_as_half2(v.z), u32_as_half2(v.w))));
  }
  uint32_t mb = half2_as_u32(m);
  mb = max(mb & 0xffffu, mb >> 16);
  mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
  mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
  return mb == 0 ? 0 : 14 - (int)(mb >> 10);   // mb >> 10: biased exponent
}

// fp16x2 {2^E 4^-p, ..} for p = 0..4 (INT2) or {2^E 16^-p, ..} for p = 0, 1
// (INT4) (exact: powers of two >= 2^-24).
template <int BITS>
__device__ __forceinline__ void step_scales(uint32_t (&c)[5], int E) {
  const float f = __int_as_float((127 + E) << 23);
  c[0] = half2_as_u32(__floats2half2_rn(f, f));
  if constexpr (BITS == 2) {
#pragma unroll
    for (int p = 1; p < 5; ++p) c[p] = hmul2_u(c[0], pow4_inv_h2(p));
  } else {
    c[1] = hmul2_u(c[0], 0x2C002C00u);   // 16^-1
  }
}

// Value code pair at slot k as centred fp16 values (c - 1.5) * 2^(2p - 9):
// the masked pair is the subnormal c * 4^p * 2^-24 (as for the keys), and
// one exact HFMA2 scales it by 2^15 and subtracts 1.5 * 2^(2p - 9).  p is
// the code's 2-bit position (slots 0..4 in w, 5..7 in w10 = w >> 10); the
// row factor 2^(2p - 9) is undone once per split (value_unscale).  Unlike a
// subnormal MMA operand (whose products with subnormal probabilities were
// lost), the operand is a normal, centred number.
template <int K>
__device__ __forceinline__ uint32_t value_pair(uint32_t w, uint32_t w10) {
  constexpr uint32_t B[5] = {0x9A009A00u, 0xA200A200u, 0xAA00AA00u, 0xB200B200u, 0xBA00BA00u};
  return hfma2_u(key_pair<K>(w, w10), 0x78007800u /* 2^15 */, B[key_pos(K)]);
}
// 2^(9 - 2p) for value slot k: undoes the row factor of value_pair
__host__ __device__ constexpr float value_unscale(int k) {
  return key_pos(k) == 0 ? 512.0f : key_pos(k) == 1 ? 128.0f : key_pos(k) == 2 ? 32.0f
       : key_pos(k) == 3 ? 8.0f : 2.0f;
}

// A operand of P.V m-tile mt (channels 16 mt + gid, + 8 on the row halves)
// from the lane's four value words (tokens 2 tig.. and 2 tig + 8..) and
// their copies shifted right by 10: row gid takes slot 2 (mt % 4), row
// gid + 8 slot 2 (mt % 4) + 1, of the words for channel half mt / 4.
__device__ __forceinline__ void value_frag(uint32_t (&av)[4], int mt, const uint32_t (&wv)[4],
                                           const uint32_t (&w10)[4]) {
  const int hh = mt >> 2;
  const int p0 = hh, p1 = 2 + hh;  // words of tokens (2tig,2tig+1) and (2tig+8,2tig+9)
  switch (mt & 3) {
    case 0:
      av[0] = value_pair<0>(wv[p0], w10[p0]); av[1] = value_pair<1>(wv[p0], w10[p0]);
      av[2] = value_pair<0>(wv[p1], w10[p1]); av[3] = value_pair<1>(wv[p1], w10[p1]);
      break;
    case 1:
      av[0] = value_pair<2>(wv[p0], w10[p0]); av[1] = value_pair<3>(wv[p0], w10[p0]);
      av[2] = value_pair<2>(wv[p1], w10[p1]); av[3] = value_pair<3>(wv[p1], w10[p1]);
      break;
    case 2:
      av[0] = value_pair<4>(wv[p0], w10[p0]); av[1] = value_pair<5>(wv[p0], w10[p0]);
      av[2] = value_pair<4>(wv[p1], w10[p1]); av[3] = value_pair<5>(wv[p1], w10[p1]);
      break;
    default:
      av[0] = value_pair<6>(wv[p0], w10[p0]); av[1] = value_pair<7>(wv[p0], w10[p0]);
      av[2] = value_pair<6>(wv[p1], w10[p1]); av[3] = value_pair<7>(wv[p1], w10[p1]);
      break;
  }
}

// INT4 codes.  A word holds 8 channels (keys) or 4 channels x 2 tokens
// (values), 4 bits each; nibble positions 0 and 1 of each half-word are exact
// fp16 subnormals c * 16^p * 2^-24 as they stand, positions 2 and 3 after a
// shift right by 8 (ws = w >> 8).  Slot K (0..3) of a half-word: position
// K & 1 of w (K < 2) or of ws.
template <int K>
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, uint32_t ws) {
  return (K < 2 ? w : ws) & (0x000F000Fu << (4 * (K & 1)));
}
// fp16x2 {16^-p, 16^-p} for position p = 0, 1
constexpr uint32_t pow16_inv_h2(int p) { return p == 0 ? 0x3C003C00u : 0x2C002C00u; }
// Value slot K as (c - 7.5) * 2^(4p - 9), p = K & 1: exact as for INT2.
template <int K>
__device__ __forceinline__ uint32_t value_nib(uint32_t w, uint32_t ws) {
  constexpr uint32_t B = (K & 1) ? 0xB380B380u /* -7.5 * 2^-5 */ : 0xA380A380u /* -7.5 * 2^-9 */;
  return hfma2_u(nib_pair<K>(w, ws), 0x78007800u /* 2^15 */, B);
}
// A operand of P.V m-tile mt from the lane's eight INT4 value words (4 per
// token pair: slots hold channels g + 8 (4 hh + k)): row gid takes slot
// 2 (mt % 2) of word hh = mt / 2, row gid + 8 the next slot; words 0..3 are
// tokens (2 tig, 2 tig + 1), words 4..7 tokens (2 tig + 8, 2 tig + 9).
__device__ __forceinline__ void value_frag4(uint32_t (&av)[4], int mt, const uint32_t (&wv)[8],
                                            const uint32_t (&ws)[8]) {
  const int hh = mt >> 1, p0 = hh, p1 = 4 + hh;
  if ((mt & 1) == 0) {
    av[0] = value_nib<0>(wv[p0], ws[p0]); av[1] = value_nib<1>(wv[p0], ws[p0]);
    av[2] = value_nib<0>(wv[p1], ws[p1]); av[3] = value_nib<1>(wv[p1], ws[p1]);
  } else {
    av[0] = value_nib<2>(wv[p0], ws[p0]); av[1] = value_nib<3>(wv[p0], ws[p0]);
    av[2] = value_nib<2>(wv[p1], ws[p1]); av[3] = value_nib<3>(wv[p1], ws[p1]);
  }
}
// Row factor of P.V m-tile mt, row half r (0: row gid, 1: gid + 8), undone in
// the epilogue: 2^(9 - 2p) for INT2 (p the code's 2-bit position), 2^(9 - 4p)
// for INT4 (p = r).
template <int BITS>
__host__ __device__ constexpr float row_unscale(int mt, int r) {
  return BITS == 2 ? value_unscale(2 * (mt & 3) + r) : (r ? 32.0f : 512.0f);
}

// Four fp16 values (two packed pairs) as floats.
__device__ __forceinline__ void unpack_h4(float (&f)[4], uint32_t ab, uint32_t cd) {
  const float2 x = __half22float2(u32_as_half2(ab)), y = __half22float2(u32_as_half2(cd));
  f[0] = x.x; f[1] = x.y; f[2] = y.x; f[3] = y.y;
}

// One warp's contiguous range of a row's 32-token blocks, streamed through
// the warp's own NSTAGE-deep ring: one elected lane copies block i's record
// into slot i % NSTAGE with one 1-D bulk copy completing on that slot's
// mbarrier.
template <bool PAGED, int BITS>
struct WarpRing {
  static constexpr int NSTAGE = Layout<BITS>::NSTAGE;
  static constexpr int RB = Layout<BITS>::RL::BYTES;
  uint8_t* ring;
  uint64_t* bars;
  const uint8_t* src;   // record of the range's first block (contiguous cache)
  int n;                // blocks in the range
  int lane;
  // paged cache: the index of the range's first block-table entry and the
  // offset of the row's KV head within a page; the table, the pool and the
  // page stride are read from the launch arguments where they are used, so
  // the loop keeps two 32-bit values for paging (a record's address is one
  // 32 x 32 -> 64-bit multiply-add onto the pool)
  int tab_i;                // the range's first entry in the block table
  unsigned hoff;            // the row's KV head record within a page (bytes)

  // Page id of block i of the range (paged cache; 0 past the range's end or
  // for a contiguous cache).  Loaded when block i - NSTAGE is taken up, so
  // the load's latency is hidden by that block's work.
  __device__ __forceinline__ int page_of(int i, const DecodeArgs& a) const {
    if constexpr (PAGED) return i < n ? __ldg(a.block_table + (tab_i + i)) : 0;
    else return 0;
  }
  // Record of block i of the range, `page` its page id (paged cache; the
  // range's ids were checked against the pool when the ring was made).
  __device__ __forceinline__ const uint8_t* record(int i, int page, const DecodeArgs& a) const {
    if constexpr (PAGED) {
      return a.packed + ((unsigned long long)(unsigned)page * ((unsigned)a.Hkv * (unsigned)RB) + hoff);
    } else {
      return src + (long long)i * RB;
    }
  }

  __device__ __forceinline__ void start(const DecodeArgs& a) const {
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
      mbar_fence_init();
    }
    __syncwarp();
    for (int i = 0; i < NSTAGE && i < n; ++i) issue(i, page_of(i, a), a);
  }
  __device__ __forceinline__ void issue(int i, int page, const DecodeArgs& a) const {
    // Every lane forms the (warp-uniform) addresses; one lane chosen by
    // elect.sync arms the slot's mbarrier and issues the copy, so no branch
    // on the lane index is needed.
    const uint8_t* rec = record(i, page, a);
    const unsigned bar = smem_u32(&bars[i % NSTAGE]);
    const unsigned dst = smem_u32(ring + (i % NSTAGE) * RB);
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %2;\n\t"
        "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%1], [%3], %2, [%0];\n\t}"
        :: "r"(bar), "r"(dst), "r"(RB), "l"(rec) : "memory");
  }
  // true on every lane once block i has landed; false if the wait gave up
  __device__ __forceinline__ bool wait(int i) const {
    return __all_sync(0xffffffffu, mbar_wait_bounded(&bars[i % NSTAGE],
                                                     (unsigned)((i / NSTAGE) & 1), kWaitLimit));
  }
  __device__ __forceinline__ const uint8_t* slot(int i) const {
    return ring + (i % NSTAGE) * RB;
  }
  // After consuming block i: refill its slot with block i + NSTAGE, whose
  // page id (paged cache) was loaded by page_of when block i was taken up.
  __device__ __forceinline__ void release(int i, int page, const DecodeArgs& a) const {
    __syncwarp();
    if (i + NSTAGE < n) issue(i + NSTAGE, page, a);
  }
  // The wait for block `it` gave up: record it and wait (bounded) for the
  // copies still in flight, blocks it .. min(it + NSTAGE, n) - 1, so that no
  // copy lands in shared memory after the warp has moved on.
  __device__ __forceinline__ void fail(int it, unsigned* status) const {
    if (lane == 0) {
      record_error(status, kDevErrWaitTimeout);
      for (int s = it; s < it + NSTAGE && s < n; ++s)
        if (!mbar_wait_bounded(&bars[s % NSTAGE], (unsigned)((s / NSTAGE) & 1), kDrainLimit))
          record_error(status, kDevErrDrainTimeout);
    }
    __syncwarp();
  }
};

// Blocks of row (b, h): the cache's n_packed, or for a paged cache the
// sequence's own length (checked: a bad length is reported and gives none).
template <bool PAGED>
__device__ __forceinline__ int row_blocks(const DecodeArgs& a, int b) {
  if constexpr (PAGED) {
    const int n = __ldg(a.seq_packed + b);
    if (n < 0 || n % kG != 0 || n / kG > a.max_blocks) {
      record_error(a.status, kDevErrBadPaged);
      return 0;
    }
    return n / kG;
  } else {
    return a.n_packed / kG;
  }
}

// Number of packed splits that sequence b of a paged batch fills: chunks of
// at most c = ceil(longest / splits) blocks, the longest sequence's split
// size (n_packed carries that bound), so sequence b takes ceil(n_b / c)
// splits of equal length; a short sequence fills fewer splits, each nearly
// as long as a long sequence's (no half-empty last chunk), and the per-CTA
// setup is paid per chunk of work.  A sequence longer than the bound spreads
// over all the splits.
__device__ __forceinline__ int paged_splits_used(const DecodeArgs& a, int nblk) {
  const int c = max(1, (a.n_packed / kG + a.num_splits - 1) / a.num_splits);
  return max(1, min(a.num_splits, (nblk + c - 1) / c));
}

template <bool PAGED, int BITS>
__device__ __forceinline__ WarpRing<PAGED, BITS> make_ring(const DecodeArgs& a, uint8_t* smem,
                                                           int b, int h, int split) {
  constexpr int NSTAGE = Layout<BITS>::NSTAGE, RB = Layout<BITS>::RL::BYTES;
  const int warp = threadIdx.x >> 5;
  const int nblk = row_blocks<PAGED>(a, b);
  int b0, b1;
  if constexpr (PAGED) {
    const int sb = paged_splits_used(a, nblk);
    b0 = split < sb ? (int)((long long)nblk * split / sb) : nblk;
    b1 = split < sb ? (int)((long long)nblk * (split + 1) / sb) : nblk;
  } else {
    b0 = (int)((long long)nblk * split / a.num_splits);
    b1 = (int)((long long)nblk * (split + 1) / a.num_splits);
  }
  const int wb0 = b0 + (int)((long long)(b1 - b0) * warp / NW);
  const int wb1 = b0 + (int)((long long)(b1 - b0) * (warp + 1) / NW);
  const long long row = (long long)b * a.Hkv + h;
  WarpRing<PAGED, BITS> r;
  r.ring = smem + warp * NSTAGE * RB;
  r.bars = reinterpret_cast<uint64_t*>(smem + NW * NSTAGE * RB) + warp * NSTAGE;
  r.src = a.packed + (row * (long long)(a.T_cap / kG) + wb0) * RB;
  r.n = wb1 - wb0;
  r.lane = threadIdx.x & 31;
  r.tab_i = PAGED ? b * a.max_blocks + wb0 : 0;
  r.hoff = (unsigned)h * (unsigned)RB;
  if constexpr (PAGED) {
    // Every page id of the range is checked once, before any copy: one out
    // of range is reported and the warp reads nothing (its result is void).
    bool bad = false;
    for (int j = r.lane; j < r.n; j += 32) bad |= (unsigned)__ldg(a.block_table + (r.tab_i + j)) >= (unsigned)a.n_pages;
    if (__any_sync(0xffffffffu, bad)) {
      if (r.lane == 0) record_error(a.status, kDevErrBadPaged);
      r.n = 0;
    }
  }
  return r;
}

// 8x8 fp16 tile transpose across the warp: the lane holding row r, columns
// 2c and 2c+1 receives row r, columns 2c and 2c+1 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}

// Query scaling shared by both layouts: q' times softmax_scale * log2(e) and
// a power of two sigma chosen per head so that the fp16 parts stay in range.
// qf holds channels 32*tig .. 32*tig+31 of the head; the lanes xor 1 and xor 2
// hold the rest of it.  Returns sigma; qf is scaled in place.
__device__ __forceinline__ void load_query(float4 (&qv)[8], const float* qrow, int tig) {
  const float4* qp = reinterpret_cast<const float4*>(qrow + 32 * tig);
#pragma unroll
  for (int i = 0; i < 8; ++i) qv[i] = qp[i];
}
// Fused decode step: the rotated query from its raw bf16 elements 4l .. 4l
// + 3 (lane l), formed exactly as rotate_q_kernel forms it (same butterflies
// in the same order), so the fused step and the separate calls agree bit
// for bit.
__device__ __forceinline__ float4 rotate_query_raw(const DecodeArgs& a, uint2 raw, int lane) {
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  if (!(a.flags & OSCAR_NO_ROTATE)) {
    fht128(x, lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) x[r] *= kInvSqrtD;
  }
  return make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ float4 rotated_query(const DecodeArgs& a, long long v, int lane) {
  return rotate_query_raw(a, reinterpret_cast<const uint2*>(a.q_raw + v * kD)[lane], lane);
}

// Fused decode step: the queries, staged as float [heads][128] in shared
// memory past the end of the non-fused kernel's dynamic shared memory (the
// fused launch alone enlarges it), in two phases.  load_raw_queries issues
// the raw loads before the ring's first copies, so that they do not queue
// behind them; stage_rotated_queries rotates and stores them.  For groups of
// up to 4 heads every warp rotates all of them into its own area and waits
// only for itself, so a starting CTA's warps do not wait on one another; for
// groups of 8 warp w rotates heads w and w + 4 into one area shared by the
// CTA, behind a barrier.  Both are called by every thread; the result points
// at the row's first query head.
template <int GQ>
struct RawQueries {
  static constexpr int N = GQ <= NW ? GQ : GQ / NW;   // heads loaded per warp
  uint2 v[N];
};
template <int GQ>
__device__ __forceinline__ void load_raw_queries(const DecodeArgs& a, long long qrow0, int nh,
                                                 RawQueries<GQ>& raw) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < RawQueries<GQ>::N; ++k) {
    const int j = GQ <= NW ? k : warp + NW * k;
    raw.v[k] = reinterpret_cast<const uint2*>(a.q_raw + (qrow0 + min(j, nh - 1)) * kD)[lane];
  }
}
template <int GQ>
__device__ __forceinline__ const float* stage_rotated_queries(const DecodeArgs& a,
                                                              const RawQueries<GQ>& raw,
                                                              uint8_t* stage) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* qs = reinterpret_cast<float*>(stage) + (GQ <= NW ? warp * GQ * kD : 0);
#pragma unroll
  for (int k = 0; k < RawQueries<GQ>::N; ++k) {
    const int j = GQ <= NW ? k : warp + NW * k;
    reinterpret_cast<float4*>(qs + j * kD)[lane] = rotate_query_raw(a, raw.v[k], lane);
  }
  if constexpr (GQ <= NW) {
    __syncwarp();
  } else {
    __syncthreads();
  }
  return qs;
}

__device__ __forceinline__ float scale_query(float (&qf)[32], const float4 (&qv)[8],
                                            const DecodeArgs& a) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = qv[i];
    qf[4 * i] = v.x * a.scale_log2; qf[4 * i + 1] = v.y * a.scale_log2;
    qf[4 * i + 2] = v.z * a.scale_log2; qf[4 * i + 3] = v.w * a.scale_log2;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qf[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  int e = 0;
  if (amax > 0.0f) frexpf(amax, &e);
  int sh = (amax > 0.0f) ? (a.q_exp - e) : 0;
  sh = max(-100, min(100, sh));
  const float sigma = ldexpf(1.0f, sh);
#pragma unroll
  for (int i = 0; i < 32; ++i) qf[i] *= sigma;
  return sigma;
}

// ---------------------------------------------------------------- columns
// Groups of up to 4 query heads.  Lane (gid, tig):
//  * Q.K B operand: column gid = (head (gid/2) mod GQ, limb gid%2) of q~;
//  * Q.K A operand: key codes of tokens 16 mt + gid and 16 mt + gid + 8;
//  * scores, softmax and outputs: head tig mod GQ (columns 2 tig, 2 tig + 1
//    are its hi and lo limbs), tokens gid + 8 j, j = 0..3;
//  * P.V: channels on M as in the row layout, (head, limb of p~) on N.
template <int GQ, bool BSCALE, int BITS, class Ring>
__device__ __forceinline__ void packed_cols(const DecodeArgs& a, const Ring& R,
                                            MergeSmem<GQ, NW>& E, long long qrow0, int nh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  // head of this lane's q~ column (a padding head of a partial group works
  // on the last active head's query; its results are not merged)
  const int hq = min((gid >> 1) % GQ, nh - 1);
  const int limb = gid & 1;         // 0: hi part, 1: lo part
  const int hs = tig % GQ;          // head of this lane's scores and outputs
  using RL = typename Layout<BITS>::RL;
  constexpr int LW = BITS == 2 ? 2 : 4;   // key words per token and lane
  // The query's loads go out first, then the ring's first copies, which
  // travel while the query is prepared (INT4: the copies first, which keeps
  // its instantiations free of spills).
  float4 qv[8];
  if (a.q_raw != nullptr) {   // fused step: rotate the CTA's queries here
    RawQueries<GQ> raw;
    load_raw_queries<GQ>(a, qrow0, nh, raw);
    R.start(a);
    const float* qs = stage_rotated_queries<GQ>(a, raw, dyn_smem() + smem_bytes<GQ, BITS>());
    load_query(qv, qs + hq * kD, tig);
  } else if constexpr (BITS == 2) {
    load_query(qv, a.q_rot + (qrow0 + hq) * kD, tig);
    R.start(a);
  } else {
    R.start(a);
    load_query(qv, a.q_rot + (qrow0 + hq) * kD, tig);
  }

  // This lane's column of q' for channels 32 tig + 4 k8 + {0,1} (pair 0) and
  // + {2,3} (pair 1): qz = the column's own limb (the Z operand), qhm = the hi
  // limb on lo columns and 0 on hi columns.  Per block, with step s,
  //   r = qz s + (qhm s - fp16(qhm s))
  // is fp16(q' s) on hi columns and the exact remainder's fp16 on lo columns.
  uint32_t qz[8][2], qhm[8][2];
  float inv_sigma;
  {
    float qf[32];
    const float sigma = scale_query(qf, qv, a);
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float x0 = qf[4 * k8 + 2 * j], x1 = qf[4 * k8 + 2 * j + 1];
        const __half2 hh = __floats2half2_rn(x0, x1);
        const float2 hv = __half22float2(hh);
        const __half2 ll = __floats2half2_rn(x0 - hv.x, x1 - hv.y);
        qz[k8][j] = half2_as_u32(limb ? ll : hh);
        qhm[k8][j] = limb ? half2_as_u32(hh) : 0u;
      }
    // the score head's 1/sigma lives on the lanes whose column head is hs
    inv_sigma = __shfl_sync(0xffffffffu, ldexpf(1.0f, -ilogbf(sigma)), 8 * hs);
  }
  // the Q.K sums carry 2^-24 (subnormal key codes) and sigma
  const float qk_scale = 16777216.0f * inv_sigma;

  float O[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) O[mt][e] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f, z_run = 0.0f;

  int it = 0;
  for (; it < R.n; ++it) {
    if (!R.wait(it)) break;
    const int page_next = R.page_of(it + Ring::NSTAGE, a);
    const uint8_t* st = R.slot(it);
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st + RL::KC);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + RL::VC);
    const uint4* ks4 = reinterpret_cast<const uint4*>(st + RL::KS) + tig * 4;
    const uint4* kz4 = reinterpret_cast<const uint4*>(st + RL::KZ) + tig * 4;
    // norms, value steps and zeros of tokens gid + 8 j, j = 0..3 (adjacent
    // in the record)
    const uint2 kn4 = *reinterpret_cast<const uint2*>(st + RL::KN + 8 * gid);
    const uint2 vs4 = *reinterpret_cast<const uint2*>(st + RL::VS + 8 * gid);
    const uint2 vz4 = *reinterpret_cast<const uint2*>(st + RL::VZ + 8 * gid);

    // key words of tokens 16 mt + gid + 8 r: INT2 words 2 tig, 2 tig + 1
    // (16 channels each, shifted copies w >> 10), INT4 words 4 tig .. 4 tig + 3
    // (8 channels each, shifted copies w >> 8)
    uint32_t kw[2][2][LW], kw10[2][2][LW];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if constexpr (BITS == 2) {
          const uint2 v = *reinterpret_cast<const uint2*>(kc + (16 * mt + gid + 8 * r) * 8 + 2 * tig);
          kw[mt][r][0] = v.x; kw[mt][r][1] = v.y;
          kw10[mt][r][0] = v.x >> 10; kw10[mt][r][1] = v.y >> 10;
        } else {
          const uint4 v = *reinterpret_cast<const uint4*>(kc + (16 * mt + gid + 8 * r) * 16 + 4 * tig);
          kw[mt][r][0] = v.x; kw[mt][r][1] = v.y; kw[mt][r][2] = v.z; kw[mt][r][3] = v.w;
#pragma unroll
          for (int q = 0; q < 4; ++q) kw10[mt][r][q] = kw[mt][r][q] >> 8;
        }
      }
    uint32_t cs[5];
    float qk_blk = qk_scale;
    if constexpr (BSCALE) {
      const int E = block_step_exp(ks4);
      step_scales<BITS>(cs, E);
      qk_blk = qk_scale * __int_as_float((127 - E) << 23);
    }
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 sv = ks4[i];
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        const int k8 = 2 * i + hk;
        constexpr int P01[4] = {key_pos(0), key_pos(2), key_pos(4), key_pos(6)};
        constexpr int P23[4] = {key_pos(1), key_pos(3), key_pos(5), key_pos(7)};
        uint32_t s01 = hk ? sv.z : sv.x, s23 = hk ? sv.w : sv.y;
        if constexpr (BITS == 2) {
          if constexpr (BSCALE) {
            s01 = hmul2_u(s01, cs[P01[k8 & 3]]);
            s23 = hmul2_u(s23, cs[P23[k8 & 3]]);
          } else {
            if (P01[k8 & 3] != 0) s01 = hmul2_u(s01, pow4_inv_h2(P01[k8 & 3]));
            if (P23[k8 & 3] != 0) s23 = hmul2_u(s23, pow4_inv_h2(P23[k8 & 3]));
          }
        } else {
          // INT4: pair 0 sits at nibble position 0, pair 1 at position 1
          if constexpr (BSCALE) {
            s01 = hmul2_u(s01, cs[0]);
            s23 = hmul2_u(s23, cs[1]);
          } else {
            s23 = hmul2_u(s23, pow16_inv_h2(1));
          }
        }
        const uint32_t r01 =
            hfma2_u(qz[k8][0], s01, hfma2_u(qhm[k8][0], s01, neg2_u(hmul2_u(qhm[k8][0], s01))));
        const uint32_t r23 =
            hfma2_u(qz[k8][1], s23, hfma2_u(qhm[k8][1], s23, neg2_u(hmul2_u(qhm[k8][1], s23))));
        const int wd = BITS == 2 ? k8 >> 2 : k8 >> 1;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const uint32_t wa = kw[mt][0][wd], wa10 = kw10[mt][0][wd];
          const uint32_t wb = kw[mt][1][wd], wb10 = kw10[mt][1][wd];
          uint32_t ak[4];
          if constexpr (BITS == 4) {
            if ((k8 & 1) == 0) {
              ak[0] = nib_pair<0>(wa, wa10); ak[1] = nib_pair<0>(wb, wb10);
              ak[2] = nib_pair<1>(wa, wa10); ak[3] = nib_pair<1>(wb, wb10);
            } else {
              ak[0] = nib_pair<2>(wa, wa10); ak[1] = nib_pair<2>(wb, wb10);
              ak[2] = nib_pair<3>(wa, wa10); ak[3] = nib_pair<3>(wb, wb10);
            }
          } else
          switch (k8 & 3) {
            case 0: ak[0] = key_pair<0>(wa, wa10); ak[1] = key_pair<0>(wb, wb10);
                    ak[2] = key_pair<1>(wa, wa10); ak[3] = key_pair<1>(wb, wb10); break;
            case 1: ak[0] = key_pair<2>(wa, wa10); ak[1] = key_pair<2>(wb, wb10);
                    ak[2] = key_pair<3>(wa, wa10); ak[3] = key_pair<3>(wb, wb10); break;
            case 2: ak[0] = key_pair<4>(wa, wa10); ak[1] = key_pair<4>(wb, wb10);
                    ak[2] = key_pair<5>(wa, wa10); ak[3] = key_pair<5>(wb, wb10); break;
            default: ak[0] = key_pair<6>(wa, wa10); ak[1] = key_pair<6>(wb, wb10);
                     ak[2] = key_pair<7>(wa, wa10); ak[3] = key_pair<7>(wb, wb10); break;
          }
          if (k8 == 0) {
            mma_16816(acc[mt], ak, r01, r23, zero4);
          } else {
            mma_16816_acc(acc[mt], ak, r01, r23);
          }
        }
      }
    }

    // Z = q'.z (issued after the Q.K MMAs, whose chains are longer).  The A operand is the loaded z quad {x, y, z, w} (pairs 0
    // and 1 of k-steps 2i and 2i+1) as it is: with the pair-0 columns of q'
    // for both k-steps, row gid of dza sums the pair-0 terms; with the pair-1
    // columns, row gid + 8 of dzb sums the pair-1 terms (the other rows are
    // unused).  Columns 2 tig, 2 tig + 1 give the hi, lo parts for head hs.
    float dza[4] = {0.f, 0.f, 0.f, 0.f}, dzb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 zv = kz4[i];
      const uint32_t za[4] = {zv.x, zv.y, zv.z, zv.w};
      mma_16816_acc(dza, za, qz[2 * i][0], qz[2 * i + 1][0]);
      mma_16816_acc(dzb, za, qz[2 * i][1], qz[2 * i + 1][1]);
    }

    // Scores of head hs, token gid + 8 j (j = 2 mt + r), log2 domain.
    const float zs = ((dza[0] + dza[1]) + (dzb[2] + dzb[3])) * inv_sigma;
    const float2 n01 = __half22float2(u32_as_half2(kn4.x)), n23 = __half22float2(u32_as_half2(kn4.y));
    const float nf[4] = {n01.x, n01.y, n23.x, n23.y};
    float sc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int mt = j >> 1, r = j & 1;
      const float qk = r ? acc[mt][2] + acc[mt][3] : acc[mt][0] + acc[mt][1];
      sc[j] = fmaf(qk, qk_blk, zs) * nf[j];
    }
    // Lazy rescaling (see the row layout).  Each lane tests its own scores;
    // only when some lane is past the threshold does the warp form the
    // block maximum of each head (lanes xor 4, 8, 16) and rescale.  Every
    // value of this lane belongs to head hs: the lane uses its own alpha.
    const float ml = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    if (__any_sync(0xffffffffu, ml > m_run + kLazyLog2)) {
      float mb = fmaxf(ml, __shfl_xor_sync(0xffffffffu, ml, 4));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
      const float m_new = fmaxf(m_run, mb);
      const float alpha = fast_exp2(m_run - m_new);
      l_run *= alpha;
      z_run *= alpha;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[mt][e] *= alpha;
      m_run = m_new;
    }

    // p~ = p s_V as (hi, lo) fp16 pairs: the 8x8 tile of token rows gid (+8)
    // and columns (head, limb); transposed, it is the P.V B operand.
    const float2 s01 = __half22float2(u32_as_half2(vs4.x)), s23 = __half22float2(u32_as_half2(vs4.y));
    const float2 z01 = __half22float2(u32_as_half2(vz4.x)), z23 = __half22float2(u32_as_half2(vz4.y));
    const float svj[4] = {s01.x, s01.y, s23.x, s23.y}, zvj[4] = {z01.x, z01.y, z23.x, z23.y};
    uint32_t bp[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float pt[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float sv = svj[2 * mt + r], zv = zvj[2 * mt + r];
        const float p = fast_exp2(sc[2 * mt + r] - m_run);
        l_run += p;
        z_run = fmaf(p, fmaf(Layout<BITS>::CENTER, sv, zv), z_run);
        pt[r] = p * sv;
      }
      const __half2 hh = __floats2half2_rn(pt[0], pt[1]);
      const float2 hv = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(pt[0] - hv.x, pt[1] - hv.y);
      bp[mt][0] = movmatrix_t(half2_as_u32(__lows2half2(hh, ll)));
      bp[mt][1] = movmatrix_t(half2_as_u32(__highs2half2(hh, ll)));
    }

#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      if constexpr (BITS == 2) {
        const uint4 vw = *reinterpret_cast<const uint4*>(vc + kh * 128 + lane * 4);
        const uint32_t wv[4] = {vw.x, vw.y, vw.z, vw.w};  // (p,hh) = (0,0) (0,1) (1,0) (1,1)
        uint32_t w10[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) w10[q] = wv[q] >> 10;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t av[4];
          value_frag(av, mt, wv, w10);
          mma_16816_acc(O[mt], av, bp[kh][0], bp[kh][1]);
        }
      } else {
        const uint4 v0 = *reinterpret_cast<const uint4*>(vc + kh * 256 + lane * 4);
        const uint4 v1 = *reinterpret_cast<const uint4*>(vc + kh * 256 + 128 + lane * 4);
        const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t ws[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ws[q] = wv[q] >> 8;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t av[4];
          value_frag4(av, mt, wv, ws);
          mma_16816_acc(O[mt], av, bp[kh][0], bp[kh][1]);
        }
      }
    }
    R.release(it, page_next, a);
  }
  if (it < R.n) {
    R.fail(it, a.status);
    m_run = -INFINITY;   // this warp's result is void; the status word says so
  }

  // Warp results: sums over the 8 lanes of a head (lanes xor 4, 8, 16).
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    l_run += __shfl_xor_sync(0xffffffffu, l_run, m);
    z_run += __shfl_xor_sync(0xffffffffu, z_run, m);
  }
  __syncthreads();   // every warp is done with its ring: reuse it for the merge
  if (tig < GQ) {
    if (gid == 0) {
      E.m[warp][tig] = m_run;
      E.l[warp][tig] = l_run;
      E.z[warp][tig] = z_run;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {   // undo the value rows' 2^(2p - 9)
      E.o[warp][tig][16 * mt + gid] = (O[mt][0] + O[mt][1]) * row_unscale<BITS>(mt, 0);
      E.o[warp][tig][16 * mt + gid + 8] = (O[mt][2] + O[mt][3]) * row_unscale<BITS>(mt, 1);
    }
  }
}

// ------------------------------------------------------------------- rows
// Groups of 8 query heads.  Lane (gid, tig):
//  * Q.K A operand: rows gid (hi part) and gid + 8 (lo part) of q~ for head
//    gid; B operand: key codes of token 8 nt + gid, n-tiles nt = 0..3;
//  * scores and softmax: head gid, tokens 8 nt + 2 tig and + 1;
//  * P.V: channels on M, the 8 heads on N, one n-tile per limb of p~.
template <int GQ, bool BSCALE, int BITS, class Ring>
__device__ __forceinline__ void packed_rows(const DecodeArgs& a, const Ring& R,
                                            MergeSmem<GQ, NW>& E, long long qrow0, int nh) {
  static_assert(GQ == 8, "the row layout serves groups of 8 query heads");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  // this thread's head (a padding head works on the last active head's query)
  const int head = min(gid, nh - 1);
  using RL = typename Layout<BITS>::RL;
  constexpr int LW = BITS == 2 ? 2 : 4;   // key words per token and lane
  // The query's loads go out first, then the ring's first copies, which
  // travel while the query is prepared (INT4: the copies first, which keeps
  // its instantiations free of spills).
  float4 qv[8];
  if (a.q_raw != nullptr) {   // fused step: rotate the CTA's queries here
    RawQueries<GQ> raw;
    load_raw_queries<GQ>(a, qrow0, nh, raw);
    R.start(a);
    const float* qs = stage_rotated_queries<GQ>(a, raw, dyn_smem() + smem_bytes<GQ, BITS>());
    load_query(qv, qs + head * kD, tig);
  } else if constexpr (BITS == 2) {
    load_query(qv, a.q_rot + (qrow0 + head) * kD, tig);
    R.start(a);
  } else {
    R.start(a);
    load_query(qv, a.q_rot + (qrow0 + head) * kD, tig);
  }

  // Query fragments of this thread's head, staged by warp 0 in shared memory
  // after the ring's barriers (all warps of the CTA serve the same 8 heads);
  // every k-step reads its quad back, which keeps the kernel at 128 registers
  // and 4 CTAs per SM.
  uint4* const qs = reinterpret_cast<uint4*>(dyn_smem() + Layout<BITS>::SMEM);
  float inv_sigma;
  {
    float qf[32];
    const float sigma = scale_query(qf, qv, a);
    inv_sigma = ldexpf(1.0f, -ilogbf(sigma));
    if (warp == 0) {
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) {
        uint32_t f[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float x0 = qf[4 * k8 + 2 * j], x1 = qf[4 * k8 + 2 * j + 1];
          const __half2 hh = __floats2half2_rn(x0, x1);
          const float2 hv = __half22float2(hh);
          f[2 * j] = half2_as_u32(hh);
          f[2 * j + 1] = half2_as_u32(__floats2half2_rn(x0 - hv.x, x1 - hv.y));
        }
        qs[k8 * 32 + lane] = make_uint4(f[0], f[1], f[2], f[3]);
      }
    }
  }
  __syncthreads();
  // the Q.K sums carry 2^-24 (subnormal key codes) and sigma
  const float qk_scale = 16777216.0f * inv_sigma;

  float O[2][8][4];   // P.V accumulators of the hi and lo limbs of p~
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[t][mt][e] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f, z_run = 0.0f;

  int it = 0;
  for (; it < R.n; ++it) {
    if (!R.wait(it)) break;
    const int page_next = R.page_of(it + Ring::NSTAGE, a);
    const uint8_t* st = R.slot(it);
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(st + RL::KC);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + RL::VC);
    const uint4* ks4 = reinterpret_cast<const uint4*>(st + RL::KS) + tig * 4;
    const uint4* kz4 = reinterpret_cast<const uint4*>(st + RL::KZ) + tig * 4;
    // norms, value steps and zeros: halves 0..3 are tokens 2 tig + 8 nt,
    // halves 4..7 tokens 2 tig + 1 + 8 nt (nt = 0..3)
    const uint4 kn8 = *reinterpret_cast<const uint4*>(st + RL::KN + 16 * tig);
    const uint4 vs8 = *reinterpret_cast<const uint4*>(st + RL::VS + 16 * tig);
    const uint4 vz8 = *reinterpret_cast<const uint4*>(st + RL::VZ + 16 * tig);

    float dz[4] = {0.f, 0.f, 0.f, 0.f};

    // Q.K^T, k-step outer: q~ fragment for k-step k8, then the 4 n-tiles.
    uint32_t kw[4][LW], kw10[4][LW];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      if constexpr (BITS == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(kc + (8 * nt + gid) * 8 + 2 * tig);
        kw[nt][0] = v.x; kw[nt][1] = v.y;
        kw10[nt][0] = v.x >> 10; kw10[nt][1] = v.y >> 10;
      } else {
        const uint4 v = *reinterpret_cast<const uint4*>(kc + (8 * nt + gid) * 16 + 4 * tig);
        kw[nt][0] = v.x; kw[nt][1] = v.y; kw[nt][2] = v.z; kw[nt][3] = v.w;
#pragma unroll
        for (int q = 0; q < 4; ++q) kw10[nt][q] = kw[nt][q] >> 8;
      }
    }
    // The Q.K accumulators start from zero (not from Z) so their MMA chains
    // do not wait for the Z chain; Z joins each score below.
    uint32_t cs[5];
    float qk_blk = qk_scale;
    if constexpr (BSCALE) {
      const int E = block_step_exp(ks4);
      step_scales<BITS>(cs, E);
      qk_blk = qk_scale * __int_as_float((127 - E) << 23);
    }
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 sv = ks4[i];
      const uint4 zv = kz4[i];
#pragma unroll
      for (int hk = 0; hk < 2; ++hk) {
        const int k8 = 2 * i + hk;
        const uint4 q4 = qs[k8 * 32 + lane];
        const uint32_t aqk[4] = {q4.x, q4.y, q4.z, q4.w};
        // Z = q'.z of the block: rows g (hi) and g+8 (lo), every column alike.
        mma_16816_acc(dz, aqk, hk ? zv.z : zv.x, hk ? zv.w : zv.y);
        // key step of the pair's channels times 4^-p of the pair's code
        // position (exact: a power of two)
        constexpr int P01[4] = {key_pos(0), key_pos(2), key_pos(4), key_pos(6)};
        constexpr int P23[4] = {key_pos(1), key_pos(3), key_pos(5), key_pos(7)};
        uint32_t s01 = hk ? sv.z : sv.x, s23 = hk ? sv.w : sv.y;
        if constexpr (BITS == 2) {
          if constexpr (BSCALE) {
            s01 = hmul2_u(s01, cs[P01[k8 & 3]]);
            s23 = hmul2_u(s23, cs[P23[k8 & 3]]);
          } else {
            if (P01[k8 & 3] != 0) s01 = hmul2_u(s01, pow4_inv_h2(P01[k8 & 3]));
            if (P23[k8 & 3] != 0) s23 = hmul2_u(s23, pow4_inv_h2(P23[k8 & 3]));
          }
        } else {
          // INT4: pair 0 sits at nibble position 0, pair 1 at position 1
          if constexpr (BSCALE) {
            s01 = hmul2_u(s01, cs[0]);
            s23 = hmul2_u(s23, cs[1]);
          } else {
            s23 = hmul2_u(s23, pow16_inv_h2(1));
          }
        }
        uint32_t at[4];
        at[0] = hmul2_u(aqk[0], s01);
        at[1] = hfma2_u(aqk[1], s01, hfma2_u(aqk[0], s01, neg2_u(at[0])));
        at[2] = hmul2_u(aqk[2], s23);
        at[3] = hfma2_u(aqk[3], s23, hfma2_u(aqk[2], s23, neg2_u(at[2])));
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int wd = BITS == 2 ? k8 >> 2 : k8 >> 1;
          const uint32_t w = kw[nt][wd], w10 = kw10[nt][wd];
          uint32_t b0v, b1v;
          if constexpr (BITS == 4) {
            if ((k8 & 1) == 0) {
              b0v = nib_pair<0>(w, w10); b1v = nib_pair<1>(w, w10);
            } else {
              b0v = nib_pair<2>(w, w10); b1v = nib_pair<3>(w, w10);
            }
          } else
          switch (k8 & 3) {
            case 0: b0v = key_pair<0>(w, w10); b1v = key_pair<1>(w, w10); break;
            case 1: b0v = key_pair<2>(w, w10); b1v = key_pair<3>(w, w10); break;
            case 2: b0v = key_pair<4>(w, w10); b1v = key_pair<5>(w, w10); break;
            default: b0v = key_pair<6>(w, w10); b1v = key_pair<7>(w, w10); break;
          }
          if (k8 == 0) {
            mma_16816(acc[nt], at, b0v, b1v, zero4);
          } else {
            mma_16816_acc(acc[nt], at, b0v, b1v);
          }
        }
      }
    }

    // Scores of this thread's tokens (log2 domain): hi row + lo row, times
    // the token norm.  Token j of the thread: n-tile nt(j), tokens 2tig, +1.
    // Z of this thread's head (hi row + lo row); the Q.K sums carry 2^-24
    const float zs = (dz[0] + dz[2]) * inv_sigma;
    float ne[4], no[4];
    unpack_h4(ne, kn8.x, kn8.y);
    unpack_h4(no, kn8.z, kn8.w);
    float sc[8];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      sc[2 * nt] = fmaf(acc[nt][0] + acc[nt][2], qk_blk, zs) * ne[nt];
      sc[2 * nt + 1] = fmaf(acc[nt][1] + acc[nt][3], qk_blk, zs) * no[nt];
    }

    // Online softmax for this thread's head.
    float ml = sc[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) ml = fmaxf(ml, sc[i]);
    // Lazy rescaling: the running max moves only when a score exceeds it by
    // more than 2^kLazyLog2, so p = 2^(score - m_run) stays below 2^kLazyLog2
    // (well inside fp16 and fp32) and the accumulators are rescaled rarely.
    // Each lane tests its own scores; only then are the heads' block maxima
    // formed (lanes xor 1, 2).
    if (__any_sync(0xffffffffu, ml > m_run + kLazyLog2)) {
      float mb = fmaxf(ml, __shfl_xor_sync(0xffffffffu, ml, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      const float m_new = fmaxf(m_run, mb);
      const float alpha = fast_exp2(m_run - m_new);
      l_run *= alpha;
      z_run *= alpha;
      // the P.V columns 2 tig, 2 tig + 1 of this lane are heads 2 tig, 2 tig + 1
      const float al_a = __shfl_sync(0xffffffffu, alpha, 8 * tig);
      const float al_b = __shfl_sync(0xffffffffu, alpha, 8 * tig + 4);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          O[t][mt][0] *= al_a; O[t][mt][1] *= al_b;
          O[t][mt][2] *= al_a; O[t][mt][3] *= al_b;
        }
      m_run = m_new;
    }

    float se[4], so[4], ze[4], zo[4];
    unpack_h4(se, vs8.x, vs8.y);
    unpack_h4(so, vs8.z, vs8.w);
    unpack_h4(ze, vz8.x, vz8.y);
    unpack_h4(zo, vz8.z, vz8.w);
    float pt[8];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = fast_exp2(sc[2 * nt] - m_run);
      const float p1 = fast_exp2(sc[2 * nt + 1] - m_run);
      l_run += p0 + p1;
      z_run = fmaf(p0, fmaf(Layout<BITS>::CENTER, se[nt], ze[nt]), z_run);
      z_run = fmaf(p1, fmaf(Layout<BITS>::CENTER, so[nt], zo[nt]), z_run);
      pt[2 * nt] = p0 * se[nt];
      pt[2 * nt + 1] = p1 * so[nt];
    }

    // P~ as the B operand of P.V: k-half kh uses n-tiles 2kh (tokens 2tig,
    // 2tig+1) and 2kh+1 (2tig+8, 2tig+9); bp holds the hi limb, bq the lo.
    uint32_t bp[2][2], bq[2][2];
#pragma unroll
    for (int kh = 0; kh < 2; ++kh)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float x0 = pt[4 * kh + 2 * r], x1 = pt[4 * kh + 2 * r + 1];
        const __half2 hv = __floats2half2_rn(x0, x1);
        const float2 hf2 = __half22float2(hv);
        bp[kh][r] = half2_as_u32(hv);
        bq[kh][r] = half2_as_u32(__floats2half2_rn(x0 - hf2.x, x1 - hf2.y));
      }

#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      if constexpr (BITS == 2) {
        const uint4 vw = *reinterpret_cast<const uint4*>(vc + kh * 128 + lane * 4);
        const uint32_t wv[4] = {vw.x, vw.y, vw.z, vw.w};  // (p,hh) = (0,0) (0,1) (1,0) (1,1)
        uint32_t w10[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) w10[q] = wv[q] >> 10;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t av[4];
          value_frag(av, mt, wv, w10);
          mma_16816_acc(O[0][mt], av, bp[kh][0], bp[kh][1]);
          mma_16816_acc(O[1][mt], av, bq[kh][0], bq[kh][1]);
        }
      } else {
        const uint4 v0 = *reinterpret_cast<const uint4*>(vc + kh * 256 + lane * 4);
        const uint4 v1 = *reinterpret_cast<const uint4*>(vc + kh * 256 + 128 + lane * 4);
        const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t ws[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ws[q] = wv[q] >> 8;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t av[4];
          value_frag4(av, mt, wv, ws);
          mma_16816_acc(O[0][mt], av, bp[kh][0], bp[kh][1]);
          mma_16816_acc(O[1][mt], av, bq[kh][0], bq[kh][1]);
        }
      }
    }
    R.release(it, page_next, a);
  }
  if (it < R.n) {
    R.fail(it, a.status);
    m_run = -INFINITY;   // this warp's result is void; the status word says so
  }

  // Warp results: sums over the lanes of a head, limbs folded.
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  z_run += __shfl_xor_sync(0xffffffffu, z_run, 1);
  z_run += __shfl_xor_sync(0xffffffffu, z_run, 2);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) O[0][mt][e] += O[1][mt][e];
  __syncthreads();   // every warp is done with its ring: reuse it for the merge
  if (tig == 0) {
    E.m[warp][gid] = m_run;
    E.l[warp][gid] = l_run;
    E.z[warp][gid] = z_run;
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int nc = 2 * tig + e;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {   // undo the value rows' 2^(2p - 9)
      E.o[warp][nc][16 * mt + gid] = O[0][mt][e] * row_unscale<BITS>(mt, 0);
      E.o[warp][nc][16 * mt + gid + 8] = O[0][mt][2 + e] * row_unscale<BITS>(mt, 1);
    }
  }
}

// --------------------------------------------------------------- residual
template <int GQ, bool PAGED>
__device__ __forceinline__ void residual_split(const DecodeArgs& a, MergeSmem<GQ, NW>& E,
                                               long long row, long long qrow0, int nh, int b) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n_res = a.n_res;
  if constexpr (PAGED) {
    n_res = __ldg(a.seq_res + b);
    if (n_res < 0 || n_res > kR) {
      if (threadIdx.x == 0) record_error(a.status, kDevErrBadPaged);
      n_res = 0;
    }
  }
  if (!PAGED && a.k_new != nullptr) {
    // Fused step: the new token goes to residual slot n_res - 1 first,
    // rotated and scaled as rotate_scale_k_kernel does it (warp 0) and its
    // value copied (warp 1); only this CTA reads the row's residual window.
    const long long tok = row * kR + (n_res - 1);
    if (warp == 0) {
      const KeyScale ks{a.flags, a.norm_target};
      float s_all = 0.0f;
      if (ks.flags & OSCAR_NORM_ALL_HEADS)
        s_all = all_heads_sq(a.k_new + (long long)b * a.Hkv * kD, (long long)kD, a.Hkv, lane);
      const uint2 raw = reinterpret_cast<const uint2*>(a.k_new + row * kD)[lane];
      float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
      const float norm = rotate_scale_key(x, lane, ks, s_all);
      reinterpret_cast<uint2*>(const_cast<uint16_t*>(a.k_res) + tok * kD)[lane] = pack_bf16x4(x);
      if (lane == 0) const_cast<__half*>(a.k_res_norm)[tok] = __float2half_rn(norm);
    } else if (warp == 1) {
      reinterpret_cast<uint2*>(const_cast<uint16_t*>(a.v_res) + tok * kD)[lane] =
          reinterpret_cast<const uint2*>(a.v_new + row * kD)[lane];
    }
    __syncthreads();
  }
  // Unit-norm bf16 keys times their fp16 norms, bf16 values; CUDA cores.
  float mr[GQ], lr[GQ], orr[GQ][4];
#pragma unroll
  for (int j = 0; j < GQ; ++j) {
    mr[j] = -INFINITY;
    lr[j] = 0.0f;
    orr[j][0] = orr[j][1] = orr[j][2] = orr[j][3] = 0.0f;
  }
  if constexpr (GQ == 8) {
    // Groups of 8: warp w takes the window's tokens 32 w .. 32 w + 31 (the
    // window holds at most NW * 32 = R of them), one pass, no cross-lane sums
    // for the scores (8 heads would need 8 reduction chains per token):
    //  * Q.K with a token per lane: lane t reads its key row and forms all GQ
    //    dot products over the 128 channels against the queries, which every
    //    lane reads from shared memory (the ring area, unused by this CTA);
    //  * the warp's maximum and sum of each head's weights (five shuffles);
    //  * P.V with four channels per lane: each token's weights reach the
    //    lanes by shuffle, its value row is one 8-byte load per lane.
    static_assert(kR == NW * 32, "one 32-token slice of the window per warp");
    float* qs = reinterpret_cast<float*>(dyn_smem());   // [GQ][128] fp32
    for (int i = threadIdx.x; i < GQ * 32; i += NW * 32) {   // every lane of a warp alike
      const int j = min(i >> 5, nh - 1);
      const float4 v = a.q_raw != nullptr ? rotated_query(a, qrow0 + j, lane)
                                          : reinterpret_cast<const float4*>(a.q_rot + (qrow0 + j) * kD)[lane];
      reinterpret_cast<float4*>(qs)[i] = v;
    }
    __syncthreads();
    const int t0 = 32 * warp, nt = min(32, n_res - t0);   // this warp's tokens (warp-uniform)
    if (nt > 0) {
      const bool mine = lane < nt;
      const long long tok = row * kR + t0 + (mine ? lane : 0);
      float d[GQ];
#pragma unroll
      for (int j = 0; j < GQ; ++j) d[j] = 0.0f;
      const uint4* kr = reinterpret_cast<const uint4*>(a.k_res + tok * kD);
      const float4* q4 = reinterpret_cast<const float4*>(qs);
#pragma unroll 4
      for (int c8 = 0; c8 < kD / 8; ++c8) {
        const uint4 u = kr[c8];
        const float k8[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                             bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
          const float4 qa = q4[j * 32 + 2 * c8], qb = q4[j * 32 + 2 * c8 + 1];
          d[j] = fmaf(k8[0], qa.x, d[j]); d[j] = fmaf(k8[1], qa.y, d[j]);
          d[j] = fmaf(k8[2], qa.z, d[j]); d[j] = fmaf(k8[3], qa.w, d[j]);
          d[j] = fmaf(k8[4], qb.x, d[j]); d[j] = fmaf(k8[5], qb.y, d[j]);
          d[j] = fmaf(k8[6], qb.z, d[j]); d[j] = fmaf(k8[7], qb.w, d[j]);
        }
      }
      const float nrm = __half2float(a.k_res_norm[tok]);
      float p[GQ];
#pragma unroll
      for (int j = 0; j < GQ; ++j) {
        const float sc = mine ? d[j] * nrm * a.scale_log2 : -INFINITY;
        float m = sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        p[j] = fast_exp2(sc - m);
        float l = p[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        mr[j] = m;
        lr[j] = l;
      }
      const uint2* vr = reinterpret_cast<const uint2*>(a.v_res + (row * kR + t0) * kD) + lane;
#pragma unroll 4
      for (int u = 0; u < nt; ++u) {
        const uint2 w = vr[u * (kD / 4)];
        const float v4[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
          const float pj = __shfl_sync(0xffffffffu, p[j], u);
#pragma unroll
          for (int i = 0; i < 4; ++i) orr[j][i] = fmaf(pj, v4[i], orr[j][i]);
        }
      }
    }
  } else {
    // Groups of up to 4: channels 4l .. 4l + 3 per lane, warp w takes tokens
    // 4 w .. 4 w + 3, then 4 (w + NW) .., four at a time: their 4 x GQ dot
    // products reduce across the warp as independent chains, and the running
    // maximum is raised once per four tokens.
    float qv[GQ][4];
#pragma unroll
    for (int j = 0; j < GQ; ++j) {
      const long long qj = qrow0 + min(j, nh - 1);
      const float4 v = a.q_raw != nullptr ? rotated_query(a, qj, lane)
                                          : reinterpret_cast<const float4*>(a.q_rot + qj * kD)[lane];
      qv[j][0] = v.x; qv[j][1] = v.y; qv[j][2] = v.z; qv[j][3] = v.w;
    }
    constexpr int TU = 4;
    for (int t0 = TU * warp; t0 < n_res; t0 += TU * NW) {
      float k4[TU][4], v4[TU][4], nrm[TU];
#pragma unroll
      for (int u = 0; u < TU; ++u) {
        const long long tok = row * kR + min(t0 + u, n_res - 1);
        const uint2 kr = reinterpret_cast<const uint2*>(a.k_res + tok * kD)[lane];
        const uint2 vr = reinterpret_cast<const uint2*>(a.v_res + tok * kD)[lane];
        k4[u][0] = bf16_lo(kr.x); k4[u][1] = bf16_hi(kr.x); k4[u][2] = bf16_lo(kr.y); k4[u][3] = bf16_hi(kr.y);
        v4[u][0] = bf16_lo(vr.x); v4[u][1] = bf16_hi(vr.x); v4[u][2] = bf16_lo(vr.y); v4[u][3] = bf16_hi(vr.y);
        nrm[u] = __half2float(a.k_res_norm[tok]);
      }
      float d[TU][GQ];
#pragma unroll
      for (int u = 0; u < TU; ++u)
#pragma unroll
        for (int j = 0; j < GQ; ++j)
          d[u][j] = qv[j][0] * k4[u][0] + qv[j][1] * k4[u][1] + qv[j][2] * k4[u][2] + qv[j][3] * k4[u][3];
#pragma unroll
      for (int m = 16; m > 0; m >>= 1)
#pragma unroll
        for (int u = 0; u < TU; ++u)
#pragma unroll
          for (int j = 0; j < GQ; ++j) d[u][j] += __shfl_xor_sync(0xffffffffu, d[u][j], m);
#pragma unroll
      for (int j = 0; j < GQ; ++j) {
        float sc[TU], m_new = mr[j];
#pragma unroll
        for (int u = 0; u < TU; ++u) {
          sc[u] = t0 + u < n_res ? d[u][j] * nrm[u] * a.scale_log2 : -INFINITY;
          m_new = fmaxf(m_new, sc[u]);
        }
        const float al = fast_exp2(mr[j] - m_new);
        lr[j] *= al;
#pragma unroll
        for (int i = 0; i < 4; ++i) orr[j][i] *= al;
#pragma unroll
        for (int u = 0; u < TU; ++u) {
          const float p = fast_exp2(sc[u] - m_new);
          lr[j] += p;
#pragma unroll
          for (int i = 0; i < 4; ++i) orr[j][i] = fmaf(p, v4[u][i], orr[j][i]);
        }
        mr[j] = m_new;
      }
    }
  }
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < GQ; ++j) {
      E.m[warp][j] = mr[j];
      E.l[warp][j] = lr[j];
      E.z[warp][j] = 0.0f;
    }
  }
#pragma unroll
  for (int j = 0; j < GQ; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) E.o[warp][j][4 * lane + i] = orr[j][i];
}

// Log-sum-exp combine of the `parts` partial records of each of the CTA's GQ
// query heads (flash-decoding): m* = max_s m_s, out = sum_s 2^(m_s - m*) o_s /
// sum_s 2^(m_s - m*) l_s, scores in the log2 domain.  Partials that saw no
// token carry m = -inf and drop out; a row with none gives zeros.  Run by
// the row's last CTA, after every other CTA's records are visible.  Warp w
// takes head w (and w + 4 for groups of 8); for groups smaller than 4 the
// warps of a head split its partials and add their sums in shared memory.
// The records were written by other CTAs during this launch, so they are
// read past L1 (ld.global.cg), and the combine sits on the row's critical
// path, so its loads are issued in few round trips: each lane takes the
// (m, l) pair of up to two partials in one pass, and the outputs are read
// kCombineBatch partials at a time, all loads of a batch in flight before
// the first is used.  Lane l holds channels 4 l .. 4 l + 3, summed in four
// interleaved fp32 chains (partial q into chain q mod 4, in order of q).
constexpr int kCombineBatch = 16;

template <int GQ>
__device__ __forceinline__ void row_combine(const DecodeArgs& a, MergeSmem<GQ, NW>& E,
                                            long long qrow0, int nh, int parts) {
  constexpr int HPW = GQ > NW ? GQ / NW : 1;   // heads per warp
  constexpr int PG = GQ >= NW ? 1 : NW / GQ;   // warps per head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    const int j = GQ >= NW ? warp + NW * hh : warp % GQ;
    const int pg = GQ >= NW ? 0 : warp / GQ;
    if (j >= nh) continue;   // a padding head (warp-uniform): no partials, no output
    const float* r0 = a.ws + (qrow0 + j) * parts * kRecFloats;
    const int np = (parts - pg + PG - 1) / PG;   // this warp's partials pg + PG i
    auto rec = [&](int i) { return r0 + (long long)(pg + PG * i) * kRecFloats; };
    // (m, l) of partials lane and lane + 32 in registers; the rest (more than
    // 64 partials per warp) are read again where needed.
    float2 ml0 = make_float2(-INFINITY, 0.0f), ml1 = make_float2(-INFINITY, 0.0f);
    if (lane < np) ml0 = __ldcg(reinterpret_cast<const float2*>(rec(lane)));
    if (lane + 32 < np) ml1 = __ldcg(reinterpret_cast<const float2*>(rec(lane + 32)));
    // the first batch of outputs is loaded with the (m, l) pairs: its loads
    // do not wait for m*
    const int nfast = min(np, 64);
    float4 x[kCombineBatch];
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k)
      if (k < nfast) x[k] = __ldcg(reinterpret_cast<const float4*>(rec(k) + 4) + lane);
    // m* over all the row's partials (for groups smaller than 4 the warps of
    // a head add their sums unscaled, so they share one m*)
    float M = fmaxf(ml0.x, ml1.x);
    if constexpr (PG == 1) {
      for (int i = lane + 64; i < np; i += 32) M = fmaxf(M, __ldcg(rec(i)));
    } else {
      for (int s = lane; s < parts; s += 32) M = fmaxf(M, __ldcg(r0 + (long long)s * kRecFloats));
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    float L = 0.0f;
    float4 op[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) op[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      const float w0 = ml0.x == -INFINITY ? 0.0f : fast_exp2(ml0.x - M);
      const float w1 = ml1.x == -INFINITY ? 0.0f : fast_exp2(ml1.x - M);
      L = fmaf(w0, ml0.y, L);
      L = fmaf(w1, ml1.y, L);
      for (int i0 = 0; i0 < nfast; i0 += kCombineBatch) {
        if (i0 > 0) {
#pragma unroll
          for (int k = 0; k < kCombineBatch; ++k)
            if (i0 + k < nfast)
              x[k] = __ldcg(reinterpret_cast<const float4*>(rec(i0 + k) + 4) + lane);
        }
#pragma unroll
        for (int k = 0; k < kCombineBatch; ++k) {
          const int q = i0 + k;
          const float wq = __shfl_sync(0xffffffffu, q < 32 ? w0 : w1, q & 31);
          if (q < nfast) {
            op[k & 3].x = fmaf(wq, x[k].x, op[k & 3].x); op[k & 3].y = fmaf(wq, x[k].y, op[k & 3].y);
            op[k & 3].z = fmaf(wq, x[k].z, op[k & 3].z); op[k & 3].w = fmaf(wq, x[k].w, op[k & 3].w);
          }
        }
      }
      // partials beyond 64 of this warp (more than 64 splits): four at a time,
      // each lane adding the l of its own partials
      for (int i0 = 64; i0 < np; i0 += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = i0 + k;
          if (i < np) {
            const float ms = __ldcg(rec(i));
            const float wq = ms == -INFINITY ? 0.0f : fast_exp2(ms - M);
            if (((i - lane) & 31) == 0) L = fmaf(wq, __ldcg(rec(i) + 1), L);
            const float4 x = __ldcg(reinterpret_cast<const float4*>(rec(i) + 4) + lane);
            op[k].x = fmaf(wq, x.x, op[k].x); op[k].y = fmaf(wq, x.y, op[k].y);
            op[k].z = fmaf(wq, x.z, op[k].z); op[k].w = fmaf(wq, x.w, op[k].w);
          }
        }
      }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) L += __shfl_xor_sync(0xffffffffu, L, m);
    const float4 o = make_float4((op[0].x + op[1].x) + (op[2].x + op[3].x),
                                 (op[0].y + op[1].y) + (op[2].y + op[3].y),
                                 (op[0].z + op[1].z) + (op[2].z + op[3].z),
                                 (op[0].w + op[1].w) + (op[2].w + op[3].w));
    if constexpr (PG == 1) {
      reinterpret_cast<float4*>(a.out + (qrow0 + j) * kD)[lane] =
          L > 0.0f ? make_float4(o.x / L, o.y / L, o.z / L, o.w / L)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      if (lane == 0) E.l[warp][0] = L;
      reinterpret_cast<float4*>(E.o[warp][0])[lane] = o;
    }
  }
  if constexpr (PG > 1) {
    __syncthreads();
    const int c = threadIdx.x;   // NW * 32 == kD channels, one per thread
#pragma unroll
    for (int j = 0; j < GQ; ++j) {
      if (j >= nh) break;
      float Lt = 0.0f, oc = 0.0f;
#pragma unroll
      for (int g = 0; g < PG; ++g) {
        Lt += E.l[j + GQ * g][0];
        oc += E.o[j + GQ * g][0][c];
      }
      a.out[(qrow0 + j) * kD + c] = Lt > 0.0f ? oc / Lt : 0.0f;
    }
  }
}

// 4 CTAs per SM (128 registers), except the INT4 row layout (3).
// BSCALE: per-block step scale (caches with the all-heads norm scope);
// BITS: code width of the records (2, or the INT4 option); PAD: query groups
// of another size than GQ (padding heads, or slices of a group above 8), so
// that the kernels of whole groups keep their code.
template <int GQ, bool PAGED, bool BSCALE, int BITS, bool PAD>
__global__ void __launch_bounds__(NW * 32, GQ <= 4 || BITS == 2 ? 4 : 3) decode_int2_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  auto& E = *reinterpret_cast<MergeSmem<GQ, NW>*>(smem);
  static_assert(sizeof(MergeSmem<GQ, NW>) <= NW * Layout<BITS>::NSTAGE * Layout<BITS>::RL::BYTES,
                "merge area");
  // One-dimensional grid, the residual CTAs first: CTA L < rows is row L's
  // residual split, and the others take the packed splits row by row.  So
  // every residual CTA starts in the first wave, where its work (up to a
  // full 128-token window) runs beside the packed CTAs instead of after
  // them at the end of a many-wave grid.  A row is one slice of up to GQ of
  // the g query heads that share KV head h of sequence b (slices = ceil(g /
  // GQ)); the last slice of a group that GQ does not divide, or a group
  // smaller than GQ, has padding heads, which the CTA works but neither
  // merges nor outputs.
  const long long rows = (long long)a.B * a.Hkv * (PAD ? a.slices : 1);
  long long vrow;
  int split;
  if ((long long)blockIdx.x < rows) {
    vrow = blockIdx.x;
    split = a.num_splits;
  } else {
    const long long q = (long long)blockIdx.x - rows;
    vrow = q / a.num_splits;
    split = (int)(q - vrow * a.num_splits);
  }
  long long row = vrow;   // the cache row (b, h)
  int sl = 0;
  if (PAD && a.slices > 1) {
    row = vrow / a.slices;
    sl = (int)(vrow - row * a.slices);
  }
  const int b = (int)(row / a.Hkv), h = (int)(row - (long long)b * a.Hkv);
  const int g = PAD ? a.Hq / a.Hkv : GQ;
  const int nh = PAD ? min(GQ, g - GQ * sl) : GQ;   // active heads of the slice
  const long long qrow0 = (long long)b * a.Hq + (long long)h * g + GQ * sl;  // first query head
  // (padded groups) kept in shared memory through the block loop
  __shared__ int s_nh;
  if (PAD && threadIdx.x == 0) s_nh = nh;

  if (split < a.num_splits) {
    if (PAGED && split >= paged_splits_used(a, row_blocks<PAGED>(a, b))) {
      // A split that a short sequence of a paged batch does not fill skips
      // the query and writes an empty partial, which the combine ignores.
      if (threadIdx.x < NW * GQ) E.m[threadIdx.x / GQ][threadIdx.x % GQ] = -INFINITY;
    } else {
      const WarpRing<PAGED, BITS> R = make_ring<PAGED, BITS>(a, smem, b, h, split);
      if constexpr (GQ <= 4) {
        packed_cols<GQ, BSCALE, BITS>(a, R, E, qrow0, nh);
      } else {
        packed_rows<GQ, BSCALE, BITS>(a, R, E, qrow0, nh);
      }
    }
  } else {
    residual_split<GQ, PAGED>(a, E, row, qrow0, nh, b);
  }
  __syncthreads();
  const int parts = a.num_splits + 1;
  const int nh_e = PAD ? s_nh : GQ;
  cta_merge_write<GQ, NW>(E, a.ws + (qrow0 * parts + split) * kRecFloats,
                          (long long)parts * kRecFloats, nh_e);
  // Arrival: after the CTA barrier, one thread counts the CTA in on the
  // row's counter with one acquire-release atomic at GPU scope, which makes
  // the CTA's records visible with the count.  The CTA that brings the count
  // to `parts` has acquired the other CTAs' records with it; it combines the
  // row and sets the counter back to zero for the next call on this
  // workspace.  A count
  // already at or above `parts` means the counters were not zero when the
  // call began: reported, and the row is left uncombined.
  __shared__ int last_cta;
  __syncthreads();
  if (threadIdx.x == 0) {
    // acquire-release at GPU scope: the CTA's records (ordered before this
    // thread by the barrier) are released with the count, and the CTA that
    // completes it acquires every other CTA's records before its reads
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev) : "l"(a.row_count + vrow) : "memory");
    if (prev >= (unsigned)parts) record_error(a.status, kDevErrArrival);
    last_cta = prev == (unsigned)(parts - 1);
    if (last_cta) a.row_count[vrow] = 0u;
  }
  __syncthreads();
  if (!last_cta) return;
  row_combine<GQ>(a, E, qrow0, nh_e, parts);
}

// Opt in to the kernel's dynamic shared memory (above 48 KB for INT2), once
// per instantiation and device.
template <int GQ, bool PAGED, bool BSCALE, int BITS, bool PAD>
cudaError_t allow_smem() {
  static int done[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 128 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(decode_int2_kernel<GQ, PAGED, BSCALE, BITS, PAD>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<GQ, BITS>() + kQRotStage);
  if (e == cudaSuccess && dev >= 0 && dev < 128) done[dev] = 1;
  return e;
}

template <int GQ, bool PAGED, bool BSCALE, int BITS, bool PAD>
cudaError_t launch_k(const DecodeArgs& a, cudaStream_t s) {
  cudaError_t e0 = allow_smem<GQ, PAGED, BSCALE, BITS, PAD>();
  if (e0 != cudaSuccess) return e0;
  const long long ctas = (long long)a.B * a.Hkv * a.slices * (a.num_splits + 1);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)ctas);
  const int smem = smem_bytes<GQ, BITS>() + (a.q_raw != nullptr ? kQRotStage : 0);
  decode_int2_kernel<GQ, PAGED, BSCALE, BITS, PAD><<<grid, NW * 32, smem, s>>>(a);
  return cudaGetLastError();
}

// This translation unit builds the kernels of whole groups (g = 1, 2, 4, 8);
// decode_int2_pad.cu includes this file with OSCAR_DECODE_PAD_TU defined and
// builds the padded ones (groups of 4 or 8 heads per CTA for the other g),
// so the two compile in parallel.
#ifdef OSCAR_DECODE_PAD_TU
constexpr bool kPadTU = true;
#else
constexpr bool kPadTU = false;
#endif

template <bool PAGED, bool BSCALE, int BITS>
cudaError_t launch_p(const DecodeArgs& a, cudaStream_t s) {
  if (a.slices != decode_slices(a.Hq / a.Hkv)) return cudaErrorInvalidValue;
  if constexpr (kPadTU) {
    switch (decode_group_width(a.Hq / a.Hkv)) {
      case 4: return launch_k<4, PAGED, BSCALE, BITS, true>(a, s);
      case 8: return launch_k<8, PAGED, BSCALE, BITS, true>(a, s);
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (a.Hq / a.Hkv) {
      case 1: return launch_k<1, PAGED, BSCALE, BITS, false>(a, s);
      case 2: return launch_k<2, PAGED, BSCALE, BITS, false>(a, s);
      case 4: return launch_k<4, PAGED, BSCALE, BITS, false>(a, s);
      case 8: return launch_k<8, PAGED, BSCALE, BITS, false>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
}

template <int BITS>
cudaError_t launch_b(const DecodeArgs& a, cudaStream_t s) {
  if (a.flags & OSCAR_NORM_ALL_HEADS)
    return a.block_table ? launch_p<true, true, BITS>(a, s) : launch_p<false, true, BITS>(a, s);
  return a.block_table ? launch_p<true, false, BITS>(a, s) : launch_p<false, false, BITS>(a, s);
}

#ifndef OSCAR_DECODE_PAD_TU
template <int GQ>
int occupancy_g() {
  if (allow_smem<GQ, false, false, 2, false>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_int2_kernel<GQ, false, false, 2, false>,
                                                    NW * 32, smem_bytes<GQ, 2>()) != cudaSuccess)
    return 0;
  return n;
}

#endif

}  // namespace

#ifdef OSCAR_DECODE_PAD_TU
cudaError_t launch_decode_int2_padded(const DecodeArgs& a, cudaStream_t s) {
  switch (a.bits) {
    case 2: return launch_b<2>(a, s);
    case 4: return launch_b<4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}
#else
cudaError_t launch_decode_int2(const DecodeArgs& a, cudaStream_t s) {
  if (a.Hkv <= 0 || a.Hq % a.Hkv != 0) return cudaErrorInvalidValue;
  const int g = a.Hq / a.Hkv;
  if (g != decode_group_width(g)) return launch_decode_int2_padded(a, s);
  switch (a.bits) {
    case 2: return launch_b<2>(a, s);
    case 4: return launch_b<4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_int2_ctas_per_sm(int g) {
  switch (decode_group_width(g)) {
    case 1: return occupancy_g<1>();
    case 2: return occupancy_g<2>();
    case 4: return occupancy_g<4>();
    case 8: return occupancy_g<8>();
    default: return 0;
  }
}
#endif

}  // namespace oscar
