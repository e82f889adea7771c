// Fused INT2 dequantisation + inverse token scaling + split-K decode attention
// over the packed cache and the bf16 residual window (kernel (3) of the news
// article on arXiv 2605.19660, 三; "OScaR: The Occam's Razor for Extreme KV
// Cache Quantization in LLMs and Beyond", II. End-to-End Flow and III.
// Efficiency: "Q.K^T and dequantization fused into a single kernel").
//
// Grid (num_splits + 1, Hkv, B): CTA (s, h, b) with s < num_splits streams an
// equal share of the 32-token blocks of row (b, h); CTA num_splits handles the
// residual window.  Each CTA writes one log-sum-exp partial per query head;
// combine_kernel folds them.
//
// Packed path, per 32-token block and warp (all on mma.sync m16n8k16 f16):
//  * no per-element dequantisation: the key step s_c of the block is folded
//    into the query (q~_c = q'_c s_c, split into fp16 hi + lo parts so the
//    product keeps ~22 bits), the key zero z_c becomes one dot product
//    Z = q'.z per block (itself an MMA), and the norm multiplies the score:
//      score_t = tau * n_t * (sum_c q~_c code_tc + Z);
//    Q.K^T runs with the query group as the M rows (hi parts in rows 0-7,
//    lo parts in rows 8-15) and 8 tokens as the N columns;
//  * values: p~_t = p_t s_t (hi + lo fp16) multiplies the centred codes
//    code - 1.5 on the tensor cores; the per-token constant z_t + 1.5 s_t is
//    accumulated as sum_t p_t (z_t + 1.5 s_t) and added per channel at the end;
//  * 2-bit codes become fp16 operands in registers: a masked OR with the fp16
//    bit pattern of 1024 places a code in the mantissa, one fp16 FMA removes
//    the bias (exact), so the codes never travel through shared memory twice;
//  * for groups of 4 or fewer query heads the MMA rows repeat; the two lane
//    halves that hold the same rows split the softmax work by token and swap
//    one fp16 limb of p~ with a shuffle.
// Each warp streams its own contiguous range of blocks through its own
// NSTAGE-deep shared-memory ring: one 1-D bulk copy (TMA, cp.async.bulk) of
// the block's 2752-byte record per block, completing on the warp's mbarrier.  Waits are
// bounded and record kDevErrWaitTimeout instead of hanging; no CTA-wide
// barrier runs inside the main loop.
#include "common.cuh"
#include "cta_merge.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int NW = 4;       // warps per CTA
constexpr int NSTAGE = 4;   // ring depth per warp (blocks in flight)
// one 32-token block record: key codes, value codes, key step, key zero,
// norms, value step, value zero
constexpr int KC_OFF = kRecKC, VC_OFF = kRecVC, KS_OFF = kRecKS, KZ_OFF = kRecKZ,
              KN_OFF = kRecKN, VS_OFF = kRecVS, VZ_OFF = kRecVZ;
constexpr int kSmemBytes = NW * NSTAGE * kBlkBytes + NW * NSTAGE * 8;

constexpr uint32_t kMagic = 0x64006400u;  // fp16x2 {1024, 1024}
constexpr float kLazyLog2 = 8.0f;         // lazy softmax rescale threshold (log2 units)

__device__ __forceinline__ uint32_t hfma2_u(uint32_t x, uint32_t s, uint32_t b) {
  return half2_as_u32(__hfma2(u32_as_half2(x), u32_as_half2(s), u32_as_half2(b)));
}
// (a & MASK) | c in one LOP3 (truth table 0xEA), MASK an immediate.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
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

// Value code pair at slot k as fp16x2 centred values code - 1.5.
// w2 = w << 2 carries slot 0 to position 1, w8 = w >> 8 slots 5..7 to 1..3.
template <int K>
__device__ __forceinline__ uint32_t value_pair(uint32_t w, uint32_t w2, uint32_t w8,
                                                  uint32_t magic) {
  // position p = 1..4: scale 4^-p, bias -(1024 * 4^-p + 1.5)
  constexpr uint32_t S[4] = {0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};
  constexpr uint32_t B[4] = {0xDC06DC06u, 0xD418D418u, 0xCC60CC60u, 0xC580C580u};
  if constexpr (K == 0) {
    return hfma2_u(and_or<0x000C000Cu>(w2, magic), S[0], B[0]);
  } else if constexpr (K < 5) {
    return hfma2_u(and_or<(0x00030003u << (2 * K))>(w, magic), S[K - 1], B[K - 1]);
  } else {
    return hfma2_u(and_or<(0x00030003u << (2 * (K - 4)))>(w8, magic), S[K - 5], B[K - 5]);
  }
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

template <int GQ>
__global__ void __launch_bounds__(NW * 32, 3) decode_int2_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + NW * NSTAGE * kBlkBytes);
  auto& E = *reinterpret_cast<MergeSmem<GQ, NW>*>(smem);
  static_assert(sizeof(MergeSmem<GQ, NW>) <= NW * NSTAGE * kBlkBytes, "merge area");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long long row = (long long)b * a.Hkv + h;
  const long long qrow0 = (long long)b * a.Hq + (long long)h * GQ;  // first query head

  if (split < a.num_splits) {
    // ------------------------------------------------------------ packed
    constexpr bool kSplitHalves = GQ <= 4;         // rows repeat: halves share the softmax
    constexpr int NT = kSplitHalves ? 1 : 2;       // P.V n-tiles (GQ = 8: hi, lo limbs)
    constexpr int NTOK = kSplitHalves ? 4 : 8;     // softmax tokens per thread per block
    const int head = kSplitHalves ? (gid % GQ) : gid;
    const int hf = kSplitHalves ? (gid >> 2) : 0;  // which n-tile pair this lane scores
    const int nblk = a.n_packed / kG;
    const int b0 = (int)((long long)nblk * split / a.num_splits);
    const int b1 = (int)((long long)nblk * (split + 1) / a.num_splits);
    const int wb0 = b0 + (int)((long long)(b1 - b0) * warp / NW);
    const int wb1 = b0 + (int)((long long)(b1 - b0) * (warp + 1) / NW);
    const int n = wb1 - wb0;
    uint8_t* ring = smem + warp * NSTAGE * kBlkBytes;
    uint64_t* bars = bars_all + warp * NSTAGE;

    // Query fragments of this thread's head, channels c0 = 32*tig + 4*k8 ..+3,
    // as {hi(c0,c0+1), lo(c0,c0+1), hi(c0+2,c0+3), lo(c0+2,c0+3)} (the MMA A
    // layout of rows g and g+8).  The query carries softmax_scale * log2(e)
    // and a power of two sigma that keeps the fp16 parts in range.
    uint32_t aq[8][4];
    float inv_sigma;
    {
      const float4* qp = reinterpret_cast<const float4*>(a.q_rot + (qrow0 + head) * kD + 32 * tig);
      float qf[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = qp[i];
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
      int sh = (amax > 0.0f) ? (((a.flags & OSCAR_NO_SCALE) ? 1 : 14) - e) : 0;
      sh = max(-100, min(100, sh));
      const float sigma = ldexpf(1.0f, sh);
      inv_sigma = ldexpf(1.0f, -sh);
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float x0 = qf[4 * k8 + 2 * j] * sigma, x1 = qf[4 * k8 + 2 * j + 1] * sigma;
          const __half2 hh = __floats2half2_rn(x0, x1);
          const float2 hv = __half22float2(hh);
          aq[k8][2 * j] = half2_as_u32(hh);
          aq[k8][2 * j + 1] = half2_as_u32(__floats2half2_rn(x0 - hv.x, x1 - hv.y));
        }
      }
    }

    float O[NT][8][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[t][mt][e] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f, z_run = 0.0f;
    // The fp16x2 bit pattern of {1024, 1024}, kept in a register so that each
    // code extraction is one LOP3 (mask immediate, this register).
    uint32_t magic = kMagic;
    asm volatile("" : "+r"(magic));

    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
      mbar_fence_init();
    }
    __syncwarp();

    // Block i of this warp into ring slot `slot`: lane 0 copies its record
    // (one 1-D bulk copy; the shared-memory slot has the record's layout).
    const uint8_t* rows_rec = a.packed + row * (long long)(a.T_cap / kG) * kBlkBytes;
    auto issue = [&](int i, int slot) {
      if (lane == 0) {
        uint64_t* bar = &bars[slot];
        mbar_arrive_expect_tx(bar, kBlkBytes);
        bulk_g2s(ring + slot * kBlkBytes, rows_rec + (long long)(wb0 + i) * kBlkBytes, kBlkBytes,
                 bar);
      }
    };

    int issued = min(NSTAGE, n);
    for (int s = 0; s < issued; ++s) issue(s, s);

    bool ok = true;
    int it = 0;
    for (; it < n; ++it) {
      const int slot = it % NSTAGE;
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(&bars[slot], (unsigned)((it / NSTAGE) & 1), kWaitLimit));
      if (!ok) break;
      const uint8_t* st = ring + slot * kBlkBytes;
      const uint32_t* kc = reinterpret_cast<const uint32_t*>(st + KC_OFF);
      const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + VC_OFF);
      const uint4* ks4 = reinterpret_cast<const uint4*>(st + KS_OFF) + tig * 4;
      const uint4* kz4 = reinterpret_cast<const uint4*>(st + KZ_OFF) + tig * 4;
      const uint32_t* kn2 = reinterpret_cast<const uint32_t*>(st + KN_OFF);
      const uint32_t* vs2 = reinterpret_cast<const uint32_t*>(st + VS_OFF);
      const uint32_t* vz2 = reinterpret_cast<const uint32_t*>(st + VZ_OFF);

      // Z = q'.z of the block: rows g (hi) and g+8 (lo), every column alike.
      float dz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 zv = kz4[i];
        mma_16816_acc(dz, aq[2 * i], zv.x, zv.y);
        mma_16816_acc(dz, aq[2 * i + 1], zv.z, zv.w);
      }

      // Q.K^T, k-step outer: q~ fragment for k-step k8, then the 4 n-tiles.
      uint32_t kw[4][2], kw10[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint2 v = *reinterpret_cast<const uint2*>(kc + (8 * nt + gid) * 8 + 2 * tig);
        kw[nt][0] = v.x; kw[nt][1] = v.y;
        kw10[nt][0] = v.x >> 10; kw10[nt][1] = v.y >> 10;
      }
      // The Q.K accumulators start from zero (not from Z) so their MMA chains
      // do not wait for the Z chain; Z joins each score below.
      const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 sv = ks4[i];
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          const int k8 = 2 * i + hk;
          // key step of the pair's channels times 4^-p of the pair's code
          // position (exact: a power of two)
          constexpr int P01[4] = {key_pos(0), key_pos(2), key_pos(4), key_pos(6)};
          constexpr int P23[4] = {key_pos(1), key_pos(3), key_pos(5), key_pos(7)};
          uint32_t s01 = hk ? sv.z : sv.x, s23 = hk ? sv.w : sv.y;
          if (P01[k8 & 3] != 0) s01 = hmul2_u(s01, pow4_inv_h2(P01[k8 & 3]));
          if (P23[k8 & 3] != 0) s23 = hmul2_u(s23, pow4_inv_h2(P23[k8 & 3]));
          uint32_t at[4];
          at[0] = hmul2_u(aq[k8][0], s01);
          at[1] = hfma2_u(aq[k8][1], s01, hfma2_u(aq[k8][0], s01, neg2_u(at[0])));
          at[2] = hmul2_u(aq[k8][2], s23);
          at[3] = hfma2_u(aq[k8][3], s23, hfma2_u(aq[k8][2], s23, neg2_u(at[2])));
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const uint32_t w = kw[nt][k8 >> 2], w10 = kw10[nt][k8 >> 2];
            uint32_t b0v, b1v;
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
      const float zsum = dz[0] + dz[2];
      float sc[NTOK];
#pragma unroll
      for (int j = 0; j < NTOK / 2; ++j) {
        const int nt = kSplitHalves ? (2 * hf + j) : j;
        float c0, c1, c2, c3;
        if (kSplitHalves) {
          c0 = hf ? acc[2 + j][0] : acc[j][0]; c1 = hf ? acc[2 + j][1] : acc[j][1];
          c2 = hf ? acc[2 + j][2] : acc[j][2]; c3 = hf ? acc[2 + j][3] : acc[j][3];
        } else {
          c0 = acc[j][0]; c1 = acc[j][1]; c2 = acc[j][2]; c3 = acc[j][3];
        }
        const float2 nf = __half22float2(u32_as_half2(kn2[4 * nt + tig]));
        sc[2 * j] = fmaf(c0 + c2, 16777216.0f, zsum) * (nf.x * inv_sigma);
        sc[2 * j + 1] = fmaf(c1 + c3, 16777216.0f, zsum) * (nf.y * inv_sigma);
      }

      // Online softmax for this thread's head.
      float mb = sc[0];
#pragma unroll
      for (int i = 1; i < NTOK; ++i) mb = fmaxf(mb, sc[i]);
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      if (kSplitHalves) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
      // Lazy rescaling: the running max moves only when a score exceeds it by
      // more than 2^kLazyLog2, so p = 2^(score - m_run) stays below 2^kLazyLog2
      // (well inside fp16 and fp32) and the accumulators are rescaled rarely.
      const float m_new = fmaxf(m_run, mb);
      if (__any_sync(0xffffffffu, m_new > m_run + kLazyLog2)) {
        const float alpha = fast_exp2(m_run - m_new);
        l_run *= alpha;
        z_run *= alpha;
        const int ha = kSplitHalves ? (2 * tig) % GQ : 2 * tig;
        const int hb = kSplitHalves ? (2 * tig + 1) % GQ : 2 * tig + 1;
        const float al_a = __shfl_sync(0xffffffffu, alpha, 4 * ha);
        const float al_b = __shfl_sync(0xffffffffu, alpha, 4 * hb);
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            O[t][mt][0] *= al_a; O[t][mt][1] *= al_b;
            O[t][mt][2] *= al_a; O[t][mt][3] *= al_b;
          }
        m_run = m_new;
      }

      float pt[NTOK];
#pragma unroll
      for (int j = 0; j < NTOK / 2; ++j) {
        const int nt = kSplitHalves ? (2 * hf + j) : j;
        const float2 sv = __half22float2(u32_as_half2(vs2[4 * nt + tig]));
        const float2 zv = __half22float2(u32_as_half2(vz2[4 * nt + tig]));
        const float p0 = fast_exp2(sc[2 * j] - m_run);
        const float p1 = fast_exp2(sc[2 * j + 1] - m_run);
        l_run += p0 + p1;
        z_run = fmaf(p0, fmaf(1.5f, sv.x, zv.x), z_run);
        z_run = fmaf(p1, fmaf(1.5f, sv.y, zv.y), z_run);
        pt[2 * j] = p0 * sv.x;
        pt[2 * j + 1] = p1 * sv.y;
      }

      // P~ as the B operand of P.V: k-half kh uses n-tiles 2kh (tokens 2tig,
      // 2tig+1) and 2kh+1 (2tig+8, 2tig+9); column gid is limb gid/4 (GQ <= 4).
      uint32_t bp[2][2], bq[2][2];  // bp: limb for n-tile 0 of P.V; bq: lo limb (GQ = 8)
      if (kSplitHalves) {
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const __half2 hv = __floats2half2_rn(pt[2 * r], pt[2 * r + 1]);
          const float2 hf2 = __half22float2(hv);
          hi[r] = half2_as_u32(hv);
          lo[r] = half2_as_u32(__floats2half2_rn(pt[2 * r] - hf2.x, pt[2 * r + 1] - hf2.y));
        }
        // own limb for k-half hf; the partner lane (other half) needs my other limb
        const uint32_t mine0 = hf ? lo[0] : hi[0], mine1 = hf ? lo[1] : hi[1];
        const uint32_t give0 = hf ? hi[0] : lo[0], give1 = hf ? hi[1] : lo[1];
        const uint32_t got0 = __shfl_xor_sync(0xffffffffu, give0, 16);
        const uint32_t got1 = __shfl_xor_sync(0xffffffffu, give1, 16);
        bp[0][0] = hf ? got0 : mine0; bp[0][1] = hf ? got1 : mine1;
        bp[1][0] = hf ? mine0 : got0; bp[1][1] = hf ? mine1 : got1;
      } else {
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
      }

#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        const uint4 vw = *reinterpret_cast<const uint4*>(vc + kh * 128 + lane * 4);
        const uint32_t wv[4] = {vw.x, vw.y, vw.z, vw.w};  // (p,hh) = (0,0) (0,1) (1,0) (1,1)
        uint32_t w2[4], w8[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) { w2[q] = wv[q] << 2; w8[q] = wv[q] >> 8; }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int hh = mt >> 2;
          const int p0 = hh, p1 = 2 + hh;  // words of tokens (2tig,2tig+1) and (2tig+8,2tig+9)
          uint32_t av[4];
          switch (mt & 3) {
            case 0:
              av[0] = value_pair<0>(wv[p0], w2[p0], w8[p0], magic); av[1] = value_pair<1>(wv[p0], w2[p0], w8[p0], magic);
              av[2] = value_pair<0>(wv[p1], w2[p1], w8[p1], magic); av[3] = value_pair<1>(wv[p1], w2[p1], w8[p1], magic);
              break;
            case 1:
              av[0] = value_pair<2>(wv[p0], w2[p0], w8[p0], magic); av[1] = value_pair<3>(wv[p0], w2[p0], w8[p0], magic);
              av[2] = value_pair<2>(wv[p1], w2[p1], w8[p1], magic); av[3] = value_pair<3>(wv[p1], w2[p1], w8[p1], magic);
              break;
            case 2:
              av[0] = value_pair<4>(wv[p0], w2[p0], w8[p0], magic); av[1] = value_pair<5>(wv[p0], w2[p0], w8[p0], magic);
              av[2] = value_pair<4>(wv[p1], w2[p1], w8[p1], magic); av[3] = value_pair<5>(wv[p1], w2[p1], w8[p1], magic);
              break;
            default:
              av[0] = value_pair<6>(wv[p0], w2[p0], w8[p0], magic); av[1] = value_pair<7>(wv[p0], w2[p0], w8[p0], magic);
              av[2] = value_pair<6>(wv[p1], w2[p1], w8[p1], magic); av[3] = value_pair<7>(wv[p1], w2[p1], w8[p1], magic);
              break;
          }
          mma_16816_acc(O[0][mt], av, bp[kh][0], bp[kh][1]);
          if (!kSplitHalves) mma_16816_acc(O[NT - 1][mt], av, bq[kh][0], bq[kh][1]);
        }
      }
      __syncwarp();
      if (it + NSTAGE < n) issue(it + NSTAGE, slot);
    }
    if (!ok) {
      if (lane == 0) {
        record_error(a.status, kDevErrWaitTimeout);
        for (int s = it; s < issued && s < n; ++s)
          if (!mbar_wait_bounded(&bars[s % NSTAGE], (unsigned)((s / NSTAGE) & 1), kDrainLimit))
            record_error(a.status, kDevErrDrainTimeout);
      }
      m_run = -INFINITY;   // this warp's result is void; the status word says so
    }

    // Warp results: sums over the lanes of a head, limbs folded.
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    z_run += __shfl_xor_sync(0xffffffffu, z_run, 1);
    z_run += __shfl_xor_sync(0xffffffffu, z_run, 2);
    if (kSplitHalves) {
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
      z_run += __shfl_xor_sync(0xffffffffu, z_run, 16);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[0][mt][e] += __shfl_xor_sync(0xffffffffu, O[0][mt][e], 2);
    } else {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[0][mt][e] += O[NT - 1][mt][e];
    }
    __syncthreads();   // every warp is done with its ring: reuse it for the merge
    if (tig == 0 && gid < GQ) {
      E.m[warp][gid] = m_run;
      E.l[warp][gid] = l_run;
      E.z[warp][gid] = z_run;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int nc = 2 * tig + e;
      if (nc < GQ) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          E.o[warp][nc][16 * mt + gid] = O[0][mt][e];
          E.o[warp][nc][16 * mt + gid + 8] = O[0][mt][2 + e];
        }
      }
    }
  } else {
    // ------------------------------------------------------------ residual
    // Unit-norm bf16 keys times their fp16 norms, bf16 values; CUDA cores.
    float qv[GQ][4], mr[GQ], lr[GQ], orr[GQ][4];
#pragma unroll
    for (int j = 0; j < GQ; ++j) {
      const float4 v = reinterpret_cast<const float4*>(a.q_rot + (qrow0 + j) * kD)[lane];
      qv[j][0] = v.x; qv[j][1] = v.y; qv[j][2] = v.z; qv[j][3] = v.w;
      mr[j] = -INFINITY; lr[j] = 0.0f;
      orr[j][0] = orr[j][1] = orr[j][2] = orr[j][3] = 0.0f;
    }
    for (int t = warp; t < a.n_res; t += NW) {
      const long long tok = row * kR + t;
      const uint2 kr = reinterpret_cast<const uint2*>(a.k_res + tok * kD)[lane];
      const uint2 vr = reinterpret_cast<const uint2*>(a.v_res + tok * kD)[lane];
      const float k4[4] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y)};
      const float v4[4] = {bf16_lo(vr.x), bf16_hi(vr.x), bf16_lo(vr.y), bf16_hi(vr.y)};
      const float nrm = __half2float(a.k_res_norm[tok]);
#pragma unroll
      for (int j = 0; j < GQ; ++j) {
        float d = qv[j][0] * k4[0] + qv[j][1] * k4[1] + qv[j][2] * k4[2] + qv[j][3] * k4[3];
        d = warp_allsum(d);
        const float s = d * nrm * a.scale_log2;
        const float m_new = fmaxf(mr[j], s);
        const float al = fast_exp2(mr[j] - m_new);
        const float p = fast_exp2(s - m_new);
        lr[j] = lr[j] * al + p;
#pragma unroll
        for (int i = 0; i < 4; ++i) orr[j][i] = orr[j][i] * al + p * v4[i];
        mr[j] = m_new;
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
  __syncthreads();
  cta_merge_write<GQ, NW>(E, a.ws + (qrow0 * (a.num_splits + 1) + split) * kRecFloats,
                          (long long)(a.num_splits + 1) * kRecFloats);
}

template <int GQ>
cudaError_t launch_g(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.num_splits + 1, a.Hkv, a.B);
  decode_int2_kernel<GQ><<<grid, NW * 32, kSmemBytes, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(a.ws, a.out, a.B * a.Hq, a.num_splits + 1, s);
}

template <int GQ>
int occupancy_g() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_int2_kernel<GQ>, NW * 32,
                                                    kSmemBytes) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace

cudaError_t launch_decode_int2(const DecodeArgs& a, cudaStream_t s) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_g<1>(a, s);
    case 2: return launch_g<2>(a, s);
    case 4: return launch_g<4>(a, s);
    case 8: return launch_g<8>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_int2_ctas_per_sm(int g) {
  switch (g) {
    case 1: return occupancy_g<1>();
    case 2: return occupancy_g<2>();
    case 4: return occupancy_g<4>();
    case 8: return occupancy_g<8>();
    default: return 0;
  }
}

}  // namespace oscar
