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
//  * values: p~_t = p_t s_t (hi + lo fp16) multiplies the centred codes
//    code - 1.5 on the tensor cores; the per-token constant z_t + 1.5 s_t is
//    accumulated as sum_t p_t (z_t + 1.5 s_t) and added per channel at the end;
//  * 2-bit codes become fp16 operands in registers: a masked OR with the fp16
//    bit pattern of 1024 places a code in the mantissa, one fp16 FMA removes
//    the bias (exact), so the codes never travel through shared memory twice.
// Stage ring: thread 0 issues seven 1-D bulk copies (TMA, cp.async.bulk) per
// stage of NW blocks into a NSTAGE-deep shared-memory ring; mbarrier waits are
// bounded and record kDevErrWaitTimeout instead of hanging.
#include "common.cuh"
#include "cta_merge.cuh"
#include "launch.h"

namespace oscar {
namespace {

constexpr int NW = 4;       // warps per CTA = blocks per stage
constexpr int NSTAGE = 4;   // ring depth
constexpr int kBlkBytes = 1024 + 1024 + 256 + 256 + 64 + 64 + 64;
constexpr int kStageBytes = NW * kBlkBytes;
constexpr int KC_OFF = 0;
constexpr int VC_OFF = NW * 1024;
constexpr int KS_OFF = NW * 2048;
constexpr int KZ_OFF = NW * 2304;
constexpr int KN_OFF = NW * 2560;
constexpr int VS_OFF = NW * 2624;
constexpr int VZ_OFF = NW * 2688;
constexpr int kSmemBytes = NSTAGE * kStageBytes + NSTAGE * 8;
static_assert(VZ_OFF + NW * 64 == kStageBytes, "stage layout");

constexpr uint32_t kMagic = 0x64006400u;  // fp16x2 {1024, 1024}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t x, uint32_t s, uint32_t b) {
  return half2_as_u32(__hfma2(u32_as_half2(x), u32_as_half2(s), u32_as_half2(b)));
}

// Key word -> 8 fp16x2 code pairs (slot k: low/high half-word codes), values 0..3.
__device__ __forceinline__ void unpack_k8(uint32_t w, uint32_t (&o)[8]) {
  const uint32_t S[5] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};
  const uint32_t B[5] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u, 0xC400C400u};
#pragma unroll
  for (int k = 0; k < 5; ++k) o[k] = hfma2_u((w & (0x00030003u << (2 * k))) | kMagic, S[k], B[k]);
  const uint32_t w2 = w >> 10;
#pragma unroll
  for (int k = 5; k < 8; ++k)
    o[k] = hfma2_u((w2 & (0x00030003u << (2 * (k - 5)))) | kMagic, S[k - 5], B[k - 5]);
}

// Value word -> 8 fp16x2 centred code pairs (code - 1.5).
__device__ __forceinline__ void unpack_v8(uint32_t w, uint32_t (&o)[8]) {
  // index k-1 for k = 1..4: scale 4^-k, bias -(1024*4^-k + 1.5)
  const uint32_t S[4] = {0x34003400u, 0x2C002C00u, 0x24002400u, 0x1C001C00u};
  const uint32_t B[4] = {0xDC06DC06u, 0xD418D418u, 0xCC60CC60u, 0xC580C580u};
  o[0] = hfma2_u(((w << 2) & 0x000C000Cu) | kMagic, S[0], B[0]);
#pragma unroll
  for (int k = 1; k < 5; ++k)
    o[k] = hfma2_u((w & (0x00030003u << (2 * k))) | kMagic, S[k - 1], B[k - 1]);
  const uint32_t w8 = w >> 8;
#pragma unroll
  for (int k = 5; k < 8; ++k)
    o[k] = hfma2_u((w8 & (0x00030003u << (2 * (k - 4)))) | kMagic, S[k - 5], B[k - 5]);
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

template <int GQ>
__global__ void __launch_bounds__(NW * 32) decode_int2_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NSTAGE * kStageBytes);
  auto& E = *reinterpret_cast<MergeSmem<GQ, NW>*>(smem);
  static_assert(sizeof(MergeSmem<GQ, NW>) <= NSTAGE * kStageBytes, "merge area");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long long row = (long long)b * a.Hkv + h;
  const long long qrow0 = (long long)b * a.Hq + (long long)h * GQ;  // first query head

  if (split < a.num_splits) {
    // ------------------------------------------------------------ packed
    constexpr int NT = (GQ == 8) ? 2 : 1;        // PV n-tiles (hi / lo limbs for GQ = 8)
    const int head = (GQ == 8) ? gid : (gid % GQ);
    const int nblk = a.n_packed / kG;
    const int b0 = (int)((long long)nblk * split / a.num_splits);
    const int b1 = (int)((long long)nblk * (split + 1) / a.num_splits);
    const int n_iter = (b1 - b0 + NW - 1) / NW;

    // Query fragments: this thread's head, channels 32*tig .. 32*tig+31,
    // scaled by a power of two sigma so that fp16 hi/lo parts keep range.
    uint32_t qh[8][2], ql[8][2];
    float cst;
    {
      const float4* qp = reinterpret_cast<const float4*>(a.q_rot + (qrow0 + head) * kD + 32 * tig);
      float qf[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = qp[i];
        qf[4 * i] = v.x; qf[4 * i + 1] = v.y; qf[4 * i + 2] = v.z; qf[4 * i + 3] = v.w;
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
      cst = ldexpf(a.scale_log2, -sh);
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float x0 = qf[4 * k8 + 2 * j] * sigma, x1 = qf[4 * k8 + 2 * j + 1] * sigma;
          const __half2 hh = __floats2half2_rn(x0, x1);
          const float2 hf = __half22float2(hh);
          qh[k8][j] = half2_as_u32(hh);
          ql[k8][j] = half2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
        }
      }
    }

    float O[NT][8][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[n][mt][e] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f, z_run = 0.0f;

    if (tid == 0) {
#pragma unroll
      for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
      mbar_fence_init();
    }
    __syncthreads();

    auto issue = [&](int it, int slot) {
      const int blk = b0 + it * NW;
      const int nb = min(NW, b1 - blk);
      uint8_t* st = smem + slot * kStageBytes;
      uint64_t* bar = &bars[slot];
      mbar_arrive_expect_tx(bar, nb * kBlkBytes);
      const long long kb = row * (a.T_cap / kG) + blk;
      const long long kt = row * (long long)a.T_cap + (long long)blk * kG;
      bulk_g2s(st + KC_OFF, a.k_codes + kt * 8, nb * 1024, bar);
      bulk_g2s(st + VC_OFF, a.v_codes + kb * 256, nb * 1024, bar);
      bulk_g2s(st + KS_OFF, a.k_scale + kb * kD, nb * 256, bar);
      bulk_g2s(st + KZ_OFF, a.k_zero + kb * kD, nb * 256, bar);
      bulk_g2s(st + KN_OFF, a.k_norm + kt, nb * 64, bar);
      bulk_g2s(st + VS_OFF, a.v_scale + kt, nb * 64, bar);
      bulk_g2s(st + VZ_OFF, a.v_zero + kt, nb * 64, bar);
    };

    int issued = 0;
    if (tid == 0) {
      issued = min(NSTAGE, n_iter);
      for (int s = 0; s < issued; ++s) issue(s, s);
    }

    bool bad = false;
    int it = 0;
    for (; it < n_iter; ++it) {
      const int slot = it % NSTAGE;
      bool ok = mbar_wait_bounded(&bars[slot], (unsigned)((it / NSTAGE) & 1), kWaitLimit);
      ok = __all_sync(0xffffffffu, ok);
      const int blk = b0 + it * NW + warp;
      if (ok && blk < b1) {
        const uint8_t* st = smem + slot * kStageBytes;
        const uint32_t* kc = reinterpret_cast<const uint32_t*>(st + KC_OFF) + warp * 256;
        const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + VC_OFF) + warp * 256;
        const uint4* ks4 = reinterpret_cast<const uint4*>(st + KS_OFF + warp * 256) + tig * 4;
        const uint4* kz4 = reinterpret_cast<const uint4*>(st + KZ_OFF + warp * 256) + tig * 4;
        const uint32_t* kn2 = reinterpret_cast<const uint32_t*>(st + KN_OFF + warp * 64);
        const uint32_t* vs2 = reinterpret_cast<const uint32_t*>(st + VS_OFF + warp * 64);
        const uint32_t* vz2 = reinterpret_cast<const uint32_t*>(st + VZ_OFF + warp * 64);

        // Z = q'.z_block (hi row g, lo row g+8), broadcast to all 8 columns.
        float dz[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t at[8][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 sv = ks4[i];
          const uint4 zv = kz4[i];
          const uint32_t sr[4] = {sv.x, sv.y, sv.z, sv.w};
          const uint32_t zr[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
          for (int hk = 0; hk < 2; ++hk) {
            const int k8 = 2 * i + hk;
            const uint32_t aq[4] = {qh[k8][0], ql[k8][0], qh[k8][1], ql[k8][1]};
            mma_16816(dz, aq, zr[2 * hk], zr[2 * hk + 1], dz);
            // q~ = q' * s as fp16 hi + lo (exact product error via FMA).
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const __half2 s = u32_as_half2(sr[2 * hk + j]);
              const __half2 q1 = u32_as_half2(qh[k8][j]);
              const __half2 hi = __hmul2(q1, s);
              const __half2 lo =
                  __hadd2(__hfma2(q1, s, __hneg2(hi)), __hmul2(u32_as_half2(ql[k8][j]), s));
              at[k8][2 * j] = half2_as_u32(hi);
              at[k8][2 * j + 1] = half2_as_u32(lo);
            }
          }
        }

        // Scores for 4 n-tiles of 8 tokens: thread holds tokens 8nt+2tig, +1.
        float sc[8];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const uint2 kw = *reinterpret_cast<const uint2*>(kc + (8 * nt + gid) * 8 + 2 * tig);
          uint32_t bk0[8], bk1[8];
          unpack_k8(kw.x, bk0);
          unpack_k8(kw.y, bk1);
          float acc[4] = {dz[0], dz[1], dz[2], dz[3]};
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8) mma_16816(acc, at[k8], bk0[2 * k8], bk0[2 * k8 + 1], acc);
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8)
            mma_16816(acc, at[4 + k8], bk1[2 * k8], bk1[2 * k8 + 1], acc);
          const float2 nf = __half22float2(u32_as_half2(kn2[4 * nt + tig]));
          sc[2 * nt] = (acc[0] + acc[2]) * (nf.x * cst);
          sc[2 * nt + 1] = (acc[1] + acc[3]) * (nf.y * cst);
        }

        // Online softmax (log2 domain) for this thread's head.
        float mb = sc[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) mb = fmaxf(mb, sc[i]);
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        const float m_new = fmaxf(m_run, mb);
        if (__any_sync(0xffffffffu, m_new > m_run)) {
          const float alpha = fast_exp2(m_run - m_new);
          l_run *= alpha;
          z_run *= alpha;
          const int ha = (GQ == 8) ? 2 * tig : (2 * tig) % GQ;
          const int hb = (GQ == 8) ? 2 * tig + 1 : (2 * tig + 1) % GQ;
          const float al_a = __shfl_sync(0xffffffffu, alpha, 4 * ha);
          const float al_b = __shfl_sync(0xffffffffu, alpha, 4 * hb);
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              O[n][mt][0] *= al_a; O[n][mt][1] *= al_b;
              O[n][mt][2] *= al_a; O[n][mt][3] *= al_b;
            }
          m_run = m_new;
        }

        float pt[8];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const float2 sv = __half22float2(u32_as_half2(vs2[4 * nt + tig]));
          const float2 zv = __half22float2(u32_as_half2(vz2[4 * nt + tig]));
          const float p0 = fast_exp2(sc[2 * nt] - m_run);
          const float p1 = fast_exp2(sc[2 * nt + 1] - m_run);
          l_run += p0 + p1;
          z_run = fmaf(p0, fmaf(1.5f, sv.x, zv.x), z_run);
          z_run = fmaf(p1, fmaf(1.5f, sv.y, zv.y), z_run);
          pt[2 * nt] = p0 * sv.x;
          pt[2 * nt + 1] = p1 * sv.y;
        }

        // P~ as the B operand of P.V (tokens 2tig,2tig+1 | 2tig+8,2tig+9 per k-half).
        uint32_t bh[2][2], bl[2][2];
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float x0 = pt[4 * kh + 2 * r], x1 = pt[4 * kh + 2 * r + 1];
            const __half2 hi = __floats2half2_rn(x0, x1);
            const float2 hf = __half22float2(hi);
            bh[kh][r] = half2_as_u32(hi);
            bl[kh][r] = half2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
          }

#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
          const uint4 vw = *reinterpret_cast<const uint4*>(vc + kh * 128 + lane * 4);
          uint32_t b0v, b1v;
          if (GQ == 8) {
            b0v = bh[kh][0]; b1v = bh[kh][1];
          } else {
            const bool lo_limb = gid >= 4;
            b0v = lo_limb ? bl[kh][0] : bh[kh][0];
            b1v = lo_limb ? bl[kh][1] : bh[kh][1];
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t va[8], vb[8];
            unpack_v8(hh ? vw.y : vw.x, va);   // p = 0 (tokens 2tig, 2tig+1)
            unpack_v8(hh ? vw.w : vw.z, vb);   // p = 1 (tokens 2tig+8, 2tig+9)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int mt = 4 * hh + q4;
              const uint32_t av[4] = {va[2 * q4], va[2 * q4 + 1], vb[2 * q4], vb[2 * q4 + 1]};
              mma_16816(O[0][mt], av, b0v, b1v, O[0][mt]);
              if (GQ == 8) mma_16816(O[NT - 1][mt], av, bl[kh][0], bl[kh][1], O[NT - 1][mt]);
            }
          }
        }
      }
      bad = __syncthreads_or(!ok);
      if (bad) break;
      if (tid == 0 && it + NSTAGE < n_iter) {
        issue(it + NSTAGE, slot);
        ++issued;
      }
    }
    if (bad) {
      if (tid == 0) {
        record_error(a.status, kDevErrWaitTimeout);
        for (int s = it; s < issued; ++s)
          if (!mbar_wait_bounded(&bars[s % NSTAGE], (unsigned)((s / NSTAGE) & 1), kDrainLimit))
            record_error(a.status, kDevErrDrainTimeout);
      }
      return;
    }

    // Warp results: sums over the four lanes of a head, limbs folded.
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    z_run += __shfl_xor_sync(0xffffffffu, z_run, 1);
    z_run += __shfl_xor_sync(0xffffffffu, z_run, 2);
    if (GQ != 8) {
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
    __syncthreads();   // the stage ring is dead: reuse it for the merge
    if (tig == 0 && gid < GQ) {
      E.m[warp][gid] = m_run;
      E.l[warp][gid] = l_run;
      E.z[warp][gid] = z_run;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 2 * tig + e;
      if (n < GQ) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          E.o[warp][n][16 * mt + gid] = O[0][mt][e];
          E.o[warp][n][16 * mt + gid + 8] = O[0][mt][2 + e];
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
