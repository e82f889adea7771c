// C ABI of liboscar (include/oscar.h): argument validation, split planning,
// state bookkeeping of oscar_cache, and dispatch to the kernels.
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "launch.h"

__device__ unsigned g_oscar_status;  // OR of kDevErr* bits since the last read

namespace {

using namespace oscar;

std::atomic<unsigned long long> g_launches{0};
std::mutex g_mu;
unsigned* g_status_ptr[128] = {};

unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_oscar_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

oscar_status from_cuda(cudaError_t e) { return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA; }

oscar_status check_cache(const oscar_cache* c) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (c->B <= 0 || c->Hkv <= 0 || c->T_cap <= 0 || c->T_cap % kG != 0)
    return OSCAR_ERR_INVALID_ARG;
  const void* ptrs[] = {c->packed, c->k_res, c->v_res, c->k_res_norm};
  for (const void* p : ptrs) {
    if (!p) return OSCAR_ERR_INVALID_ARG;
    if (!al16(p)) return OSCAR_ERR_ALIGNMENT;
  }
  if (c->n_packed < 0 || c->n_packed % kG != 0 || c->n_packed > c->T_cap)
    return OSCAR_ERR_INVALID_ARG;
  if (c->n_res < 0 || c->n_res > kR) return OSCAR_ERR_INVALID_ARG;
  if ((c->flags & ~kAllFlags) || !target_ok(c->norm_target)) return OSCAR_ERR_INVALID_ARG;
  if (!key_group_ok(c->key_group) || c->n_packed % key_group(c->key_group) != 0 ||
      !code_bits_ok(c->bits))
    return OSCAR_ERR_INVALID_ARG;
  return OSCAR_OK;
}

// Split planning.  A launch runs rows * (s + 1) CTAs: s packed splits of
// about nblk / s blocks per row, whose four warps take a quarter each, and
// one short residual split per row, in grid order with a row's CTAs
// adjacent.  The planner models the launch's time for each s and takes the
// cheapest:
//  * One wave (rows * s packed CTAs fit in the resident slots): one packed
//    CTA's time, (kFixedBlocks + blocks per warp) x the time a warp takes
//    per block when n CTAs share its SM, n the most CTAs any SM gets
//    (ceil(rows * (s + 1) / SMs): the residual CTAs sit between the packed
//    ones in grid order, so an SM's share may be all packed).  kBlockUs holds
//    those per-block times for n = 1..4: the SM's issue slots are shared, so
//    a warp runs slower as more warps share them, but the SM's throughput
//    still rises up to four CTAs.  If the residual CTAs spill past the wave,
//    kLateUs more.
//  * More waves: the same per-CTA time at four CTAs per SM times the waves
//    W = rows * s / slots, plus kTailShare of a wave for the unfilled part
//    of the last one (CTAs of unequal start times fill it partly).
//  * Plus kCombineUsPerSplit per split for the combine of the row's
//    partials, which runs after the row's last CTA.
// Each warp keeps at least kMinBlocksPerWarp blocks when the packed CTAs
// take more than one wave, and kMinBlocksPerWarpOneWave within one wave.
// Ties keep fewer splits.
//
// The constants are fitted to sweeps of split counts on GB300 (152 SMs,
// four INT2 decode CTAs per SM; L2 flushed for the shapes that fit in it):
// 19 shapes from 1 to 384 rows and 128 to 4096 blocks (batch 1-48, 4K-128K
// tokens, 32/8 and 32/4 heads).  The planned count is within 2.2 % of the
// fastest swept count on every one (0.3 % on average).  The earlier model,
// ceil(CTAs / SMs) x (blocks + 32) at full speed from two CTAs per SM on,
// planned 1 split for batch 48 at 16K-112K tokens, 1.4-1.6 x slower than the
// best count.
//
// On grids of more than two waves, an even count that wins is then compared
// with its odd neighbours, and the cheaper of them is taken if its modelled
// cost is within kEvenSplitPenalty of the winner's: there, on GB300, even
// counts measured 1-3 % slower than their odd neighbours (batch 48 x 128K:
// 12 splits 982 us, 11 and 13 splits 969-972 us; batch 48 x 80K: 8 and 10
// splits 632 and 628 us, 9 splits 618 us), with the residual CTA placed
// anywhere in the row, with a padded grid and without the combine; the
// cause is not known.
constexpr double kBlockUs[5] = {0.0, 0.60, 0.80, 1.20, 1.55};
constexpr double kFixedBlocks = 1.0;
constexpr double kTailShare = 0.4;
constexpr double kLateUs = 1.5;
constexpr double kCombineUsPerSplit = 0.05;
constexpr long long kMinBlocksPerWarp = 16;
constexpr long long kMinBlocksPerWarpOneWave = 2;
constexpr int kWarpsPerCta = 4;
constexpr double kEvenSplitPenalty = 1.02;

int plan_splits_for(long long rows, long long nblk, int ctas_per_sm, int sms, int max_splits) {
  if (nblk <= 0 || rows <= 0 || sms <= 0 || max_splits < 1) return 1;
  const long long cps = ctas_per_sm > 0 ? ctas_per_sm : 1;
  const long long slots = (long long)sms * cps;
  const long long most = std::max<long long>(1, nblk / (kWarpsPerCta * kMinBlocksPerWarp));
  const long long most1 = std::max<long long>(1, nblk / (kWarpsPerCta * kMinBlocksPerWarpOneWave));
  const int hi = (int)std::min<long long>(max_splits, most);
  const int hi1 = (int)std::min<long long>(max_splits, most1);
  auto block_us = [&](long long n) { return kBlockUs[std::min<long long>(std::max<long long>(n, 1), 4)]; };
  auto cost_of = [&](int s) {
    const double per_warp = (double)nblk / s / kWarpsPerCta;
    const double waves = (double)(rows * s) / (double)slots;
    double t;
    if (waves <= 1.0) {
      const long long n = std::min(cps, (rows * (s + 1) + sms - 1) / sms);
      t = (kFixedBlocks + per_warp) * block_us(n);
      if (rows * (s + 1) > slots) t += kLateUs;
    } else {
      const double d = (kFixedBlocks + per_warp) * block_us(cps);
      t = d * (waves + kTailShare * (std::ceil(waves) - waves));
    }
    return t + kCombineUsPerSplit * (s + 1);
  };
  int best = 1;
  double best_cost = cost_of(1);
  for (int s = 2; s <= hi1; ++s) {
    if (s > hi && rows * s > slots) continue;   // short ranges only within one wave
    const double cost = cost_of(s);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  if (best % 2 == 0 && rows * (best + 1) > 2 * slots) {
    int odd = 0;
    double odd_cost = 1e300;
    for (int s : {best - 1, best + 1}) {
      if (s < 1 || s > hi) continue;
      const double c = cost_of(s);
      if (c < odd_cost - 1e-9) {
        odd_cost = c;
        odd = s;
      }
    }
    if (odd > 0 && odd_cost <= best_cost * kEvenSplitPenalty) best = odd;
  }
  return best;
}

int plan_splits(long long rows, long long nblk, int ctas_per_sm, int max_splits) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return plan_splits_for(rows, nblk, ctas_per_sm, sms, max_splits);
}

// Split count of the bf16 comparison kernel (no residual split): waves of
// sms * ctas_per_sm CTAs times the chunks per split, plus 0.25 per split.
int plan_splits_bf16(long long rows, long long nchunk, int ctas_per_sm, int max_splits) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  if (nchunk <= 0 || rows <= 0) return 1;
  const long long slots = (long long)sms * (ctas_per_sm > 0 ? ctas_per_sm : 1);
  int best = 1;
  double best_cost = 1e300;
  const int hi = (int)std::min<long long>(max_splits, nchunk);
  for (int s = 1; s <= hi; ++s) {
    const long long waves = (rows * s + slots - 1) / slots;
    const long long per = (nchunk + s - 1) / s;
    const double cost = (double)waves * (double)per + 0.25 * s;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

size_t ws_bytes_for(int B, int Hq, int parts) {
  return (size_t)B * (size_t)Hq * (size_t)parts * kRecFloats * sizeof(float);
}

oscar_status flush_residual(oscar_cache* c, cudaStream_t s) {
  if (c->n_packed + kR > c->T_cap) return OSCAR_ERR_CAPACITY;
  cudaError_t e = launch_quantize_kv(
      c->k_res, reinterpret_cast<const __half*>(c->k_res_norm), c->v_res, kR, kR, c->B, c->Hkv,
      c->T_cap, c->n_packed, key_group(c->key_group), code_bits(c->bits), c->packed, s);
  g_launches++;
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  c->n_packed += kR;
  c->n_res = 0;
  return OSCAR_OK;
}

}  // namespace

namespace oscar {
// Internal accessors for other translation units of the library.
oscar_status validate_cache(const oscar_cache* c) { return check_cache(c); }

unsigned* device_status_word() { return status_ptr(); }
void count_launches(int n) { g_launches += (unsigned long long)n; }
}  // namespace oscar

extern "C" {

oscar_status oscar_rotate_q(const oscar_bf16* q, float* q_rot, int B, int Hq, unsigned flags,
                            void* stream) {
  if (!q || !q_rot || B <= 0 || Hq <= 0 || (flags & ~kAllFlags)) return OSCAR_ERR_INVALID_ARG;
  if (!al16(q) || !al16(q_rot)) return OSCAR_ERR_ALIGNMENT;
  const long long n = (long long)B * Hq;
  if (n > (1LL << 30)) return OSCAR_ERR_INVALID_ARG;
  cudaError_t e = launch_rotate_q(q, q_rot, (int)n, flags, as_stream(stream));
  g_launches++;
  return from_cuda(e);
}

oscar_status oscar_rotate_scale_k(const oscar_bf16* k, int in_T, oscar_bf16* k_hat,
                                  oscar_f16* norm_out, int out_T, int out_t0, int B, int Hkv,
                                  int n_tok, unsigned flags, float norm_target, void* stream) {
  if (!k || !k_hat || !norm_out || B <= 0 || Hkv <= 0 || n_tok <= 0 || (flags & ~kAllFlags) ||
      !target_ok(norm_target))
    return OSCAR_ERR_INVALID_ARG;
  if (in_T < n_tok || out_t0 < 0 || out_t0 + (long long)n_tok > out_T)
    return OSCAR_ERR_INVALID_ARG;
  if (!al16(k) || !al16(k_hat) || !al16(norm_out)) return OSCAR_ERR_ALIGNMENT;
  const long long rows = (long long)B * Hkv;
  if (rows * n_tok > (1LL << 34)) return OSCAR_ERR_INVALID_ARG;
  cudaError_t e = launch_rotate_scale_k(k, in_T, k_hat, reinterpret_cast<__half*>(norm_out),
                                        out_T, out_t0, (int)rows, Hkv, n_tok, nullptr, nullptr,
                                        key_scale(flags, norm_target), as_stream(stream));
  g_launches++;
  return from_cuda(e);
}

oscar_status oscar_quantize_kv(oscar_cache* c, const oscar_bf16* k_hat, const oscar_f16* k_norm,
                               const oscar_bf16* v, int src_T, int n_tok, void* stream) {
  oscar_status st = check_cache(c);
  if (st != OSCAR_OK) return st;
  if (!k_hat && !k_norm && !v) {
    if (c->n_res != kR) return OSCAR_ERR_INVALID_ARG;
    return flush_residual(c, as_stream(stream));
  }
  if (!k_hat || !k_norm || !v) return OSCAR_ERR_INVALID_ARG;
  if (!al16(k_hat) || !al16(k_norm) || !al16(v)) return OSCAR_ERR_ALIGNMENT;
  const int G = key_group(c->key_group);
  if (n_tok < G || n_tok % G != 0 || src_T < n_tok) return OSCAR_ERR_INVALID_ARG;
  if (c->n_res != 0) return OSCAR_ERR_INVALID_ARG;  // packed tokens must precede residual ones
  if ((long long)c->n_packed + n_tok > c->T_cap) return OSCAR_ERR_CAPACITY;
  cudaError_t e = launch_quantize_kv(
      k_hat, reinterpret_cast<const __half*>(k_norm), v, src_T, n_tok, c->B, c->Hkv, c->T_cap,
      c->n_packed, G, code_bits(c->bits), c->packed, as_stream(stream));
  g_launches++;
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  c->n_packed += n_tok;
  return OSCAR_OK;
}

oscar_status oscar_prefill_kv(oscar_cache* c, const oscar_bf16* k, const oscar_bf16* v, int in_T,
                              int n_tok, void* stream) {
  oscar_status st = check_cache(c);
  if (st != OSCAR_OK) return st;
  if (!k || !v) return OSCAR_ERR_INVALID_ARG;
  if (!al16(k) || !al16(v)) return OSCAR_ERR_ALIGNMENT;
  const int G = key_group(c->key_group);
  if (n_tok < G || n_tok % G != 0 || in_T < n_tok) return OSCAR_ERR_INVALID_ARG;
  if (c->n_res != 0) return OSCAR_ERR_INVALID_ARG;  // packed tokens must precede residual ones
  if ((long long)c->n_packed + n_tok > c->T_cap) return OSCAR_ERR_CAPACITY;
  cudaError_t e = launch_prefill_kv(k, v, in_T, n_tok, c->B, c->Hkv, c->T_cap, c->n_packed, G,
                                    code_bits(c->bits), key_scale(c->flags, c->norm_target),
                                    c->packed,
                                    as_stream(stream));
  g_launches++;
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  c->n_packed += n_tok;
  return OSCAR_OK;
}

oscar_status oscar_append_kv(oscar_cache* c, const oscar_bf16* k_new, const oscar_bf16* v_new,
                             int n_tok, void* stream) {
  oscar_status st = check_cache(c);
  if (st != OSCAR_OK) return st;
  if (!k_new || !v_new || n_tok <= 0) return OSCAR_ERR_INVALID_ARG;
  if (!al16(k_new) || !al16(v_new)) return OSCAR_ERR_ALIGNMENT;
  // capacity of the whole call, checked before anything is launched
  {
    long long res = c->n_res, packed = c->n_packed;
    for (long long left = n_tok; left > 0;) {
      if (res == kR) {
        packed += kR;
        res = 0;
      }
      const long long m = std::min<long long>(left, kR - res);
      res += m;
      left -= m;
    }
    if (packed > c->T_cap) return OSCAR_ERR_CAPACITY;
  }
  const cudaStream_t s = as_stream(stream);
  const int rows = c->B * c->Hkv;
  for (int done = 0; done < n_tok;) {
    if (c->n_res == kR) {
      st = flush_residual(c, s);
      if (st != OSCAR_OK) return st;
    }
    const int m = std::min(n_tok - done, kR - c->n_res);
    cudaError_t e = launch_rotate_scale_k(
        k_new + (size_t)done * kD, n_tok, c->k_res, reinterpret_cast<__half*>(c->k_res_norm), kR,
        c->n_res, rows, c->Hkv, m, v_new + (size_t)done * kD, c->v_res,
        key_scale(c->flags, c->norm_target), s);
    g_launches++;
    if (e != cudaSuccess) return OSCAR_ERR_CUDA;
    c->n_res += m;
    done += m;
  }
  return OSCAR_OK;
}

int oscar_decode_num_splits(int B, int Hkv, int Hq, int n_packed) {
  const long long rows = decode_rows(B, Hkv, Hq);
  if (rows == 0) return 1;
  return plan_splits(rows, n_packed / kG, decode_int2_ctas_per_sm(Hq / Hkv), 512);
}

int oscar_decode_plan_splits(long long rows, long long n_blocks, int ctas_per_sm, int sms) {
  return plan_splits_for(rows, n_blocks, ctas_per_sm, sms, 512);
}

size_t oscar_decode_workspace_bytes(int B, int Hkv, int Hq, int n_packed, int num_splits) {
  if (B <= 0 || Hq <= 0) return 0;
  const int s = num_splits > 0 ? num_splits : oscar_decode_num_splits(B, Hkv, Hq, n_packed);
  return decode_ws_bytes(B, Hkv > 0 ? Hkv : 1, Hq, s + 1);
}

oscar_status oscar_decode_attention(const oscar_cache* c, const float* q_rot, int Hq,
                                    float softmax_scale, float* out, int num_splits,
                                    void* workspace, size_t ws_bytes, void* stream) {
  oscar_status st = check_cache(c);
  if (st != OSCAR_OK) return st;
  if (!q_rot || !out || Hq <= 0 || num_splits < 0 || num_splits > 4096 ||
      !std::isfinite(softmax_scale))
    return OSCAR_ERR_INVALID_ARG;
  const long long rows = decode_rows(c->B, c->Hkv, Hq);
  if (rows == 0 || rows > kMaxDecodeRows) return OSCAR_ERR_UNSUPPORTED;
  if (!al16(q_rot) || !al16(out)) return OSCAR_ERR_ALIGNMENT;
  int S = num_splits > 0 ? num_splits : oscar_decode_num_splits(c->B, c->Hkv, Hq, c->n_packed);
  if (!workspace || ws_bytes < decode_ws_bytes(c->B, c->Hkv, Hq, S + 1))
    return OSCAR_ERR_WORKSPACE;
  if (!al16(workspace)) return OSCAR_ERR_ALIGNMENT;
  DecodeArgs a;
  a.packed = c->packed;
  a.k_res = c->k_res;
  a.v_res = c->v_res;
  a.k_res_norm = reinterpret_cast<const __half*>(c->k_res_norm);
  a.q_rot = q_rot;
  a.ws = decode_partials(workspace);
  a.row_count = decode_row_counters(workspace);
  a.out = out;
  a.status = status_ptr();
  a.B = c->B;
  a.Hkv = c->Hkv;
  a.Hq = Hq;
  a.T_cap = c->T_cap;
  a.n_packed = c->n_packed;
  a.n_res = c->n_res;
  a.num_splits = S;
  a.slices = decode_slices(Hq / c->Hkv);
  a.flags = c->flags;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.q_exp = query_exponent(key_scale(c->flags, c->norm_target));
  a.bits = code_bits(c->bits);
  cudaError_t e = launch_decode_int2(a, as_stream(stream));
  g_launches += 1;
  return from_cuda(e);
}

oscar_status oscar_decode_step(oscar_cache* c, const oscar_bf16* q, const oscar_bf16* k_new,
                               const oscar_bf16* v_new, int Hq, float softmax_scale, float* out,
                               int num_splits, void* workspace, size_t ws_bytes, void* stream) {
  oscar_status st = check_cache(c);
  if (st != OSCAR_OK) return st;
  if (!q || !k_new || !v_new || !out || Hq <= 0 || num_splits < 0 || num_splits > 4096 ||
      !std::isfinite(softmax_scale))
    return OSCAR_ERR_INVALID_ARG;
  const long long rows = decode_rows(c->B, c->Hkv, Hq);
  if (rows == 0 || rows > kMaxDecodeRows) return OSCAR_ERR_UNSUPPORTED;
  if (!al16(q) || !al16(k_new) || !al16(v_new) || !al16(out)) return OSCAR_ERR_ALIGNMENT;
  // a full window is flushed first (flush-before-append); everything is
  // checked before anything is launched
  const bool flush = c->n_res == kR;
  const int n_packed = c->n_packed + (flush ? kR : 0);
  if (n_packed > c->T_cap) return OSCAR_ERR_CAPACITY;
  const int S = num_splits > 0 ? num_splits : oscar_decode_num_splits(c->B, c->Hkv, Hq, n_packed);
  if (!workspace || ws_bytes < decode_ws_bytes(c->B, c->Hkv, Hq, S + 1))
    return OSCAR_ERR_WORKSPACE;
  if (!al16(workspace)) return OSCAR_ERR_ALIGNMENT;
  const cudaStream_t s = as_stream(stream);
  if (flush) {
    st = flush_residual(c, s);
    if (st != OSCAR_OK) return st;
  }
  const KeyScale ks = key_scale(c->flags, c->norm_target);
  DecodeArgs a;
  a.packed = c->packed;
  a.k_res = c->k_res;
  a.v_res = c->v_res;
  a.k_res_norm = reinterpret_cast<const __half*>(c->k_res_norm);
  a.q_rot = nullptr;
  a.q_raw = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.norm_target = ks.target;
  a.ws = decode_partials(workspace);
  a.row_count = decode_row_counters(workspace);
  a.out = out;
  a.status = status_ptr();
  a.B = c->B;
  a.Hkv = c->Hkv;
  a.Hq = Hq;
  a.T_cap = c->T_cap;
  a.n_packed = c->n_packed;
  a.n_res = c->n_res + 1;   // the new token, written by the kernel
  a.num_splits = S;
  a.slices = decode_slices(Hq / c->Hkv);
  a.flags = c->flags;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.q_exp = query_exponent(ks);
  a.bits = code_bits(c->bits);
  cudaError_t e = launch_decode_int2(a, s);
  g_launches += 1;
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  c->n_res += 1;
  return OSCAR_OK;
}

// ------------------------------------------------------------------ paged

}  // extern "C"

namespace {

inline bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

oscar_status check_paged(const oscar_paged_cache* c) {
  if (!c) return OSCAR_ERR_INVALID_ARG;
  if (c->B <= 0 || c->Hkv <= 0 || c->max_blocks <= 0 || c->n_pages <= 0)
    return OSCAR_ERR_INVALID_ARG;
  // the kernels index the block table with 32-bit entry numbers
  if ((long long)c->B * c->max_blocks > 0x7fffffffLL) return OSCAR_ERR_UNSUPPORTED;
  const void* p16[] = {c->pages, c->k_res, c->v_res, c->k_res_norm};
  for (const void* p : p16) {
    if (!p) return OSCAR_ERR_INVALID_ARG;
    if (!al16(p)) return OSCAR_ERR_ALIGNMENT;
  }
  const void* p4[] = {c->block_table, c->n_packed, c->n_res};
  for (const void* p : p4) {
    if (!p) return OSCAR_ERR_INVALID_ARG;
    if (!al4(p)) return OSCAR_ERR_ALIGNMENT;
  }
  if ((c->flags & ~kAllFlags) || !target_ok(c->norm_target) || !key_group_ok(c->key_group) ||
      !code_bits_ok(c->bits))
    return OSCAR_ERR_INVALID_ARG;
  return OSCAR_OK;
}

PagedArgs paged_args(const oscar_paged_cache* c) {
  PagedArgs p;
  p.pages = c->pages;
  p.block_table = c->block_table;
  p.seq_packed = c->n_packed;
  p.seq_res = c->n_res;
  p.k_res = c->k_res;
  p.v_res = c->v_res;
  p.k_res_norm = reinterpret_cast<__half*>(c->k_res_norm);
  p.status = status_ptr();
  p.B = c->B;
  p.Hkv = c->Hkv;
  p.max_blocks = c->max_blocks;
  p.n_pages = c->n_pages;
  p.ks = key_scale(c->flags, c->norm_target);
  p.group = key_group(c->key_group);
  p.bits = code_bits(c->bits);
  return p;
}

}  // namespace

extern "C" {

oscar_status oscar_paged_prefill_kv(oscar_paged_cache* c, const oscar_bf16* k,
                                    const oscar_bf16* v, int in_T, const int32_t* n_tok,
                                    int max_tok, void* stream) {
  oscar_status st = check_paged(c);
  if (st != OSCAR_OK) return st;
  if (!k || !v || !n_tok) return OSCAR_ERR_INVALID_ARG;
  if (!al16(k) || !al16(v) || !al4(n_tok)) return OSCAR_ERR_ALIGNMENT;
  const int G = key_group(c->key_group);
  if (max_tok < G || max_tok % G != 0 || in_T < max_tok) return OSCAR_ERR_INVALID_ARG;
  if (max_tok / kG > c->max_blocks) return OSCAR_ERR_CAPACITY;
  const PagedArgs p = paged_args(c);
  if (!p.status) return OSCAR_ERR_CUDA;
  cudaError_t e = launch_paged_prefill(p, k, v, in_T, n_tok, max_tok, as_stream(stream));
  g_launches += 2;
  return from_cuda(e);
}

oscar_status oscar_paged_append_kv(oscar_paged_cache* c, const oscar_bf16* k_new,
                                   const oscar_bf16* v_new, const int32_t* active, void* stream) {
  oscar_status st = check_paged(c);
  if (st != OSCAR_OK) return st;
  if (!k_new || !v_new) return OSCAR_ERR_INVALID_ARG;
  if (!al16(k_new) || !al16(v_new) || (active && !al4(active))) return OSCAR_ERR_ALIGNMENT;
  const PagedArgs p = paged_args(c);
  if (!p.status) return OSCAR_ERR_CUDA;
  cudaError_t e = launch_paged_append(p, k_new, v_new, active, as_stream(stream));
  g_launches += 3;
  return from_cuda(e);
}

oscar_status oscar_paged_decode_attention(const oscar_paged_cache* c, const float* q_rot, int Hq,
                                          float softmax_scale, int max_packed, float* out,
                                          int num_splits, void* workspace, size_t ws_bytes,
                                          void* stream) {
  oscar_status st = check_paged(c);
  if (st != OSCAR_OK) return st;
  if (!q_rot || !out || Hq <= 0 || num_splits < 0 || num_splits > 4096 ||
      !std::isfinite(softmax_scale) || max_packed < 0 || max_packed % kG != 0 ||
      max_packed / kG > c->max_blocks)
    return OSCAR_ERR_INVALID_ARG;
  const long long rows = decode_rows(c->B, c->Hkv, Hq);
  if (rows == 0 || rows > kMaxDecodeRows) return OSCAR_ERR_UNSUPPORTED;
  if (!al16(q_rot) || !al16(out)) return OSCAR_ERR_ALIGNMENT;
  int S = num_splits > 0 ? num_splits : oscar_decode_num_splits(c->B, c->Hkv, Hq, max_packed);
  if (!workspace || ws_bytes < decode_ws_bytes(c->B, c->Hkv, Hq, S + 1))
    return OSCAR_ERR_WORKSPACE;
  if (!al16(workspace)) return OSCAR_ERR_ALIGNMENT;
  DecodeArgs a;
  a.packed = c->pages;
  a.k_res = c->k_res;
  a.v_res = c->v_res;
  a.k_res_norm = reinterpret_cast<const __half*>(c->k_res_norm);
  a.q_rot = q_rot;
  a.ws = decode_partials(workspace);
  a.row_count = decode_row_counters(workspace);
  a.out = out;
  a.status = status_ptr();
  if (!a.status) return OSCAR_ERR_CUDA;
  a.B = c->B;
  a.Hkv = c->Hkv;
  a.Hq = Hq;
  a.T_cap = 0;
  a.n_packed = max_packed;  // sizes the equal chunks of the splits
  a.n_res = 0;
  a.num_splits = S;
  a.slices = decode_slices(Hq / c->Hkv);
  a.flags = c->flags;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.q_exp = query_exponent(key_scale(c->flags, c->norm_target));
  a.bits = code_bits(c->bits);
  a.block_table = c->block_table;
  a.seq_packed = c->n_packed;
  a.seq_res = c->n_res;
  a.max_blocks = c->max_blocks;
  a.n_pages = c->n_pages;
  cudaError_t e = launch_decode_int2(a, as_stream(stream));
  g_launches += 1;
  return from_cuda(e);
}

oscar_status oscar_bf16_decode_attention(const oscar_bf16* q, const oscar_bf16* K,
                                         const oscar_bf16* V, int B, int Hq, int Hkv, int T,
                                         int T_stride, float softmax_scale, float* out,
                                         int num_splits, void* workspace, size_t ws_bytes,
                                         void* stream) {
  if (!q || !K || !V || !out || B <= 0 || Hq <= 0 || Hkv <= 0 || T < 0 || T_stride < T ||
      num_splits < 0 || num_splits > 4096 || !std::isfinite(softmax_scale))
    return OSCAR_ERR_INVALID_ARG;
  const long long rows = decode_rows(B, Hkv, Hq);
  if (rows == 0) return OSCAR_ERR_UNSUPPORTED;
  // grid (splits, Hkv x slices, B)
  if (B > 65535 || rows / B > 65535) return OSCAR_ERR_UNSUPPORTED;
  if (!al16(q) || !al16(K) || !al16(V) || !al16(out)) return OSCAR_ERR_ALIGNMENT;
  int S = num_splits;
  if (S == 0) {
    const long long chunk = 16;  // tokens per warp chunk, the unit of work here
    S = plan_splits_bf16(rows, (T + chunk - 1) / chunk, decode_bf16_ctas_per_sm(Hq / Hkv), 512);
  }
  if (!workspace || ws_bytes < ws_bytes_for(B, Hq, S)) return OSCAR_ERR_WORKSPACE;
  if (!al16(workspace)) return OSCAR_ERR_ALIGNMENT;
  Bf16DecodeArgs a;
  a.q = q;
  a.K = K;
  a.V = V;
  a.ws = static_cast<float*>(workspace);
  a.out = out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.T = T;
  a.T_stride = T_stride;
  a.num_splits = S;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  cudaError_t e = launch_decode_bf16(a, as_stream(stream));
  g_launches += 2;
  return from_cuda(e);
}

oscar_status oscar_selftest_wait_timeout(unsigned iterations, void* stream) {
  if (iterations == 0 || iterations > (1u << 20)) return OSCAR_ERR_INVALID_ARG;
  unsigned* p = status_ptr();
  if (!p) return OSCAR_ERR_CUDA;
  cudaError_t e = launch_wait_timeout_selftest(p, iterations, as_stream(stream));
  g_launches++;
  return from_cuda(e);
}

oscar_status oscar_device_status(void* stream) {
  unsigned* p = status_ptr();
  if (!p) return OSCAR_ERR_CUDA;
  const cudaStream_t s = as_stream(stream);
  unsigned v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return OSCAR_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(unsigned), s) != cudaSuccess) return OSCAR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return OSCAR_ERR_CUDA;
  return v ? OSCAR_ERR_DEVICE_STATUS : OSCAR_OK;
}

const char* oscar_status_string(oscar_status s) {
  switch (s) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported configuration";
    case OSCAR_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case OSCAR_ERR_CAPACITY: return "cache capacity exceeded";
    case OSCAR_ERR_WORKSPACE: return "workspace missing or too small";
    case OSCAR_ERR_CUDA: return "CUDA runtime error";
    case OSCAR_ERR_DEVICE_STATUS: return "a kernel recorded an error";
  }
  return "unknown status";
}

unsigned long long oscar_kernel_launches(void) { return g_launches.load(); }

}  // extern "C"
