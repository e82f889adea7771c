// oscar_decode_attention_static_ws: the fused INT2 decode attention for
// callers that cannot allocate device memory.
//
// oscar_decode_attention needs a caller-provided workspace for its split-K
// partial records.  Some callers have no way to provide one: code that runs
// where every device allocation must happen once at start-up (a serving loop
// that forbids cudaMalloc after warm-up because it can block the device and
// fragment memory), or a plug-in inside a runtime that owns all device memory
// and exposes no allocator to it.  This entry point keeps the partials in a
// fixed array in the library's own device memory instead, so the caller
// passes only the cache, the queries and the output.
//
// The array is a file-scope static __device__ variable: every GPU that loads
// the library holds OSCAR_STATIC_SCRATCH_BYTES of it until the process exits.
// Host code only sees a stand-in for it, so its device address is looked up
// with cudaGetSymbolAddress, once per device, on the first call made while
// that device is current; make that first call before any stream capture.
// All calls share the one array: calls whose kernels overlap on the GPU (two
// streams, say) race on it and give wrong results.  The array is laid out as
// a decode workspace: a header of per-row arrival counters, which must be
// zero when a call starts (static device memory starts zeroed and every call
// leaves them zero), then the partial records, which every call writes
// before it reads them.  Otherwise it keeps whatever the last call left.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

using namespace oscar;

constexpr size_t kScratchBytes = OSCAR_STATIC_SCRATCH_BYTES;
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

std::mutex g_scratch_mu;
float* g_scratch_addr[128] = {};

// Device address of g_decode_scratch on the current device (set up on first use).
float* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  return g_scratch_addr[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" oscar_status oscar_decode_attention_static_ws(const oscar_cache* c,
                                                         const float* q_rot, int Hq,
                                                         float softmax_scale, float* out,
                                                         int num_splits, void* stream) {
  // the same argument checks as oscar_decode_attention
  const oscar_status st = validate_cache(c);
  if (st != OSCAR_OK) return st;
  if (!q_rot || !out || Hq <= 0 || num_splits < 0 || num_splits > 4096 ||
      !std::isfinite(softmax_scale))
    return OSCAR_ERR_INVALID_ARG;
  const long long rows = decode_rows(c->B, c->Hkv, Hq);
  if (rows == 0 || rows > kMaxDecodeRows) return OSCAR_ERR_UNSUPPORTED;
  if (!aligned16(q_rot) || !aligned16(out)) return OSCAR_ERR_ALIGNMENT;

  // The partial records and counters must fit in the static array.  An
  // automatic split count is lowered to the largest that fits; an explicit
  // one that does not fit is refused.
  int S = num_splits;
  if (S == 0) {
    S = oscar_decode_num_splits(c->B, c->Hkv, Hq, c->n_packed);
    const size_t per_part = (size_t)c->B * (size_t)Hq * kRecFloats * sizeof(float);
    const long long parts = (long long)((kScratchBytes - kDecodeWsHeader) / per_part);
    if (S + 1 > parts) S = (int)(parts - 1);
    if (S < 1) return OSCAR_ERR_WORKSPACE;
  }
  if (decode_ws_bytes(c->B, c->Hkv, Hq, S + 1) > kScratchBytes) return OSCAR_ERR_WORKSPACE;

  float* ws = scratch_address();
  if (!ws) return OSCAR_ERR_CUDA;

  DecodeArgs a;
  a.packed = c->packed;
  a.k_res = c->k_res;
  a.v_res = c->v_res;
  a.k_res_norm = reinterpret_cast<const __half*>(c->k_res_norm);
  a.q_rot = q_rot;
  a.ws = decode_partials(ws);
  a.row_count = decode_row_counters(ws);
  a.out = out;
  a.status = device_status_word();
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
  cudaError_t e = launch_decode_int2(a, static_cast<cudaStream_t>(stream));
  count_launches(1);
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
