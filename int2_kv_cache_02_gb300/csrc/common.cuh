// Device helpers shared by the liboscar kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/oscar.h"

namespace oscar {

constexpr int kD = OSCAR_HEAD_DIM;
constexpr int kG = OSCAR_GROUP;
constexpr int kR = OSCAR_RESIDUAL;

// Byte offsets inside one packed 32-token block record (include/oscar.h).
constexpr int kBlkBytes = OSCAR_BLOCK_BYTES;
constexpr int kRecKC = 0, kRecVC = 1024, kRecKS = 2048, kRecKZ = 2304, kRecKN = 2560,
              kRecVS = 2624, kRecVZ = 2688;
static_assert(kRecVZ + 64 == kBlkBytes, "record layout");
// The record of one 32-token block for a code width of BITS (2: the method's
// INT2 record above; 4: the INT4 option, twice the code bytes, the same side
// arrays after them).
template <int BITS>
struct Rec;
template <>
struct Rec<2> {
  static constexpr int KC = 0, VC = 1024, KS = 2048, KZ = 2304, KN = 2560, VS = 2624, VZ = 2688,
                       BYTES = 2752;
};
template <>
struct Rec<4> {
  static constexpr int KC = 0, VC = 2048, KS = 4096, KZ = 4352, KN = 4608, VS = 4672, VZ = 4736,
                       BYTES = 4800;
};
static_assert(Rec<2>::BYTES == kBlkBytes && Rec<4>::BYTES == OSCAR_BLOCK_BYTES_INT4, "records");
__host__ __device__ constexpr int rec_bytes(int bits) { return bits == 4 ? Rec<4>::BYTES : Rec<2>::BYTES; }

// Position of token t (0..31) of a block in the record's per-token arrays
// (norms, value step, value zero): tokens i, i+8, i+16, i+24 are adjacent.
__host__ __device__ constexpr int tok_slot(int t) { return 4 * (t & 7) + (t >> 3); }

// Bits a kernel may OR into the device status word.
enum : unsigned {
  kDevErrWaitTimeout = 1u,   // an mbarrier wait hit its iteration limit
  kDevErrDrainTimeout = 2u,  // copies still in flight after the drain limit
  kDevErrBadPaged = 4u,      // a page id or a per-sequence length out of range
  kDevErrArrival = 8u,       // a decode row's arrival counter was not zero at the start
};

// Iteration limits of the bounded spin-waits.  One try_wait may itself
// suspend for a while, so these bound the wait at a few seconds.
constexpr unsigned kWaitLimit = 1u << 24;
constexpr unsigned kDrainLimit = 1u << 20;

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` at most `limit` polls.  Returns false on
// timeout (the caller records it and leaves).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, unsigned limit) {
  for (unsigned i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared through the TMA unit, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void record_error(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

// ---- small numeric helpers ------------------------------------------------

__device__ __forceinline__ __half2 u32_as_half2(uint32_t u) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = u;
  return h;
}

__device__ __forceinline__ uint32_t half2_as_u32(__half2 h) {
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
// Both bf16 of a packed pair as fp32, the low one in x.
__device__ __forceinline__ float2 bf16_pair(uint32_t u) { return make_float2(bf16_lo(u), bf16_hi(u)); }

// Packed fp32 arithmetic (one instruction for two IEEE operations, each half
// rounded to nearest even exactly as the scalar operation).  a - b is the
// fused multiply-add b * -1 + a: one rounding of the exact difference.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, const float (&c)[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// D += A(16x16 f16, row) * B(16x8 f16, col), fp32 accumulate in place (the
// accumulator registers are both read and written, so no copies are needed).
__device__ __forceinline__ void mma_16816_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace oscar
