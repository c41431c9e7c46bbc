// mv_device.cuh -- device helpers shared by the decode matvec kernels (matvec.cu,
// matvec_kq.cu and xplane.cu): the warp-level f16 tensor-core MMA, packed f16 arithmetic,
// f16 / bf16 packing, mbarrier waits bounded by %globaltimer, 1-D bulk copies, and the layout
// of the activation fragment plane.
#pragma once

#include <cuda_bf16.h>

#include "mq_common.cuh"

namespace mq {
namespace mvd {

constexpr uint64_t kWaitNs = 2000000000ull;  // bounded mbarrier waits: 2 s

// The activation fragment plane of a Q4_K / Q5_K two-tile call (B = 5..8) of the persistent
// matvec: x
// converted once per call by xplane_kernel (xplane.cu) into the B fragments that the x warps
// would otherwise form in every CTA; the kernel bulk-copies each chunk's part into a fragment
// slot.  Per 256-element chunk, NT n8 tiles (4 batch rows each): the fragment groups
// [kXpGroups][NT][32 + xp_pad(NT)] of uint2 (the kernel's shared-memory slot layout: 16
// groups of 16 elements, then the Q4_K / Q5_K min-term group), then the unscale factor 2^-e
// of each of the 4 NT rows (0 for rows past B), padded to 8 floats.  Both sections are
// multiples of 16 bytes.
constexpr int kXpGroups = 17;
__host__ __device__ constexpr int xp_pad(int nt) { return nt == 1 ? 4 : 2; }
__host__ __device__ constexpr int xp_group_bytes(int nt) { return nt * (32 + xp_pad(nt)) * 8; }
__host__ __device__ constexpr int xp_off_unscale(int nt) { return kXpGroups * xp_group_bytes(nt); }
__host__ __device__ constexpr int xp_chunk_bytes(int nt) { return xp_off_unscale(nt) + 32; }
static_assert(xp_group_bytes(1) % 16 == 0 && xp_group_bytes(2) % 16 == 0,
              "fragment groups must keep the bulk copies 16-byte aligned");

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// the same with a zero accumulator (c = a * b)
__device__ __forceinline__ void mma16816_z(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// bf16 operands (unquantised bf16 weights, bf16 hi/lo activation parts)
__device__ __forceinline__ void mma16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// (a & b) | c as one three-input logic instruction (written out so that two
// constant operands do not turn it into two instructions)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ int chunk_width(int64_t K, int c) {
  const int64_t left = K - int64_t(c) * kChunk;
  return left < kChunk ? (int)left : kChunk;
}
__device__ __forceinline__ uint32_t sa(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; on expiry records (timeout, site) in the status word and returns.
__device__ __forceinline__ void mbar_wait(uint32_t a, uint32_t parity, int *status, int site) {
  if (mbar_try(a, parity)) return;
  const uint64_t t0 = gtime();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try(a, parity)) return;
    if (gtime() - t0 > kWaitNs) {
      if (atomicCAS(status, 0, kStatusTimeout) == 0) atomicExch(status + 1, site);
      return;
    }
  }
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
// arrive, and expect `bytes` more of the transaction count (one arrival of the barrier)
__device__ __forceinline__ void mbar_arrive_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_1d(uint32_t dst, const void *src, uint32_t bytes,
                                        uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Shift left by sh (right by -sh when negative); sh is a constant once the loops that
// compute it are unrolled, so the branch folds away.
__device__ __forceinline__ uint32_t shl(uint32_t v, int sh) {
  return sh >= 0 ? v << sh : v >> (-sh);
}

}  // namespace mvd
}  // namespace mq
