// quant_row.cuh -- the activation quantiser's work on one row, shared by the standalone
// quantiser (quantize.cu) and the MMQ's fused prologue (mmq.cu).  The arithmetic of every
// block is fixed (below) and the row maximum is order-independent, so the bytes written do
// not depend on the thread count.
//
// Per row m and 32-element block b, in IEEE binary32:
//   amax = max |x|;  s = amax / 127 (correctly rounded division);
//   q = round_half_even(x / s) clamped to [-127, 127], or 0 when s == 0;
//   S = sum q.
// Writes every section of the xq buffer (mq_act_bytes) for the row: q as int8, s as f32,
// S as int32, q as f16 (the tensor-core operand of the MMQ), the transposed s and s*S
// planes, and the min-term operand: a power of two u_m with max_b |s*S| / u_m in
// [2^13, 2^14) and the f16 pair (hi, lo) of t~ = s*S / u_m per block, laid out as
// [hi | hi | lo].
//
// quantize_row: a group of NT threads (tid = 0..NT-1 within the group) for one row (8
// threads per block, 4 elements each, NT / 8 blocks per pass, PRE passes loaded at a time);
// it synchronises the group once, with __syncthreads when bar < 0 (the group is the whole
// CTA) and otherwise with the named barrier bar of NT threads.  ttc: shared scratch of
// kTtCache floats; wmax: shared scratch of NT / 32 floats; both may be reused only after
// the group's next synchronisation.
#pragma once

#include "mq_common.cuh"

namespace mq {

constexpr int kTtCache = 2048;  // s*S of a row's first blocks kept in shared memory

// q = clamp(rint(fl(x / s)), -127, 127) for s > 0 (f32 division correctly rounded, then
// round half to even), returned as the binary32 value t = 1.5 * 2^23 + q: its low byte is q
// as int8, its bits less those of 1.5 * 2^23 are q, and t - 1.5 * 2^23 is q as a float.
// Computed as w = fl(x * r) with r = fl(1 / s), rounded to an integer by adding 1.5 * 2^23
// (ties to even, exact for |w| < 2^22), and by the division itself only when w is within
// 2^-14 of a half-integer (its residual d = w - rint(w), exact, has |d| >= 1/2 - 2^-14), or
// |w| >= 127.25, or w is not finite.  Why that is exact: |r - 1/s| <= 2^-24 / s and
// |w - x r| <= 2^-24 |x r|, so with |x / s| <= 127.25 |w - x/s| < 2^-16, and the quotient
// v = fl(x / s) has |v - x/s| < 2^-17; so |w - v| < 2^-15.  If every half-integer is at
// least 2^-14 from w, v lies on the same side of each as w and is not one itself, so both
// round to the same integer, which is within [-127, 127].  (A subnormal s can make r
// infinite; then w is not finite and the division runs.)
// s = fl(amax / 127) (correctly rounded) without the division: q0 = fl(amax * c) with
// c = fl(1 / 127), the remainder amax - 127 q0 by one fma (exact), and one fma correction
// fl(q0 + r c), the correction step of Markstein's division by a correctly rounded
// reciprocal.  It gives the correctly rounded quotient for every non-negative finite binary32
// amax (checked exhaustively, subnormals included, in tests/test_quant_rule_cpu.py); a
// non-finite amax takes the division itself.
__device__ __forceinline__ float div127(float a) {
  constexpr float c = 0x1.020408p-7f;  // fl(1 / 127)
  const float q0 = __fmul_rn(a, c);
  const float r = __fmaf_rn(-q0, 127.0f, a);
  const float q1 = __fmaf_rn(r, c, q0);
  return a < INFINITY ? q1 : __fdiv_rn(a, 127.0f);
}

constexpr float kQuantMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kQuantMagicBits = 0x4B400000;
// max that propagates NaN (a NaN operand must send its lane's codes to the division)
__device__ __forceinline__ float max_nan(float a, float b) {
  float m;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(m) : "f"(a), "f"(b));
  return m;
}
// The codes of one lane's four elements v as above: t[k] = 1.5 * 2^23 + q_k, and q_k as a
// float.  The arithmetic runs on f32 pairs (w - rint(w) as fma(rint(w), -1, w), exact), and
// one test of the four residuals and magnitudes decides; if any fails, all four codes come
// from the division (which gives every code, the passing ones included).
__device__ __forceinline__ void quant_codes4(const float4 v, float s, float r, float (&t)[4],
                                             float (&qf)[4]) {
  const float2 r2 = make_float2(r, r), m2 = make_float2(kQuantMagic, kQuantMagic);
  const float2 nm2 = make_float2(-kQuantMagic, -kQuantMagic), neg = make_float2(-1.f, -1.f);
  const float2 w01 = __fmul2_rn(make_float2(v.x, v.y), r2);
  const float2 w23 = __fmul2_rn(make_float2(v.z, v.w), r2);
  const float2 t01 = __fadd2_rn(w01, m2), t23 = __fadd2_rn(w23, m2);
  const float2 q01 = __fadd2_rn(t01, nm2), q23 = __fadd2_rn(t23, nm2);
  const float2 d01 = __ffma2_rn(q01, neg, w01), d23 = __ffma2_rn(q23, neg, w23);
  const float dm = max_nan(max_nan(fabsf(d01.x), fabsf(d01.y)), max_nan(fabsf(d23.x), fabsf(d23.y)));
  const float wm = max_nan(max_nan(fabsf(w01.x), fabsf(w01.y)), max_nan(fabsf(w23.x), fabsf(w23.y)));
  t[0] = t01.x, t[1] = t01.y, t[2] = t23.x, t[3] = t23.y;
  qf[0] = q01.x, qf[1] = q01.y, qf[2] = q23.x, qf[3] = q23.y;
  if (dm < 0.5f - 0x1p-14f && wm < 127.25f) return;
  const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    qf[k] = (float)min(max(__float2int_rn(__fdiv_rn(x[k], s)), -127), 127);
    t[k] = __fadd_rn(qf[k], kQuantMagic);
  }
}

// The loads of one round of a row (PRE passes of NT / 8 blocks from block p0 on): thread
// tid's float4 of each pass, zeros past the row's end.  xrow: the row in global memory.
template <int NT, int PRE>
__device__ __forceinline__ void quant_row_load(const float *__restrict__ xrow, int64_t K,
                                               int64_t p0, int tid, float4 (&vp)[PRE]) {
  const int64_t nb = K / 32;
  const int tb = tid >> 3, sub = tid & 7;
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int64_t b = p0 + (NT / 8) * k + tb;
    vp[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (b < nb) vp[k] = __ldg(reinterpret_cast<const float4 *>(xrow + b * 32) + sub);
  }
}

// One 32-element block of row m: the 8 lanes sub = 0..7 of a group of 8 hold its elements
// 4 sub .. 4 sub + 3 in v (every lane of the warp takes part in the shuffles; lanes of
// blocks past the row's end carry zeros and store nothing).  Writes the block's q, f16 q,
// s, S, and the transposed s and s*S; keeps s*S in ttc (blocks below TTC) and the
// largest |s*S| in rowmax (lane sub == 0).
template <int TTC = kTtCache>
__device__ __forceinline__ void quant_block(const float4 v, int64_t b, bool ok, int64_t m,
                                            int64_t nb, const ActLayout &L,
                                            uint8_t *__restrict__ xq, float *ttc, int sub,
                                            float &rowmax) {
  const int64_t blk = m * nb + b;  // global block index
  float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  const float s = div127(mx);
  float t[4] = {kQuantMagic, kQuantMagic, kQuantMagic, kQuantMagic}, qf[4] = {0.f, 0.f, 0.f, 0.f};
  if (s != 0.0f) quant_codes4(v, s, __frcp_rn(s), t, qf);
  const int i0 = __float_as_int(t[0]), i1 = __float_as_int(t[1]), i2 = __float_as_int(t[2]),
            i3 = __float_as_int(t[3]);
  int S = (i0 + i1) + (i2 + i3) - 4 * kQuantMagicBits;
  S += __shfl_xor_sync(0xffffffffu, S, 1);
  S += __shfl_xor_sync(0xffffffffu, S, 2);
  S += __shfl_xor_sync(0xffffffffu, S, 4);
  if (!ok) return;
  // the low bytes of t0..t3 are q0..q3 as int8
  const uint32_t packed =
      __byte_perm(__byte_perm(i0, i1, 0x0040u), __byte_perm(i2, i3, 0x0040u), 0x5410u);
  reinterpret_cast<uint32_t *>(xq + L.qs)[blk * 8 + sub] = packed;
  __half2 h01 = __floats2half2_rn(qf[0], qf[1]);
  __half2 h23 = __floats2half2_rn(qf[2], qf[3]);
  uint2 hv;
  hv.x = *reinterpret_cast<uint32_t *>(&h01);
  hv.y = *reinterpret_cast<uint32_t *>(&h23);
  reinterpret_cast<uint2 *>(xq + L.op)[blk * 8 + sub] = hv;
  if (sub == 0) {
    const float t = s * (float)S;
    reinterpret_cast<float *>(xq + L.scale)[blk] = s;
    reinterpret_cast<int32_t *>(xq + L.bsum)[blk] = S;
    reinterpret_cast<float *>(xq + L.st)[b * L.mt + m] = s;
    reinterpret_cast<float *>(xq + L.tt)[b * L.mt + m] = t;
    if (b < TTC) ttc[b] = t;
    rowmax = fmaxf(rowmax, fabsf(t));
  }
}

// The row's min-term operand, once its maximum |s*S| (mxr) is known: a power of two u_m
// with mxr / u_m in [2^13, 2^14), and the f16 pair (hi, lo) of s*S / u_m per block, laid out
// [hi | hi | lo]; threads tid = 0 .. NT - 1 of the row's group share the blocks; s*S from
// ttc for blocks below TTC, else read back from the xq buffer.
template <int NT, int TTC = kTtCache>
__device__ __forceinline__ void quant_row_finish(float mxr, int64_t m, int64_t nb,
                                                 const ActLayout &L, uint8_t *__restrict__ xq,
                                                 const float *ttc, int tid) {
  const int E = (int)((__float_as_uint(mxr) >> 23) & 255);
  int k = mxr == 0.f ? 0 : E - 140;
  k = min(max(k, -100), 100);
  const float inv_u = __int_as_float((127 - k) << 23);
  if (tid == 0) reinterpret_cast<float *>(xq + L.urow)[m] = __int_as_float((127 + k) << 23);
  __half *arow = reinterpret_cast<__half *>(xq + L.amin) + m * min_ld(nb);
  for (int64_t b = tid; b < nb; b += NT) {
    const float t =
        (b < TTC ? ttc[b] : reinterpret_cast<const float *>(xq + L.tt)[b * L.mt + m]) * inv_u;
    const __half hi = __float2half_rn(t);
    const __half lo = __float2half_rn(t - __half2float(hi));
    arow[b] = hi;
    arow[nb + b] = hi;
    arow[2 * nb + b] = lo;
  }
}

// xrow: row m of x; a group of NT threads (tid = 0 .. NT - 1), PRE passes of NT / 8 blocks
// loaded at a time.  It synchronises the group once, with __syncthreads when bar < 0 (the
// group is the whole CTA) and otherwise with the named barrier bar of NT threads.
template <int NT, int PRE = 4>
__device__ __forceinline__ void quantize_row(const float *__restrict__ xrow, uint8_t *__restrict__ xq,
                                             int64_t m, int64_t K, const ActLayout &L, float *ttc,
                                             float *wmax, int tid, int bar) {
  const int64_t nb = K / 32;
  const int tb = tid >> 3, sub = tid & 7;  // block in pass, lane in block
  float rowmax = 0.f;
  // passes of kPass blocks, kPre of them loaded before any is processed (one load latency
  // per kPre passes)
  constexpr int kPass = NT / 8, kPre = PRE;
  for (int64_t p0 = 0; p0 < nb; p0 += kPass * kPre) {
    float4 vp[kPre];
    quant_row_load<NT, PRE>(xrow, K, p0, tid, vp);
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const int64_t b = p0 + kPass * k + tb;
      quant_block(vp[k], b, b < nb, m, nb, L, xq, ttc, sub, rowmax);
    }
  }
  // row maximum of |s*S|
  rowmax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(rowmax)));
  if ((tid & 31) == 0) wmax[tid >> 5] = rowmax;
  if (bar < 0)
    __syncthreads();
  else
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(NT) : "memory");
  float mxr = wmax[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) mxr = fmaxf(mxr, wmax[w]);
  quant_row_finish<NT>(mxr, m, nb, L, xq, ttc, tid);
}

}  // namespace mq
