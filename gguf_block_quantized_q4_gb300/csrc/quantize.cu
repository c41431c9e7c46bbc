// quantize.cu -- activation quantiser for the prefill MMQ ("minfer CUDA Backend
// Design" §4.4: prefill quantises A into per-32 int8 blocks; "minfer
// Architecture Execution Plan" C4 S2b design decision 4: amax/127 and round
// half to even, the same steps on every backend so the bytes agree exactly).
//
// Per row m and 32-element block b, in IEEE binary32:
//   amax = max |x|;  s = amax / 127 (correctly rounded division);
//   q = round_half_even(x / s) clamped to [-127, 127], or 0 when s == 0;
//   S = sum q.
// Writes every section of the xq buffer (mq_act_bytes): q as int8, s as f32,
// S as int32, q as f16 (the tensor-core operand of mq_mmq), and the transposed
// s and s*S planes the MMQ epilogue stages per 128-row tile.
//
// Memory-bound: 8 threads per block, 4 elements (one float4) per thread; the
// block's max and sum reduce over the 8 lanes with shuffles.
#include "mq_common.cuh"

namespace mq {
namespace {

__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x,
                                                           uint8_t *__restrict__ xq, int64_t M,
                                                           int64_t K, ActLayout L) {
  const int64_t nblk = M * (K / 32);
  const int64_t gt = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  const int64_t blk = gt >> 3;  // global block index m*(K/32) + b
  const int sub = threadIdx.x & 7;
  const bool ok = blk < nblk;
  // every lane of a warp takes part in the shuffles; out-of-range lanes carry zeros
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (ok) v = __ldg(reinterpret_cast<const float4 *>(x + blk * 32) + sub);
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  const float s = __fdiv_rn(m, 127.0f);
  int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
  if (s != 0.0f) {
    q0 = min(max(__float2int_rn(__fdiv_rn(v.x, s)), -127), 127);
    q1 = min(max(__float2int_rn(__fdiv_rn(v.y, s)), -127), 127);
    q2 = min(max(__float2int_rn(__fdiv_rn(v.z, s)), -127), 127);
    q3 = min(max(__float2int_rn(__fdiv_rn(v.w, s)), -127), 127);
  }
  int S = q0 + q1 + q2 + q3;
  S += __shfl_xor_sync(0xffffffffu, S, 1);
  S += __shfl_xor_sync(0xffffffffu, S, 2);
  S += __shfl_xor_sync(0xffffffffu, S, 4);
  if (!ok) return;
  const uint32_t packed = (uint32_t)(q0 & 255) | ((uint32_t)(q1 & 255) << 8) |
                          ((uint32_t)(q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
  reinterpret_cast<uint32_t *>(xq + L.qs)[blk * 8 + sub] = packed;
  __half2 h01 = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
  __half2 h23 = __halves2half2(__int2half_rn(q2), __int2half_rn(q3));
  uint2 hv;
  hv.x = *reinterpret_cast<uint32_t *>(&h01);
  hv.y = *reinterpret_cast<uint32_t *>(&h23);
  reinterpret_cast<uint2 *>(xq + L.op)[blk * 8 + sub] = hv;
  if (sub == 0) {
    reinterpret_cast<float *>(xq + L.scale)[blk] = s;
    reinterpret_cast<int32_t *>(xq + L.bsum)[blk] = S;
    const int64_t nb = K / 32, m = blk / nb, b = blk - m * nb;
    reinterpret_cast<float *>(xq + L.st)[b * L.mt + m] = s;
    reinterpret_cast<float *>(xq + L.tt)[b * L.mt + m] = s * (float)S;
  }
}

}  // namespace

mq_status launch_quantize(const float *x, void *xq, int64_t M, int64_t K, cudaStream_t s) {
  const int64_t threads = M * (K / 32) * 8;
  const int T = 256;
  const int64_t grid = (threads + T - 1) / T;
  if (grid > 0x7fffffff) return fail(MQ_ERR_SHAPE, "mq_quantize_act: M*K too large");
  quantize_act_kernel<<<(unsigned)grid, T, 0, s>>>(x, (uint8_t *)xq, M, K, act_layout(M, K));
  MQ_LAUNCH_CHECK("quantize_act_kernel");
  return MQ_OK;
}

}  // namespace mq
