// quantize.cu -- activation quantiser for the prefill MMQ ("minfer CUDA Backend
// Design" §4.4: prefill quantises A into per-32 int8 blocks; "minfer
// Architecture Execution Plan" C4 S2b design decision 4: amax/127 and round
// half to even, the same steps on every backend so the bytes agree exactly).
//
// The per-row arithmetic and the sections written are in quant_row.cuh.  Few rows: one CTA
// of 256 threads per row: 8 threads per block, 4 elements (one float4) per thread, 32
// blocks per pass; the block's max and sum reduce over the 8 lanes with shuffles, the row
// maximum of |s*S| over the CTA.  The min-term operand lets the MMQ's tensor cores form the
// min term sum_b t~ * (dmin*m_j~) from three exact f16 products per block.  (A kernel with
// one warp per row and loads pipelined eight passes ahead measured slower at 2048 rows,
// 19.1 against 15.8 us: the per-block arithmetic, not the loads, bounds it there.)
#include "quant_row.cuh"

namespace mq {
namespace {

__global__ void __launch_bounds__(256, 4) quantize_act_kernel(const float *__restrict__ x,
                                                           uint8_t *__restrict__ xq, int64_t M,
                                                           int64_t K, ActLayout L) {
  __shared__ float ttc[kTtCache];
  __shared__ float wmax[8];
  // launched with programmatic stream serialisation: the MMQ that follows may start its
  // set-up at once, and this grid reads x and writes xq only after the previous one is done
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  quantize_row<256>(x + int64_t(blockIdx.x) * K, xq, blockIdx.x, K, L, ttc, wmax, threadIdx.x, -1);
}

}  // namespace

mq_status launch_quantize(const float *x, void *xq, int64_t M, int64_t K, cudaStream_t s) {
  if (M > 0x7fffffff) return fail(MQ_ERR_SHAPE, "mq_quantize_act: M too large");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_act_kernel, x, (uint8_t *)xq, M, K,
                                           act_layout(M, K));
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(MQ_ERR_LAUNCH, "launch of quantize_act_kernel (grid %lld) failed: %s",
                (long long)M, cudaGetErrorName(e));
  }
  return MQ_OK;
}

}  // namespace mq
