// xplane.cu -- the activation fragment plane of a Q4_K / Q5_K two-tile call (B = 5..8) of
// the persistent decode matvec ("minfer CUDA Backend Design" §4.4: the _multi matvec variants for nt 2..8).
// The call's x (B rows of K) is converted once into the tensor-core B fragments, instead of
// once in every CTA of the matvec (every one reads every chunk of x); the matvec then
// bulk-copies each chunk's fragments into its fragment slots.  The layout is in
// mv_device.cuh.
//
// Per batch row and 256-element chunk the arithmetic is that of the matvec's x warps, so the
// fragments are the same bits: a power-of-two scale 2^e that puts the chunk's max |x| in
// [2^14, 2^15), hi = f16(x 2^e) and lo = f16(x 2^e - hi), and from the sums of the scaled x
// over each 32-element sub-block (the same butterfly of warp shuffles), divided by 32, the
// Q4_K / Q5_K min-term fragment.  Rows past B are zeros.
#include "mv_device.cuh"

namespace mq {
namespace {

using namespace mvd;

// One CTA per chunk, one warp per batch row of the NT n8 tiles; lane handles the float4
// items lane and lane + 32 of the chunk.
template <int NT>
__global__ void __launch_bounds__(128 * NT) xplane_kernel(const float *__restrict__ x, int B,
                                                          int64_t K, uint8_t *__restrict__ plane) {
  __shared__ float xs[4 * NT][8];  // sub-block sums / 32 of each row
  // the matvec that reads the plane waits for this whole grid anyway: let it launch (and
  // start streaming its weights) at once
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
  const int c = blockIdx.x, lane = threadIdx.x & 31, b = threadIdx.x >> 5;
  const int cw = chunk_width(K, c);
  uint8_t *pc = plane + int64_t(c) * xp_chunk_bytes(NT);
  auto frag = reinterpret_cast<uint2(*)[NT][32 + xp_pad(NT)]>(pc);
  float *unscale = reinterpret_cast<float *>(pc + xp_off_unscale(NT));
  const bool live = b < B;
  float4 v[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int f = lane + 32 * k;
    v[k] = live && 4 * f < cw
               ? __ldg(reinterpret_cast<const float4 *>(x + int64_t(b) * K + int64_t(c) * kChunk) + f)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k)
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
  const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  const int E = (int)((mb >> 23) & 255);
  int e = mb == 0 ? 0 : 141 - max(E, 1);
  e = min(max(e, -100), 126);
  const float scale = __int_as_float((e + 127) << 23);
  if (lane == 0) unscale[b] = live ? __int_as_float((127 - e) << 23) : 0.f;
  if (lane == 0 && b + 4 * NT < 8) unscale[b + 4 * NT] = 0.f;  // the padding of NT = 1
  const int col = 2 * (b & 3);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int f = lane + 32 * k, g16 = f >> 2, t = f & 3;
    const float v0 = v[k].x * scale, v1 = v[k].y * scale, v2 = v[k].z * scale,
                v3 = v[k].w * scale;
    const uint32_t hi01 = pack_f16x2(v0, v1), hi23 = pack_f16x2(v2, v3);
    const uint32_t lo01 = pack_f16x2(v0 - f16_lo(hi01), v1 - f16_hi(hi01));
    const uint32_t lo23 = pack_f16x2(v2 - f16_lo(hi23), v3 - f16_hi(hi23));
    frag[g16][b >> 2][col * 4 + t] = make_uint2(hi01, hi23);
    frag[g16][b >> 2][(col + 1) * 4 + t] = make_uint2(lo01, lo23);
    // sum of sub-block f >> 3 (8 consecutive items) of the scaled x, scaled by 1/32 so that
    // |sum| < 2^15 fits f16
    float ps = (v0 + v1) + (v2 + v3);
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    ps += __shfl_xor_sync(0xffffffffu, ps, 4);
    if ((lane & 7) == 0) xs[b][f >> 3] = ps * 0.03125f;
  }
  __syncwarp();
  // min-term fragment: lane (col', t') of row b holds sums 2t', 2t'+1 (hi or lo part)
  if (lane < 8) {
    const int part = lane >> 2, t = lane & 3;
    const float s0 = xs[b][2 * t], s1 = xs[b][2 * t + 1];
    const uint32_t h = pack_f16x2(s0, s1);
    const uint32_t word = part == 0 ? h : pack_f16x2(s0 - f16_lo(h), s1 - f16_hi(h));
    frag[16][b >> 2][(col + part) * 4 + t] = make_uint2(word, 0u);
  }
}

}  // namespace

size_t xplane_bytes(int B, int64_t K) {
  return size_t((K + kChunk - 1) / kChunk) * xp_chunk_bytes(B > 4 ? 2 : 1);
}

mq_status launch_xplane(const float *x, int B, int64_t K, uint8_t *plane, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((K + kChunk - 1) / kChunk), 1, 1);
  cfg.blockDim = dim3(B > 4 ? 256 : 128, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const cudaError_t e = B > 4 ? cudaLaunchKernelEx(&cfg, xplane_kernel<2>, x, B, K, plane)
                              : cudaLaunchKernelEx(&cfg, xplane_kernel<1>, x, B, K, plane);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(MQ_ERR_LAUNCH, "launch of xplane_kernel (grid %u) failed: %s", cfg.gridDim.x,
                cudaGetErrorName(e));
  }
  return MQ_OK;
}

}  // namespace mq
