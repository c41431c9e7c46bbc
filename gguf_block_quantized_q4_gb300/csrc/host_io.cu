// host_io.cu -- activations in and results out for the host-buffer calls.
//
// On a GPU that reaches its host's memory over a coherent link (Grace-Blackwell), page-locked
// host memory has a device view that kernels load from and store to directly.  The
// host-buffer calls use it in place of copy-engine transfers when both ends allow it: the
// decode activations are pulled into the caller's device buffer by the small kernel below
// (the matvec, launched with programmatic stream serialisation, starts streaming its weights
// while it runs and reads x only after its grid-dependency wait), the prefill quantiser reads
// its rows straight from the host, and the matvec / MMQ stores go straight to the host
// result buffer.  The data crossing the link is the same as with the copies: x in once, y out
// once.
#include "mq_common.cuh"

namespace mq {
namespace {

constexpr int kCopyThreads = 256;

// dst[i] = src[i] for n4 16-byte items.  The dependent launch that follows may start as soon
// as every CTA of this grid has begun: it waits for this grid's completion before reading dst.
__global__ void __launch_bounds__(kCopyThreads) copy_in_kernel(const float4 *__restrict__ src,
                                                               float4 *__restrict__ dst,
                                                               int64_t n4) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t i = int64_t(blockIdx.x) * kCopyThreads + threadIdx.x; i < n4;
       i += int64_t(gridDim.x) * kCopyThreads)
    dst[i] = src[i];
}

}  // namespace

const void *host_device_view(const void *p, size_t align) {
  if (!p || (reinterpret_cast<uintptr_t>(p) & (align - 1))) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  int dev = -1;
  cudaGetDevice(&dev);
  int canmap = 0;
  cudaDeviceGetAttribute(&canmap, cudaDevAttrCanMapHostMemory, dev);
  if (!canmap) return nullptr;
  const void *v = a.devicePointer;
  return (reinterpret_cast<uintptr_t>(v) & (align - 1)) ? nullptr : v;
}

mq_status launch_copy_in(const float *src_view, float *dst, int64_t n, cudaStream_t s,
                         int sms) {
  if (n <= 0) return MQ_OK;
  if (n % 4) return fail(MQ_ERR_ARG, "copy_in: %lld floats, not a multiple of 4", (long long)n);
  const int64_t n4 = n / 4;
  const int64_t want = (n4 + kCopyThreads - 1) / kCopyThreads;
  const unsigned grid = (unsigned)(want < 2 * int64_t(sms) ? want : 2 * int64_t(sms));
  copy_in_kernel<<<grid, kCopyThreads, 0, s>>>(reinterpret_cast<const float4 *>(src_view),
                                                reinterpret_cast<float4 *>(dst), n4);
  MQ_LAUNCH_CHECK("copy_in_kernel");
  return MQ_OK;
}

}  // namespace mq
