// mq_api.cu -- the C ABI entry points of libmq: argument validation, error
// reporting, per-device state, weight registration.  Compute happens in the
// kernels of repack.cu, matvec.cu, quantize.cu and mmq.cu.
//
// Error model ("minfer CUDA Backend Design" §4.9 rules 1, 4, 5; "GPU Safety"
// CUDA rules): every invariant violation returns an mq_status and a message
// naming the call, the invariant and the values; there is no fallback path.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "mq_common.cuh"

namespace mq {

static thread_local char g_msg[1024] = "no error";

mq_status fail(mq_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

mq_status cuda_fail(cudaError_t e, const char *call, const char *site) {
  return fail(e == cudaErrorMemoryAllocation ? MQ_ERR_OOM : MQ_ERR_CUDA, "%s: %s failed: %s (%s)",
              site, call, cudaGetErrorName(e), cudaGetErrorString(e));
}

static std::mutex g_dev_mu;
static std::vector<DeviceState *> g_devs;

DeviceState *device_state(int dev) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (dev < 0 || dev >= (int)g_devs.size()) return nullptr;
  DeviceState *st = g_devs[dev];
  return (st && st->ready) ? st : nullptr;
}

mq_status current_state(DeviceState **st, const char *site) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice", site);
  *st = device_state(dev);
  if (!*st) return fail(MQ_ERR_STATE, "%s: mq_init(%d) was not called for the current device",
                        site, dev);
  return MQ_OK;
}

}  // namespace mq

using namespace mq;

#define CK(call, site)                                              \
  do {                                                              \
    cudaError_t e_ = (call);                                        \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call, site);       \
  } while (0)

extern "C" const char *mq_last_error(void) { return g_msg; }

extern "C" const char *mq_status_name(mq_status s) {
  switch (s) {
    case MQ_OK: return "MQ_OK";
    case MQ_ERR_ARG: return "MQ_ERR_ARG";
    case MQ_ERR_TYPE: return "MQ_ERR_TYPE";
    case MQ_ERR_SHAPE: return "MQ_ERR_SHAPE";
    case MQ_ERR_PAYLOAD: return "MQ_ERR_PAYLOAD";
    case MQ_ERR_ALIGN: return "MQ_ERR_ALIGN";
    case MQ_ERR_CUDA: return "MQ_ERR_CUDA";
    case MQ_ERR_OOM: return "MQ_ERR_OOM";
    case MQ_ERR_LAUNCH: return "MQ_ERR_LAUNCH";
    case MQ_ERR_TIMEOUT: return "MQ_ERR_TIMEOUT";
    case MQ_ERR_STATE: return "MQ_ERR_STATE";
  }
  return "MQ_ERR_UNKNOWN";
}

// Failure-injection seams of the tests, read from the environment by mq_init (every call,
// including those that find the device ready), never on a hot-path call:
//   MQ_TEST_FAIL_LAUNCH=1  the matvec and MMQ launches are configured with an empty grid,
//                          which the runtime refuses before any kernel runs;
//   MQ_TEST_EXPIRE_WAIT=1  the MMQ epilogue first waits on a barrier nothing arrives on;
//                          the wait expires after about a millisecond, records
//                          MQ_ERR_TIMEOUT in the status word and the kernel carries on;
//   MQ_TEST_NO_XPLANE=1    the persistent matvec's two-tile calls take no activation
//                          fragment plane (as when the pool cannot give one): its x warps
//                          convert x themselves.
static std::atomic<int> g_test_fail_launch{0}, g_test_expire_wait{0}, g_test_no_xplane{0};

static int env_flag(const char *name) {
  const char *v = getenv(name);
  return (v && v[0] == '1') ? 1 : 0;
}

int mq::test_fail_launch() { return g_test_fail_launch.load(std::memory_order_relaxed); }
int mq::test_no_xplane() { return g_test_no_xplane.load(std::memory_order_relaxed); }
static int test_expire_wait() { return g_test_expire_wait.load(std::memory_order_relaxed); }

static mq_status static_scratch(DeviceState *st, uint8_t **out, const char *site);

extern "C" mq_status mq_init(int device) {
  const char *site = "mq_init";
  g_test_fail_launch.store(env_flag("MQ_TEST_FAIL_LAUNCH"), std::memory_order_relaxed);
  g_test_expire_wait.store(env_flag("MQ_TEST_EXPIRE_WAIT"), std::memory_order_relaxed);
  g_test_no_xplane.store(env_flag("MQ_TEST_NO_XPLANE"), std::memory_order_relaxed);
  int ndev = 0;
  CK(cudaGetDeviceCount(&ndev), site);
  if (device < 0 || device >= ndev)
    return fail(MQ_ERR_ARG, "mq_init: device %d out of range [0, %d)", device, ndev);
  CK(cudaSetDevice(device), site);
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if ((int)g_devs.size() < ndev) g_devs.resize(ndev, nullptr);
    if (g_devs[device] && g_devs[device]->ready) return MQ_OK;
  }
  DeviceState *st = new DeviceState();
  cudaDeviceProp pr;
  CK(cudaGetDeviceProperties(&pr, device), site);
  if (pr.major < 10)
    return fail(MQ_ERR_ARG, "mq_init: device %d is sm_%d%d; libmq is built for sm_103a", device,
                pr.major, pr.minor);
  st->sms = pr.multiProcessorCount;
  CK(cudaDeviceGetAttribute(&st->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device),
     site);
  CK(cudaMalloc(&st->status, 64), site);
  CK(cudaMemset(st->status, 0, 64), site);
  CK(cudaStreamCreateWithFlags(&st->reg_stream, cudaStreamNonBlocking), site);
  CK(cudaStreamCreateWithFlags(&st->copy_stream, cudaStreamNonBlocking), site);
  CK(cudaEventCreateWithFlags(&st->ev_rows, cudaEventDisableTiming), site);
  CK(cudaEventCreateWithFlags(&st->ev_copied, cudaEventDisableTiming), site);
  {
    // the activation fragment planes of the persistent matvec's two-tile calls: a
    // stream-ordered pool of this device that keeps up to 64 MB reserved between calls (a
    // plane takes 36 bytes per element of K); without it the x warps convert x themselves
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    if (cudaMemPoolCreate(&st->xpool, &props) == cudaSuccess) {
      uint64_t keep = 64ull << 20;
      (void)cudaMemPoolSetAttribute(st->xpool, cudaMemPoolAttrReleaseThreshold, &keep);
    } else {
      (void)cudaGetLastError();
      st->xpool = nullptr;
    }
  }
  mq_status s = init_kernels(st);
  if (s == MQ_OK) s = init_matvec(st);
  // the static scratch of mq_mmq_fused_static: looking its address up here loads this file's
  // device code (and with it the array) now, outside any stream capture of the caller
  uint8_t *scratch = nullptr;
  if (s == MQ_OK) s = static_scratch(st, &scratch, site);
  if (s != MQ_OK) return s;
  CK(cudaDeviceSynchronize(), site);
  st->ready = true;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_devs[device] && g_devs[device]->ready) {
    // another thread finished first; keep its state
    cudaFree(st->status);
    cudaStreamDestroy(st->reg_stream);
    cudaStreamDestroy(st->copy_stream);
    cudaEventDestroy(st->ev_rows);
    cudaEventDestroy(st->ev_copied);
    if (st->xpool) cudaMemPoolDestroy(st->xpool);
    delete st;
  } else {
    g_devs[device] = st;
  }
  return MQ_OK;
}

static mq_status check_type_shape(const char *site, int type, int64_t N, int64_t K) {
  if (type != MQ_Q4_0 && type != MQ_Q4_1 && type != MQ_Q5_0 && type != MQ_Q5_1 &&
      type != MQ_Q8_0 && type != MQ_Q4_K && type != MQ_Q5_K && type != MQ_Q6_K &&
      !float_type(type))
    return fail(MQ_ERR_TYPE,
                "%s: unsupported GGUF type %d (supported: 1 F16, 2 Q4_0, 3 Q4_1, 6 Q5_0, "
                "7 Q5_1, 8 Q8_0, 12 Q4_K, 13 Q5_K, 14 Q6_K, 30 BF16)",
                site, type);
  if (N < 1 || K < 1)
    return fail(MQ_ERR_SHAPE, "%s: N=%lld K=%lld must both be >= 1", site, (long long)N,
                (long long)K);
  int be = block_elems(type);
  if (K % be)
    return fail(MQ_ERR_SHAPE, "%s: K=%lld is not a multiple of the type-%d block size %d", site,
                (long long)K, type, be);
  if (N > (int64_t(1) << 31) || K > (int64_t(1) << 24))
    return fail(MQ_ERR_SHAPE, "%s: N=%lld K=%lld beyond the supported range (N <= 2^31, K <= 2^24)",
                site, (long long)N, (long long)K);
  return MQ_OK;
}

static mq_status free_planes(mq_weight *w) {
  void *ps[] = {w->q, w->d, w->qh, w->dm, w->mw, w->mw2, w->td, w->tm, w->mb, w->vcol};
  for (void *p : ps)
    if (p) cudaFree(p);
  w->q = nullptr; w->d = nullptr; w->qh = nullptr; w->dm = nullptr; w->mw = nullptr;
  w->mw2 = nullptr; w->td = nullptr; w->tm = nullptr; w->mb = nullptr; w->vcol = nullptr;
  return MQ_OK;
}

template <class T>
static mq_status alloc_plane(T **p, size_t bytes, size_t *total, const char *what) {
  cudaError_t e = cudaMalloc((void **)p, bytes);
  if (e != cudaSuccess)
    return fail(e == cudaErrorMemoryAllocation ? MQ_ERR_OOM : MQ_ERR_CUDA,
                "mq_register_weight: cudaMalloc(%zu) for the %s plane failed: %s", bytes, what,
                cudaGetErrorName(e));
  *total += bytes;
  return MQ_OK;
}

static mq_status register_impl(const char *site, mq_type type, const void *host_bytes,
                               size_t nbytes, int64_t N, int64_t K, uint32_t flags, int ffn_gu,
                               mq_weight **out) {
  if (!out) return fail(MQ_ERR_ARG, "%s: out is NULL", site);
  *out = nullptr;
  mq_status s = check_type_shape(site, type, N, K);
  if (s != MQ_OK) return s;
  const uint32_t known = MQ_REG_NO_MMQ_PLANE | MQ_REG_MMQ_FROM_DECODE_PLANE;
  if (flags & ~known)
    return fail(MQ_ERR_ARG, "%s: unknown flag bits 0x%x", site, flags & ~known);
  if ((flags & MQ_REG_MMQ_FROM_DECODE_PLANE) && type != MQ_Q4_K)
    return fail(MQ_ERR_ARG, "%s: MQ_REG_MMQ_FROM_DECODE_PLANE is for Q4_K weights (type %d)",
                site, type);
  size_t expect = size_t(N) * size_t(K / block_elems(type)) * size_t(block_bytes(type));
  if (nbytes != expect)
    return fail(MQ_ERR_PAYLOAD,
                "%s: payload is %zu bytes but a type-%d %lld x %lld tensor is exactly %zu bytes "
                "(N * K/%d * %d)",
                site, nbytes, type, (long long)N, (long long)K, expect, block_elems(type),
                block_bytes(type));
  if (!host_bytes) return fail(MQ_ERR_ARG, "%s: host_bytes is NULL", site);
  DeviceState *st = nullptr;
  if ((s = current_state(&st, site)) != MQ_OK) return s;

  mq_weight *w = new mq_weight();
  w->type = type;
  w->ffn_gu = ffn_gu;
  w->N = N;
  w->K = K;
  w->np = round_up(N, 128);
  CK(cudaGetDevice(&w->device), site);
  w->payload = nbytes;
  size_t total = 0;
  const int64_t nsb = K / 256;
  auto cleanup = [&](mq_status r) {
    free_planes(w);
    delete w;
    return r;
  };
  // decode planes: padded to whole row groups, padding rows zero
  w->ngroup = (N + kRowGroup - 1) / kRowGroup;
  w->nchunk = (int)((K + kChunk - 1) / kChunk);
  const size_t npad = size_t(w->ngroup) * kRowGroup;
  auto zalloc = [&](auto **pp, size_t bytes, const char *what) {
    mq_status r = alloc_plane(pp, bytes, &total, what);
    if (r == MQ_OK) cudaMemsetAsync(*pp, 0, bytes, st->reg_stream);
    return r;
  };
  if (float_type(type)) {
    if ((s = zalloc(&w->q, npad * K * 2, "f16/bf16 weights")) != MQ_OK) return cleanup(s);
  } else if (type == MQ_Q8_0) {
    if ((s = zalloc(&w->q, npad * K, "q8_0 qs")) != MQ_OK) return cleanup(s);
    if ((s = zalloc(&w->d, npad * w->nchunk * 8 * 2, "q8_0 d")) != MQ_OK) return cleanup(s);
  } else if (block_elems(type) == 32) {  // Q4_0, Q4_1, Q5_0, Q5_1
    if ((s = zalloc(&w->q, npad * K / 2, "4-bit quants")) != MQ_OK) return cleanup(s);
    if ((s = zalloc(&w->d, npad * w->nchunk * 8 * 2, "block d")) != MQ_OK) return cleanup(s);
    if ((type == MQ_Q4_1 || type == MQ_Q5_1) &&
        (s = zalloc(&w->dm, npad * w->nchunk * 8 * 2, "block m")) != MQ_OK)
      return cleanup(s);
    if ((type == MQ_Q5_0 || type == MQ_Q5_1) &&
        (s = zalloc(&w->qh, npad * (K / 32) * 4, "fifth bits")) != MQ_OK)
      return cleanup(s);
  } else if (type == MQ_Q4_K) {
    if ((s = zalloc(&w->q, npad * nsb * 144, "q4_K")) != MQ_OK) return cleanup(s);
  } else if (type == MQ_Q5_K) {
    if ((s = zalloc(&w->q, npad * nsb * 176, "q5_K")) != MQ_OK) return cleanup(s);
  } else {
    if ((s = zalloc(&w->q, npad * nsb * 210, "q6_K")) != MQ_OK) return cleanup(s);
  }
  // f16 / bf16 weights have no integer form and no prefill planes
  const bool mmq = !(flags & MQ_REG_NO_MMQ_PLANE) && !float_type(type);
  if (mmq) {
    // with MQ_REG_MMQ_FROM_DECODE_PLANE the Q4_K MMQ expands the decode-plane tiles in
    // shared memory instead of reading an f16 integer plane
    if (!(flags & MQ_REG_MMQ_FROM_DECODE_PLANE) &&
        (s = alloc_plane(&w->mw, size_t(N) * K * 2, &total, "prefill operand")) != MQ_OK)
      return cleanup(s);
    if (type == MQ_Q6_K &&
        (s = alloc_plane(&w->mw2, size_t(N) * K * 2, &total, "prefill odd part")) != MQ_OK)
      return cleanup(s);
    if ((s = alloc_plane(&w->td, size_t(w->np) * (K / 32) * 4, &total, "prefill d")) != MQ_OK)
      return cleanup(s);
    const bool mins =
        type == MQ_Q4_K || type == MQ_Q5_K || type == MQ_Q4_1 || type == MQ_Q5_1;
    if (mins &&
        (s = alloc_plane(&w->tm, size_t(w->np) * (K / 32) * 4, &total, "prefill min")) != MQ_OK)
      return cleanup(s);
    // the padding columns of the transposed planes must read as zero
    cudaMemsetAsync(w->td, 0, size_t(w->np) * (K / 32) * 4, st->reg_stream);
    if (w->tm) cudaMemsetAsync(w->tm, 0, size_t(w->np) * (K / 32) * 4, st->reg_stream);
    if (mins) {
      if ((s = zalloc(&w->mb, size_t(w->np) * min_ld(K / 32) * 2, "prefill min operand")) != MQ_OK)
        return cleanup(s);
      if ((s = zalloc(&w->vcol, size_t(w->np) * 4, "prefill min scale")) != MQ_OK)
        return cleanup(s);
    }
  }
  w->device_bytes = total;

  // Upload the GGUF bytes to a staging buffer, repack on the device.
  uint8_t *raw = nullptr;
  cudaError_t e = cudaMalloc(&raw, nbytes);
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(staging)", site));
  e = cudaMemcpyAsync(raw, host_bytes, nbytes, cudaMemcpyHostToDevice, st->reg_stream);
  if (e == cudaSuccess) {
    s = repack_weight(w, raw, mmq, st->reg_stream);
    e = cudaStreamSynchronize(st->reg_stream);
  }
  cudaFree(raw);
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "upload/repack", site));
  if (s != MQ_OK) return cleanup(s);
  if (mmq && (s = encode_weight_maps(w)) != MQ_OK) return cleanup(s);
  *out = w;
  return MQ_OK;
}

extern "C" mq_status mq_register_weight(mq_type type, const void *host_bytes, size_t nbytes,
                                        int64_t N, int64_t K, uint32_t flags, mq_weight **out) {
  return register_impl("mq_register_weight", type, host_bytes, nbytes, N, K, flags, 0, out);
}

// Rows of a fused gate/up weight, in units of 16: 8 gate rows, then the same 8 rows of
// the up weight (a kernel thread then holds a gate result and its up result).
extern "C" mq_status mq_register_ffn_gu(mq_type type, const void *gate_bytes,
                                        const void *up_bytes, size_t nbytes_each, int64_t N,
                                        int64_t K, uint32_t flags, mq_weight **out) {
  const char *site = "mq_register_ffn_gu";
  if (!out) return fail(MQ_ERR_ARG, "%s: out is NULL", site);
  *out = nullptr;
  mq_status s = check_type_shape(site, type, 2 * N, K);
  if (s != MQ_OK) return s;
  if (N % 8)
    return fail(MQ_ERR_SHAPE, "%s: N=%lld gate rows must be a multiple of 8", site, (long long)N);
  const size_t row = size_t(K / block_elems(type)) * size_t(block_bytes(type));
  if (nbytes_each != size_t(N) * row)
    return fail(MQ_ERR_PAYLOAD,
                "%s: nbytes_each is %zu but a type-%d %lld x %lld tensor is exactly %zu bytes",
                site, nbytes_each, type, (long long)N, (long long)K, size_t(N) * row);
  if (!gate_bytes || !up_bytes) return fail(MQ_ERR_ARG, "%s: gate_bytes or up_bytes is NULL", site);
  std::vector<uint8_t> fused(2 * nbytes_each);
  const uint8_t *g = static_cast<const uint8_t *>(gate_bytes);
  const uint8_t *u = static_cast<const uint8_t *>(up_bytes);
  for (int64_t k = 0; k < N / 8; ++k) {
    memcpy(fused.data() + size_t(16 * k) * row, g + size_t(8 * k) * row, 8 * row);
    memcpy(fused.data() + size_t(16 * k + 8) * row, u + size_t(8 * k) * row, 8 * row);
  }
  return register_impl(site, type, fused.data(), fused.size(), 2 * N, K, flags, 1, out);
}

extern "C" mq_status mq_weight_free(mq_weight *w) {
  if (!w) return MQ_OK;
  int cur = 0;
  const int dev = w->device;
  cudaGetDevice(&cur);
  if (cur != dev) cudaSetDevice(dev);
  cudaError_t e = cudaDeviceSynchronize();
  free_planes(w);
  delete w;
  if (cur != dev) cudaSetDevice(cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize", "mq_weight_free");
  return MQ_OK;
}

extern "C" mq_status mq_weight_info(const mq_weight *w, int *type, int64_t *N, int64_t *K,
                                    size_t *device_bytes) {
  if (!w) return fail(MQ_ERR_ARG, "mq_weight_info: w is NULL");
  if (type) *type = w->type;
  if (N) *N = w->N;
  if (K) *K = w->K;
  if (device_bytes) *device_bytes = w->device_bytes;
  return MQ_OK;
}

extern "C" mq_status mq_weight_unpack(const mq_weight *w, void *host_bytes, size_t nbytes) {
  const char *site = "mq_weight_unpack";
  if (!w) return fail(MQ_ERR_ARG, "%s: w is NULL", site);
  if (!host_bytes) return fail(MQ_ERR_ARG, "%s: host_bytes is NULL", site);
  if (nbytes != w->payload)
    return fail(MQ_ERR_PAYLOAD, "%s: nbytes=%zu but the weight's payload is %zu bytes", site,
                nbytes, w->payload);
  DeviceState *st = nullptr;
  mq_status s;
  if ((s = current_state(&st, site)) != MQ_OK) return s;
  uint8_t *raw = nullptr;
  CK(cudaMalloc(&raw, nbytes), site);
  s = unpack_weight(w, raw, st->reg_stream);
  cudaError_t e = cudaSuccess;
  if (s == MQ_OK) e = cudaMemcpyAsync(host_bytes, raw, nbytes, cudaMemcpyDeviceToHost, st->reg_stream);
  cudaError_t e2 = cudaStreamSynchronize(st->reg_stream);
  cudaFree(raw);
  if (s != MQ_OK) return s;
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync", site);
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamSynchronize", site);
  if (w->ffn_gu) {  // back from the interleaved row order to gate rows, then up rows
    const size_t row = nbytes / size_t(w->N), half = nbytes / 2;
    std::vector<uint8_t> tmp(static_cast<uint8_t *>(host_bytes),
                             static_cast<uint8_t *>(host_bytes) + nbytes);
    uint8_t *dst = static_cast<uint8_t *>(host_bytes);
    for (int64_t k = 0; k < w->N / 16; ++k) {
      memcpy(dst + size_t(8 * k) * row, tmp.data() + size_t(16 * k) * row, 8 * row);
      memcpy(dst + half + size_t(8 * k) * row, tmp.data() + size_t(16 * k + 8) * row, 8 * row);
    }
  }
  return MQ_OK;
}

// A pointer the device can read/write as global memory.
static mq_status check_dev_ptr(const char *site, const char *name, const void *p, int dev,
                               size_t align) {
  if (!p) return fail(MQ_ERR_ARG, "%s: %s is NULL", site, name);
  if (reinterpret_cast<uintptr_t>(p) % align)
    return fail(MQ_ERR_ALIGN, "%s: %s=%p is not %zu-byte aligned", site, name, p, align);
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MQ_ERR_ARG, "%s: %s=%p is not a CUDA pointer (%s)", site, name, p,
                cudaGetErrorName(e));
  }
  if (a.type == cudaMemoryTypeDevice && a.device != dev)
    return fail(MQ_ERR_ARG, "%s: %s=%p lives on device %d, the weight on device %d", site, name,
                p, a.device, dev);
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return fail(MQ_ERR_ARG, "%s: %s=%p is host memory (type %d); a device pointer is required",
                site, name, p, (int)a.type);
  return MQ_OK;
}

static mq_status check_weight(const char *site, int type, const mq_weight *W, int64_t N,
                              int64_t K, int ffn_gu = 0) {
  if (!W) return fail(MQ_ERR_ARG, "%s: W is NULL", site);
  if (W->ffn_gu != ffn_gu)
    return fail(MQ_ERR_ARG,
                ffn_gu ? "%s: the weight is not a fused gate/up weight (mq_register_ffn_gu)"
                       : "%s: the weight is a fused gate/up weight; use mq_ffn_gu_matvec or "
                         "mq_ffn_gu_mmq",
                site);
  if (ffn_gu) N *= 2;  // the fused weight holds the gate and the up rows
  mq_status s = check_type_shape(site, type, N, K);
  if (s != MQ_OK) return s;
  if (W->type != type)
    return fail(MQ_ERR_TYPE, "%s: type %d but the weight was registered as type %d", site, type,
                W->type);
  if (W->N != N || W->K != K)
    return fail(MQ_ERR_SHAPE, "%s: N=%lld K=%lld but the weight is %lld x %lld", site,
                (long long)N, (long long)K, (long long)W->N, (long long)W->K);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != W->device)
    return fail(MQ_ERR_ARG, "%s: current device %d but the weight lives on device %d", site, dev,
                W->device);
  return MQ_OK;
}

static mq_status matvec_impl(const char *site, int ffn_gu, mq_type type, const mq_weight *W,
                             const float *x, float *y, int64_t N, int64_t K, int B,
                             mq_stream stream) {
  mq_status s = check_weight(site, type, W, N, K, ffn_gu);
  if (s != MQ_OK) return s;
  if (B < 1 || B > kMaxB)
    return fail(MQ_ERR_ARG, "%s: B=%d outside [1, %d]", site, B, kMaxB);
  DeviceState *st = nullptr;
  if ((s = current_state(&st, site)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "x", x, W->device, 16)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "y", y, W->device, 16)) != MQ_OK) return s;
  return launch_matvec(W, x, y, B, (cudaStream_t)stream, st);
}

extern "C" mq_status mq_matvec(mq_type type, const mq_weight *W, const float *x, float *y,
                               int64_t N, int64_t K, int B, mq_stream stream) {
  return matvec_impl("mq_matvec", 0, type, W, x, y, N, K, B, stream);
}

extern "C" mq_status mq_ffn_gu_matvec(mq_type type, const mq_weight *W, const float *x, float *h,
                                      int64_t N, int64_t K, int B, mq_stream stream) {
  return matvec_impl("mq_ffn_gu_matvec", 1, type, W, x, h, N, K, B, stream);
}

// Host buffers of the host-buffer calls: any non-null pointer CUDA does not report as device
// memory (pinned memory keeps the copies asynchronous; pageable memory works, but its
// copies then wait for the host).
static mq_status check_host_ptr(const char *site, const char *name, const void *p) {
  if (!p) return fail(MQ_ERR_ARG, "%s: %s is NULL", site, name);
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MQ_ERR_ARG, "%s: %s=%p: cudaPointerGetAttributes failed (%s)", site, name, p,
                cudaGetErrorName(e));
  }
  if (a.type == cudaMemoryTypeDevice)
    return fail(MQ_ERR_ARG, "%s: %s=%p is device memory; a host buffer is required", site, name,
                p);
  return MQ_OK;
}

extern "C" mq_status mq_matvec_host(mq_type type, const mq_weight *W, const float *x_host,
                                    float *y_host, float *x_dev, float *y_dev, int64_t N,
                                    int64_t K, int B, mq_stream stream) {
  const char *site = "mq_matvec_host";
  mq_status s = check_weight(site, type, W, N, K);
  if (s != MQ_OK) return s;
  if (B < 1 || B > kMaxB) return fail(MQ_ERR_ARG, "%s: B=%d outside [1, %d]", site, B, kMaxB);
  DeviceState *st = nullptr;
  if ((s = current_state(&st, site)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "x_dev", x_dev, W->device, 16)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "y_dev", y_dev, W->device, 16)) != MQ_OK) return s;
  if ((s = check_host_ptr(site, "x_host", x_host)) != MQ_OK) return s;
  if ((s = check_host_ptr(site, "y_host", y_host)) != MQ_OK) return s;
  cudaStream_t cs = (cudaStream_t)stream;
  // page-locked host buffers are read and written by the kernels through their device
  // views; other host memory goes through copies into and out of x_dev / y_dev
  if (const void *xv = host_device_view(x_host, 16)) {
    if ((s = launch_copy_in(static_cast<const float *>(xv), x_dev, int64_t(B) * K, cs,
                            st->sms)) != MQ_OK)
      return s;
  } else {
    CK(cudaMemcpyAsync(x_dev, x_host, size_t(B) * K * 4, cudaMemcpyHostToDevice, cs), site);
  }
  float *yv = static_cast<float *>(const_cast<void *>(host_device_view(y_host, 16)));
  if ((s = launch_matvec(W, x_dev, yv ? yv : y_dev, B, cs, st)) != MQ_OK) return s;
  if (!yv)
    CK(cudaMemcpyAsync(y_host, y_dev, size_t(B) * N * 4, cudaMemcpyDeviceToHost, cs), site);
  return MQ_OK;
}

extern "C" size_t mq_act_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 32 || K % 32) return 0;
  return act_layout(M, K).total;
}

extern "C" mq_status mq_quantize_act(const float *x, void *xq, int64_t M, int64_t K,
                                     mq_stream stream) {
  const char *site = "mq_quantize_act";
  if (M < 1) return fail(MQ_ERR_ARG, "%s: M=%lld must be >= 1", site, (long long)M);
  if (K < 32 || K % 32)
    return fail(MQ_ERR_SHAPE, "%s: K=%lld must be a positive multiple of 32", site, (long long)K);
  if (M > (int64_t(1) << 31) || K > (int64_t(1) << 24))
    return fail(MQ_ERR_SHAPE, "%s: M=%lld K=%lld beyond the supported range", site, (long long)M,
                (long long)K);
  DeviceState *st = nullptr;
  mq_status s;
  if ((s = current_state(&st, site)) != MQ_OK) return s;
  int dev = 0;
  cudaGetDevice(&dev);
  if ((s = check_dev_ptr(site, "x", x, dev, 16)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "xq", xq, dev, 256)) != MQ_OK) return s;
  return launch_quantize(x, xq, M, K, (cudaStream_t)stream);
}

static mq_status mmq_common(const char *site, mq_type type, const mq_weight *W, const void *xq,
                            const void *out, int64_t M, int64_t N, int64_t K, DeviceState **st,
                            int ffn_gu = 0) {
  mq_status s = check_weight(site, type, W, N, K, ffn_gu);
  if (s != MQ_OK) return s;
  if (float_type(type))
    return fail(MQ_ERR_TYPE, "%s: type %d is an unquantised (f16/bf16) weight: it has no "
                "integer MMQ form; use the matvec", site, type);
  if (!W->td)
    return fail(MQ_ERR_ARG, "%s: the weight was registered with MQ_REG_NO_MMQ_PLANE", site);
  if (M < 1 || M > (int64_t(1) << 31))
    return fail(MQ_ERR_ARG, "%s: M=%lld outside [1, 2^31]", site, (long long)M);
  if ((s = current_state(st, site)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "xq", xq, W->device, 256)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "out", out, W->device, 16)) != MQ_OK) return s;
  return MQ_OK;
}

extern "C" mq_status mq_mmq(mq_type type, const mq_weight *W, const void *xq, float *y, int64_t M,
                            int64_t N, int64_t K, mq_stream stream) {
  DeviceState *st = nullptr;
  mq_status s = mmq_common("mq_mmq", type, W, xq, y, M, N, K, &st);
  if (s != MQ_OK) return s;
  return launch_mmq(W, xq, y, nullptr, M, (cudaStream_t)stream, st, test_expire_wait());
}

extern "C" mq_status mq_mmq_fused(mq_type type, const mq_weight *W, const float *x, void *xq,
                                  float *y, int64_t M, int64_t N, int64_t K, mq_stream stream) {
  DeviceState *st = nullptr;
  mq_status s = mmq_common("mq_mmq_fused", type, W, xq, y, M, N, K, &st);
  if (s != MQ_OK) return s;
  if ((s = check_dev_ptr("mq_mmq_fused", "x", x, W->device, 16)) != MQ_OK) return s;
  return launch_mmq(W, xq, y, nullptr, M, (cudaStream_t)stream, st, test_expire_wait(), x);
}

// Scratch of mq_mmq_fused_static: one file-scope device array per device (zero at module
// load), its first 256 bytes the grid barrier's words (at a fixed place, so that calls of
// different shapes find the count at zero), the rest an xq buffer.  Its address is looked
// up once per device, by mq_init; nothing is allocated.
static __device__ __align__(256) uint8_t g_static_xq[MQ_STATIC_XQ_BYTES];
static std::mutex g_static_mu;
static std::mutex g_host_mu;  // mq_mmq_host's enqueue sequence (shared events)

static mq_status static_scratch(DeviceState *st, uint8_t **out, const char *site) {
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!st->static_xq) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_xq);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)", site);
    st->static_xq = static_cast<uint8_t *>(p);
  }
  *out = st->static_xq;
  return MQ_OK;
}

extern "C" mq_status mq_mmq_fused_static(mq_type type, const mq_weight *W, const float *x,
                                         float *y, int64_t M, int64_t N, int64_t K,
                                         mq_stream stream) {
  const char *site = "mq_mmq_fused_static";
  DeviceState *st = nullptr;
  mq_status s;
  if ((s = current_state(&st, site)) != MQ_OK) return s;
  if (!W) return fail(MQ_ERR_ARG, "%s: W is NULL", site);
  int dev = -1;
  CK(cudaGetDevice(&dev), site);
  if (dev != W->device)
    return fail(MQ_ERR_ARG, "%s: the weight lives on device %d, the current device is %d", site,
                W->device, dev);
  if (M >= 1 && K >= 32 && K % 32 == 0 && M <= (int64_t(1) << 31)) {
    const size_t need = act_layout(M, K).total, room = MQ_STATIC_XQ_BYTES - 256;
    if (need > room)
      return fail(MQ_ERR_SHAPE,
                  "%s: M=%lld K=%lld needs %zu bytes of scratch; the static scratch holds %zu",
                  site, (long long)M, (long long)K, need, room);
  }
  uint8_t *base = nullptr;
  if ((s = static_scratch(st, &base, site)) != MQ_OK) return s;
  if ((s = mmq_common(site, type, W, base + 256, y, M, N, K, &st)) != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "x", x, W->device, 16)) != MQ_OK) return s;
  return launch_mmq(W, base + 256, y, nullptr, M, (cudaStream_t)stream, st, test_expire_wait(), x,
                    reinterpret_cast<unsigned *>(base));
}

extern "C" mq_status mq_mmq_host(mq_type type, const mq_weight *W, const float *x_host,
                                 float *y_host, float *x_dev, void *xq_dev, float *y_dev,
                                 int64_t M, int64_t N, int64_t K, mq_stream stream) {
  const char *site = "mq_mmq_host";
  DeviceState *st = nullptr;
  mq_status s = mmq_common(site, type, W, xq_dev, y_dev, M, N, K, &st);
  if (s != MQ_OK) return s;
  if ((s = check_dev_ptr(site, "x_dev", x_dev, W->device, 16)) != MQ_OK) return s;
  if ((s = check_host_ptr(site, "x_host", x_host)) != MQ_OK) return s;
  if ((s = check_host_ptr(site, "y_host", y_host)) != MQ_OK) return s;
  cudaStream_t cs = (cudaStream_t)stream;
  // a page-locked x_host is read by the quantiser through its device view, other host
  // memory is copied into x_dev.  y always goes out through y_dev and a copy: the MMQ's
  // stores (one row's 32-column piece per thread) would cross the host link as 16-byte
  // writes, about a fifth of the copy engine's rate.
  const float *xv = static_cast<const float *>(host_device_view(x_host, 16));
  if (!xv)
    CK(cudaMemcpyAsync(x_dev, x_host, size_t(M) * K * 4, cudaMemcpyHostToDevice, cs), site);
  if ((s = launch_quantize(xv ? xv : x_dev, xq_dev, M, K, cs)) != MQ_OK) return s;
  // The MMQ in chunks of M-tiles (128 rows) on the caller's stream; each chunk's rows of y
  // go back to the host on the library's copy stream while the next chunk runs (the host
  // link, not the MMQ, bounds the call: Q4_K 512 x 18944 x 3584, 361 -> 305 us).  The copy
  // stream rejoins the caller's stream at the end, so the call stays asynchronous and
  // ordered on `stream`.  One enqueue sequence at a time per device (the two events are
  // shared).  Quantising per chunk as well measured slower (316 us): its reads of x then
  // share the host link with the copies of y.
  const int64_t mts = (M + 127) / 128;
  const int64_t chunks = mts < 4 ? mts : 4, per = (mts + chunks - 1) / chunks;
  std::lock_guard<std::mutex> lk(g_host_mu);
  for (int64_t c0 = 0; c0 < mts; c0 += per) {
    const int64_t cn = mts - c0 < per ? mts - c0 : per;
    const int64_t r0 = c0 * 128, r1 = (c0 + cn) * 128 < M ? (c0 + cn) * 128 : M;
    if ((s = launch_mmq(W, xq_dev, y_dev, nullptr, M, cs, st, test_expire_wait(), nullptr,
                        nullptr, c0, cn)) != MQ_OK)
      return s;
    CK(cudaEventRecord(st->ev_rows, cs), site);
    CK(cudaStreamWaitEvent(st->copy_stream, st->ev_rows, 0), site);
    CK(cudaMemcpyAsync(y_host + r0 * N, y_dev + r0 * N, size_t(r1 - r0) * N * 4,
                       cudaMemcpyDeviceToHost, st->copy_stream),
       site);
  }
  CK(cudaEventRecord(st->ev_copied, st->copy_stream), site);
  CK(cudaStreamWaitEvent(cs, st->ev_copied, 0), site);
  return MQ_OK;
}

extern "C" mq_status mq_ffn_gu_mmq(mq_type type, const mq_weight *W, const void *xq, float *h,
                                   int64_t M, int64_t N, int64_t K, mq_stream stream) {
  DeviceState *st = nullptr;
  mq_status s = mmq_common("mq_ffn_gu_mmq", type, W, xq, h, M, N, K, &st, 1);
  if (s != MQ_OK) return s;
  return launch_mmq(W, xq, h, nullptr, M, (cudaStream_t)stream, st, test_expire_wait());
}

extern "C" mq_status mq_mmq_blockdots(mq_type type, const mq_weight *W, const void *xq,
                                      int32_t *D, int64_t M, int64_t N, int64_t K,
                                      mq_stream stream) {
  DeviceState *st = nullptr;
  mq_status s = mmq_common("mq_mmq_blockdots", type, W, xq, D, M, N, K, &st);
  if (s != MQ_OK) return s;
  return launch_mmq(W, xq, nullptr, D, M, (cudaStream_t)stream, st, test_expire_wait());
}

extern "C" mq_status mq_stream_status(mq_stream stream) {
  const char *site = "mq_stream_status";
  DeviceState *st = nullptr;
  mq_status s;
  if ((s = current_state(&st, site)) != MQ_OK) return s;
  CK(cudaStreamSynchronize((cudaStream_t)stream), site);
  int h[2] = {0, 0};
  CK(cudaMemcpy(h, st->status, sizeof(h), cudaMemcpyDeviceToHost), site);
  if (h[0] != 0) {
    CK(cudaMemset(st->status, 0, 64), site);
    return fail(MQ_ERR_TIMEOUT, "%s: a bounded device-side wait expired (code %d, kernel id %d)",
                site, h[0], h[1]);
  }
  return MQ_OK;
}
