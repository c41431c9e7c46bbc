// mq_common.cuh -- internal declarations shared by the libmq translation units.
//
// Device planes of a registered weight ("minfer CUDA Backend Design" §2.3:
// weights are uploaded once and repacked per quant type; §4.7: the planes trade
// device memory for speed).  All planes are lossless regroupings of the GGUF
// bytes except the prefill operand planes, which hold exact integer values.
//
// Decode planes (read by the matvec).  Rows are grouped by 128 (N padded with
// zero rows to a multiple of 128) and K is cut into 256-element chunks; the tile
// of one (row group g, chunk c) is contiguous, so one bulk copy moves it into
// shared memory.  Inside a row, each fragment thread's words are contiguous and
// 16-byte aligned (t = fragment thread 0..3, r = row in the group):
//   Q4_K  q   tile (g,c) at ((g*nchunk + c)*128 + r)*144: bytes 0..15 the GGUF
//             header (d, dmin, 12 scale bytes); word 2c'+u of thread t (bytes
//             16 + 32t + 4(2c'+u) + i) holds qs bytes 32c' + 16u + 4t + {0,2,1,3}[i],
//             so that masking nibbles 0-3 / 4-7 of bytes 0 and 2 (then, after a
//             shift by 8, of bytes 1 and 3) yields the element pairs of one
//             fragment register
//   Q6_K  q   tile (g,c) at (g*nchunk + c)*128*210, three parts:
//             quants at r*192: byte 48t + 4(3(2h+v) + w) + i  <-  word w of (h, v):
//               w=0 ql[64h + 16v + 4t + i], w=1 ql[64h + 32 + 16v + 4t + i],
//               w=2 qh[32h + 16v + 4t + i];
//             int8 sub-scales at 128*192 + r*16; f16 d at 128*208 + r*2
//   Q8_0  qs  tile (g,c) at (g*K + 256c)*128 bytes, [block j][row r][32 bytes]:
//             stored byte 8t + 4u + i  <-  block byte 16u + 4t + i (u = 16-element half)
//         d   u16 at ((g*nchunk + c)*128 + r)*8 + j (8 slots per chunk; unused ones 0)
//   F16, BF16 q  tile (g,c) at (g*K + 256c)*128*2 bytes, [16-element group j][row r]
//             [16 elements]: thread t's four elements 4t..4t+3 of a group are 8 contiguous bytes
//   Q4_0, Q4_1, Q5_0, Q5_1  q  tile (g,c) at (g*K/2 + 128c)*128 bytes, [block j][row r]
//             [16 bytes]: stored byte 4t + i  <-  qs byte 4t + {0,2,1,3}[i]; d as Q8_0's;
//         dm  (Q4_1, Q5_1) u16 m, laid out as d
//         qh  (Q5_0, Q5_1) u32 at (g*K/32 + 8c + j)*128 + r: the fifth bits regrouped,
//             bit 4r' + t and 16 + 4r' + t = the two elements of fragment register r'
//             of thread t (r' = 0, 1: elements 4t + 2r', +1; r' = 2, 3: 16 + 4t + 2(r'-2), +1)
// Prefill operand planes (MQ_REG_NO_MMQ_PLANE skips them), K-major for TMA:
//   w      f16  [N][K]    integer weight W_int: Q8_0 q; Q4_0 n - 8; Q5_0 q - 16; Q4_1 / Q5_1
//                         q; Q4_K sc_j*nib (<= 945); Q5_K sc_j*q (<= 1953);
//                         Q6_K the even part 2*floor(v/2) of v = sc*(q-32) (|v| <= 4096)
//   w2     f16  [N][K]    Q6_K only: the odd part v - 2*floor(v/2) in {0, 1}
//                         (every value exact in f16; w + w2 = v)
//   td     f32  [K/32][Np] block scale d of each 32-element block (transposed;
//                          Np = N rounded up to 128, the padding is zero)
//   tm     f32  [K/32][Np] min types only: dmin*m_j (Q4_K, Q5_K) or -m (Q4_1, Q5_1) of each
//                          block (transposed)
//   mb     f16  [Np][min_ld] min-term operand (Q4_K, Q5_K: dmin*m_j; Q4_1, Q5_1: -m),
//                          row n holds hi | lo | hi over the blocks of m~ = tm / v_n
//                          (hi = f16(m~), lo = f16(m~ - hi))
//   vcol   f32  [Np]       min types only: v_n, a power of two with max_b |tm| / v_n in
//                          [2^13, 2^14) (0 for the padding rows)
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mq.h"

struct mq_weight {
  int type;
  int64_t N, K;
  int64_t np;            // N rounded up to 128: row stride of the transposed planes
  int64_t ngroup;        // decode-plane row groups (N rounded up to 128, / 128)
  int nchunk;            // decode-plane K chunks (K / 256 rounded up)
  int device;
  size_t payload;        // GGUF bytes
  int ffn_gu = 0;        // fused gate/up weight: rows in units of 16 = 8 gate rows, then
                         // the same 8 rows of the up weight (N = 2 x the gate rows)
  size_t device_bytes;   // all planes
  // decode planes
  uint8_t *q = nullptr;  // Q8_0 / Q4_0 / Q4_1 / Q5_x quants, Q4_K / Q5_K / Q6_K tiles
  uint16_t *d = nullptr; // per-32-block types: block d
  uint32_t *qh = nullptr; // Q5_0 / Q5_1: fifth-bit words, one per (block, row)
  uint16_t *dm = nullptr; // Q4_1 / Q5_1: block m (the additive min)
  // prefill operand planes
  __half *mw = nullptr;
  __half *mw2 = nullptr;
  float *td = nullptr;
  float *tm = nullptr;
  __half *mb = nullptr;
  float *vcol = nullptr;
  alignas(64) unsigned char tmap_w[128];   // TMA descriptors of w and w2 (CUtensorMap)
  alignas(64) unsigned char tmap_w2[128];
  alignas(64) unsigned char tmap_mb[128];
  alignas(64) unsigned char tmap_td[128];  // td as 8-block x 128-row boxes
};

namespace mq {

constexpr int kMaxB = 8;
constexpr int kRowGroup = 128; // decode-plane row group (rows per matvec CTA)
constexpr int kChunk = 256;    // decode-plane K chunk
constexpr int kStatusTimeout = 1;

// ---- per-thread error reporting ------------------------------------------
mq_status fail(mq_status s, const char *fmt, ...);
mq_status cuda_fail(cudaError_t e, const char *call, const char *site);

// Per-device state set up by mq_init.
struct DeviceState {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
  int *status = nullptr;  // device status word for bounded waits (code, kernel id)
  cudaStream_t reg_stream = nullptr;
  uint8_t *static_xq = nullptr;  // mq_mmq_fused_static's scratch (device symbol address)
  // mq_mmq_host: the stream that copies y back while the MMQ's next rows run, and its events
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ev_rows = nullptr, ev_copied = nullptr;
  // split-K matvec (matvec.cu): the most clusters of S CTAs that can be resident at once
  // for every kernel of a weight type, by type id (the GGUF number, < 32) and S = 1..16
  // (0: that cluster size cannot run); filled by init_matvec
  int mv_clusters[32][17] = {};
  // the stream-ordered pool of the per-call activation fragment planes of the persistent
  // matvec's Q4_K / Q5_K two-tile calls (nullptr: its x warps convert x themselves)
  cudaMemPool_t xpool = nullptr;
};
DeviceState *device_state(int dev);  // nullptr if mq_init(dev) was not called
mq_status current_state(DeviceState **st, const char *site);

// ---- kernel launchers (defined per translation unit) ----------------------
mq_status repack_weight(mq_weight *w, const uint8_t *raw_dev, bool mmq, cudaStream_t s);
mq_status unpack_weight(const mq_weight *w, uint8_t *raw_dev, cudaStream_t s);
mq_status launch_matvec(const mq_weight *W, const float *x, float *y, int B, cudaStream_t s,
                        const DeviceState *st);
// the super-block types' persistent decode matvec (matvec_kq.cu), for weights of at least
// SMs / 2 row groups of 128 (matvec_kq_applies); launch_matvec dispatches to it
bool matvec_kq_applies(int64_t N, int sms);
mq_status launch_matvec_kq(const mq_weight *W, const float *x, float *y, int B, cudaStream_t s,
                           const DeviceState *st);
// The activation fragment plane of the persistent matvec's Q4_K / Q5_K two-tile calls
// (xplane.cu): its
// size for B rows of K, and the launch that converts x into it.
size_t xplane_bytes(int B, int64_t K);
mq_status launch_xplane(const float *x, int B, int64_t K, uint8_t *plane, cudaStream_t s);
mq_status launch_quantize(const float *x, void *xq, int64_t M, int64_t K, cudaStream_t s);
// x non-null: the fused form (the kernel quantises x into xq first; cooperative launch)
// sync non-null: the grid barrier's words there instead of inside xq
// mt_begin, mt_count: only the output rows of M-tiles (128 rows) mt_begin .. + mt_count - 1
// (mt_count < 0: all; the fused form takes all)
mq_status launch_mmq(const mq_weight *W, const void *xq, float *y, int32_t *D, int64_t M,
                     cudaStream_t s, const DeviceState *st, int debug_expire,
                     const float *x = nullptr, unsigned *sync = nullptr, int64_t mt_begin = 0,
                     int64_t mt_count = -1);
mq_status encode_weight_maps(mq_weight *w);  // TMA descriptors of the prefill planes
// Host-buffer transfers (host_io.cu).  host_device_view: the device view of p if p is
// page-locked host memory that this device can map and both p and its view are aligned to
// `align` bytes, else nullptr.  launch_copy_in: dst[0..n) = src_view[0..n) by SM loads of
// the view (n a multiple of 4, both 16-byte aligned); the next launch, if it carries the
// programmatic-serialisation attribute, overlaps it and waits for it before reading dst.
const void *host_device_view(const void *p, size_t align);
mq_status launch_copy_in(const float *src_view, float *dst, int64_t n, cudaStream_t s, int sms);
// Failure-injection seam for the launch-failure test: with MQ_TEST_FAIL_LAUNCH=1 in the
// environment of the last mq_init call, the matvec and MMQ launches are configured with an
// empty grid, which the runtime refuses before any kernel runs.
int test_fail_launch();
// Test seam: with MQ_TEST_NO_XPLANE=1 at the last mq_init, the persistent matvec's two-tile
// calls run without the activation fragment plane (the path taken when the pool cannot give
// one), so that path is covered by the tests.
int test_no_xplane();
mq_status init_kernels(DeviceState *st);  // smem opt-ins of the MMQ kernels
mq_status init_matvec(DeviceState *st);   // smem opt-ins of the matvec kernels
mq_status init_matvec_kq(DeviceState *st);

// xq buffer layout (mq_act_bytes): q int8 [M][K], s f32 [M][K/32], S int32
// [M][K/32], q as f16 [M][K], then the transposed block scales sT f32
// [K/32][Mt] and the min-term factors tT = s*S f32 [K/32][Mt], Mt = M rounded up
// to 128 (the epilogue's tile rows are one contiguous 512-byte run per block);
// then the min-term operand f16 [M][min_ld] (row m: t~hi | t~hi | t~lo over the
// blocks, t~ = s*S/u_m) and the row factors u_m f32 [Mt] (powers of two); last, the two
// u32 words of the grid barrier of the fused quantise + MMQ (arrival count, zero between
// its calls; generation).
struct ActLayout {
  size_t qs, scale, bsum, op, st, tt, amin, urow, sync, total;
  int64_t mt;
};
__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
__host__ __device__ inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
// Row stride (elements) of the min-term operands [rows][3*K/32]: rounded up to 8 so that
// every row starts on a 16-byte boundary (a TMA stride rule); the columns past 3*K/32 are
// never read (the tensor maps end at 3*K/32 and fill beyond it with zeros).
__host__ __device__ inline int64_t min_ld(int64_t nb) { return (3 * nb + 7) / 8 * 8; }
__host__ __device__ inline ActLayout act_layout(int64_t M, int64_t K) {
  ActLayout L;
  L.mt = round_up(M, 128);
  L.qs = 0;
  L.scale = align256(L.qs + size_t(M) * K);
  L.bsum = align256(L.scale + size_t(M) * (K / 32) * 4);
  L.op = align256(L.bsum + size_t(M) * (K / 32) * 4);
  L.st = align256(L.op + size_t(M) * K * 2);
  L.tt = align256(L.st + size_t(L.mt) * (K / 32) * 4);
  L.amin = align256(L.tt + size_t(L.mt) * (K / 32) * 4);
  L.urow = align256(L.amin + size_t(M) * min_ld(K / 32) * 2);
  L.sync = align256(L.urow + size_t(L.mt) * 4);
  L.total = align256(L.sync + 8);
  return L;
}

inline bool float_type(int type) { return type == MQ_F16 || type == MQ_BF16; }
inline int block_elems(int type) {
  return (type == MQ_Q4_K || type == MQ_Q5_K || type == MQ_Q6_K) ? 256 : 32;
}
inline int block_bytes(int type) {
  switch (type) {
    case MQ_Q4_0: return 18;
    case MQ_Q4_1: return 20;
    case MQ_Q5_0: return 22;
    case MQ_Q5_1: return 24;
    case MQ_Q8_0: return 34;
    case MQ_Q4_K: return 144;
    case MQ_Q5_K: return 176;
    case MQ_F16: return 64;   // 32 elements of 2 bytes (the K % 32 unit)
    case MQ_BF16: return 64;
    default: return 210;
  }
}

// Checked launch: reads the launch's own error at the site ("CUDA Backend
// Design" §4.9 rule 5).
#define MQ_LAUNCH_CHECK(name)                                                      \
  do {                                                                             \
    cudaError_t e_ = cudaGetLastError();                                           \
    if (e_ != cudaSuccess)                                                         \
      return ::mq::fail(MQ_ERR_LAUNCH, "launch of %s failed: %s (%s)", name,       \
                        cudaGetErrorName(e_), cudaGetErrorString(e_));             \
  } while (0)

}  // namespace mq
