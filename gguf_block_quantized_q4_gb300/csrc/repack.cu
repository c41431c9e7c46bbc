// repack.cu -- registration-time repack of GGUF blocks into the device planes
// described in mq_common.cuh, and the inverse (unpack) used to verify that the
// decode planes are a lossless regrouping.
//
// Block formats (GGUF; byte ratios per "minfer CUDA Backend Design" §2.3):
//   Q8_0  34 B / 32 el : f16 d, int8 q[32];                 w = d*q
//   Q4_K 144 B / 256 el: f16 d, f16 dmin, u8 scales[12], u8 qs[128]
//         sub-block j (elements 32j..32j+31) has a 6-bit scale sc_j and min m_j:
//           j<4 : sc = s[j]&63,                    m = s[j+4]&63
//           j>=4: sc = (s[j+4]&15) | (s[j-4]>>6)<<4, m = (s[j+4]>>4) | (s[j]>>6)<<4
//         element 64c + 32h + l is nibble h of qs[32c + l];  w = d*sc_j*nib - dmin*m_j
//   Q4_0  18 B / 32 el : f16 d, u8 qs[16]; element j < 16 = low nibble of qs[j],
//         element 16 + j = its high nibble;                  w = d*(nib - 8)
//   Q4_1, Q5_0, Q5_1: as Q4_0 with an additive min and / or a fifth-bit word (below)
//   Q5_K 176 B / 256 el: as Q4_K (d, dmin, scales[12]), u8 qh[32], u8 qs[128];
//         element 64c + 32h + l: nibble h of qs[32c + l] plus bit 2c + h of qh[l] << 4
//   Q6_K 210 B / 256 el: u8 ql[128], u8 qh[64], int8 sc[16], f16 d
//         element 128h + 32r + l: low 4 bits from ql[64h + 32(r%2) + l] (low nibble
//         for r<2, high for r>=2), high 2 bits = (qh[32h + l] >> 2r) & 3;
//         w = d * sc[e/16] * (q - 32)
// The prefill planes hold the integer weight W_int (Q8_0 q; Q4_0 nib - 8; Q5_0 q - 16;
// Q4_1 / Q5_1 the unsigned q, their min m entering through tm = -m; Q4_K sc_j*nib,
// at most 945, and Q5_K sc_j*q, at most 1953, exact in f16; Q6_K v = sc*(q-32),
// |v| <= 4096, stored as its even
// part 2*floor(v/2) plus its odd part in {0,1}, both exact in f16) and the
// transposed f32 block-scale planes td (d) and tm (Q4_K dmin*m_j).
#include "mq_common.cuh"

namespace mq {
namespace {

__device__ __forceinline__ float f16bits(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t rd16(const uint8_t *p) {
  return (uint16_t)(p[0] | (p[1] << 8));
}

__device__ __forceinline__ void q4k_scale_min(const uint8_t *s, int j, int &sc, int &m) {
  if (j < 4) {
    sc = s[j] & 63;
    m = s[j + 4] & 63;
  } else {
    sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
}

// One thread per GGUF block.
// Byte offset of block b of row n in the Q8_0 decode plane, and index of its d.
__device__ __forceinline__ int64_t q8_0_off(int64_t n, int64_t b, int64_t K) {
  const int64_t g = n / kRowGroup, r = n % kRowGroup, c = b / 8, j = b % 8;
  return (g * K + int64_t(kChunk) * c) * kRowGroup + (j * kRowGroup + r) * 32;
}
__device__ __forceinline__ int64_t q8_0_doff(int64_t n, int64_t b, int nchunk) {
  const int64_t g = n / kRowGroup, r = n % kRowGroup, c = b / 8, j = b % 8;
  return ((g * nchunk + c) * kRowGroup + r) * 8 + j;
}
__device__ __forceinline__ int64_t tile_row(int64_t n, int64_t c, int nchunk) {
  return (n / kRowGroup * nchunk + c) * kRowGroup + n % kRowGroup;
}
// Q4_K: byte i of a stored quant word comes from element offset kQ4kPerm[i] of the
// thread's 4 consecutive qs bytes (elements 4t, 4t+1 land in bytes 0 and 2).
__constant__ int kQ4kPerm[4] = {0, 2, 1, 3};
// Q6_K: byte offset of the tile holding (row n, super-block c); the tile is
// [128 rows][192 quant bytes], then [128][16] sub-scales, then [128] f16 d.
constexpr int64_t kQ6kTile = int64_t(kRowGroup) * 210;
__device__ __forceinline__ int64_t q6k_tile(int64_t n, int64_t c, int nchunk) {
  return (n / kRowGroup * nchunk + c) * kQ6kTile;
}

__global__ void repack_q8_0(const uint8_t *__restrict__ raw, int64_t N, int64_t K, int64_t NP,
                            uint8_t *__restrict__ q, uint16_t *__restrict__ d,
                            __half *__restrict__ mw, float *__restrict__ td) {
  const int64_t nb = K / 32;
  const int nchunk = (int)((K + kChunk - 1) / kChunk);
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nb) return;
  const int64_t n = i / nb, b = i % nb;
  const uint8_t *src = raw + i * 34;
  const uint16_t dbits = rd16(src);
  d[q8_0_doff(n, b, nchunk)] = dbits;
  uint8_t *dst = q + q8_0_off(n, b, K);
  for (int t = 0; t < 4; ++t)
    for (int u = 0; u < 2; ++u)
      for (int e = 0; e < 4; ++e) dst[8 * t + 4 * u + e] = src[2 + 16 * u + 4 * t + e];
  if (mw) {
    for (int e = 0; e < 32; ++e) mw[n * K + b * 32 + e] = __int2half_rn((int8_t)src[2 + e]);
    td[b * NP + n] = f16bits(dbits);
  }
}

__global__ void unpack_q8_0(const uint8_t *__restrict__ q, const uint16_t *__restrict__ d,
                            int64_t N, int64_t K, uint8_t *__restrict__ raw) {
  const int64_t nb = K / 32;
  const int nchunk = (int)((K + kChunk - 1) / kChunk);
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nb) return;
  const int64_t n = i / nb, b = i % nb;
  uint8_t *dst = raw + i * 34;
  const uint16_t dv = d[q8_0_doff(n, b, nchunk)];
  dst[0] = dv & 255;
  dst[1] = dv >> 8;
  const uint8_t *src = q + q8_0_off(n, b, K);
  for (int t = 0; t < 4; ++t)
    for (int u = 0; u < 2; ++u)
      for (int e = 0; e < 4; ++e) dst[2 + 16 * u + 4 * t + e] = src[8 * t + 4 * u + e];
}

// One thread per super-block.
__global__ void repack_q4_k(const uint8_t *__restrict__ raw, int64_t N, int64_t K, int64_t NP,
                            uint8_t *__restrict__ q, __half *__restrict__ mw,
                            float *__restrict__ td, float *__restrict__ tm) {
  const int64_t nsb = K / 256;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nsb) return;
  const uint8_t *src = raw + i * 144;
  uint8_t *dst = q + tile_row(i / nsb, i % nsb, (int)nsb) * 144;
  for (int e = 0; e < 16; ++e) dst[e] = src[e];
  for (int t = 0; t < 4; ++t)
    for (int c = 0; c < 4; ++c)
      for (int u = 0; u < 2; ++u)
        for (int e = 0; e < 4; ++e)
          dst[16 + 32 * t + 4 * (2 * c + u) + e] = src[16 + 32 * c + 16 * u + 4 * t + kQ4kPerm[e]];
  if (td) {  // the prefill planes; the f16 integer plane only where one is asked for
    const int64_t n = i / nsb, s = i % nsb;
    const float dd = f16bits(rd16(src)), dmin = f16bits(rd16(src + 2));
    for (int j = 0; j < 8; ++j) {
      int sc, m;
      q4k_scale_min(src + 4, j, sc, m);
      const int c = j / 2, h = j % 2;
      if (mw) {
        for (int l = 0; l < 32; ++l) {
          const int nib = (src[16 + 32 * c + l] >> (4 * h)) & 15;
          mw[n * K + s * 256 + 32 * j + l] = __int2half_rn(sc * nib);
        }
      }
      td[(s * 8 + j) * NP + n] = dd;
      tm[(s * 8 + j) * NP + n] = dmin * (float)m;
    }
  }
}

__global__ void unpack_q4_k(const uint8_t *__restrict__ q, int64_t N, int64_t K,
                            uint8_t *__restrict__ raw) {
  const int64_t nsb = K / 256;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nsb) return;
  const uint8_t *src = q + tile_row(i / nsb, i % nsb, (int)nsb) * 144;
  uint8_t *dst = raw + i * 144;
  for (int e = 0; e < 16; ++e) dst[e] = src[e];
  for (int t = 0; t < 4; ++t)
    for (int c = 0; c < 4; ++c)
      for (int u = 0; u < 2; ++u)
        for (int e = 0; e < 4; ++e)
          dst[16 + 32 * c + 16 * u + 4 * t + kQ4kPerm[e]] = src[16 + 32 * t + 4 * (2 * c + u) + e];
}

// Per-32-block nibble types.  Decode plane per (row group, chunk): [8 blocks][128 rows]
// [16 bytes]; word t of a (block, row) holds quant bytes 4t + kQ4kPerm[e] (the block's
// elements 4t..4t+3 in its low nibbles, elements 16 + 4t.. in its high nibbles).  The d
// plane (and, for Q4_1 / Q5_1, the m plane) is laid out as Q8_0's d.  Q5_0 / Q5_1 add one
// 32-bit fifth-bit word per (block, row), [8 blocks][128 rows] per (row group, chunk),
// whose bits are regrouped so that fragment thread t finds the pair of elements of its
// register r (r = 0, 1: elements 4t + 2r, +1; r = 2, 3: elements 16 + 4t + 2(r - 2), +1)
// at bits 4r + t and 16 + 4r + t.
//   Q4_0  18 B: f16 d, qs[16];                        w = d*(nib - 8)
//   Q4_1  20 B: f16 d, f16 m, qs[16];                 w = d*nib + m
//   Q5_0  22 B: f16 d, u32 qh, qs[16];                w = d*(q - 16), q = nib | bit e of qh << 4
//   Q5_1  24 B: f16 d, f16 m, u32 qh, qs[16];         w = d*q + m
__device__ __forceinline__ int64_t q4_0_off(int64_t n, int64_t b, int64_t K) {
  const int64_t g = n / kRowGroup, r = n % kRowGroup, c = b / 8, j = b % 8;
  return (g * (K / 2) + int64_t(kChunk / 2) * c) * kRowGroup + (j * kRowGroup + r) * 16;
}
// index of the fifth-bit word of (row n, block b)
__device__ __forceinline__ int64_t qh_idx(int64_t n, int64_t b, int64_t K) {
  return (n / kRowGroup * (K / 32) + b) * kRowGroup + n % kRowGroup;
}
// raw element of the low bit of the pair at stored bit 4r + t
__device__ __forceinline__ int qh_elem(int r, int t) { return 16 * (r >> 1) + 4 * t + 2 * (r & 1); }
__device__ __forceinline__ uint32_t qh_regroup(uint32_t h) {
  uint32_t o = 0;
  for (int r = 0; r < 4; ++r)
    for (int t = 0; t < 4; ++t) {
      const int e = qh_elem(r, t);
      o |= ((h >> e) & 1u) << (4 * r + t);
      o |= ((h >> (e + 1)) & 1u) << (16 + 4 * r + t);
    }
  return o;
}
__device__ __forceinline__ uint32_t qh_restore(uint32_t o) {
  uint32_t h = 0;
  for (int r = 0; r < 4; ++r)
    for (int t = 0; t < 4; ++t) {
      const int e = qh_elem(r, t);
      h |= ((o >> (4 * r + t)) & 1u) << e;
      h |= ((o >> (16 + 4 * r + t)) & 1u) << (e + 1);
    }
  return h;
}
template <int TYPE>
struct Nib32 {
  static constexpr bool MADD = TYPE == MQ_Q4_1 || TYPE == MQ_Q5_1;  // additive min m
  static constexpr bool Q5 = TYPE == MQ_Q5_0 || TYPE == MQ_Q5_1;    // fifth bits
  static constexpr int BB = 18 + (MADD ? 2 : 0) + (Q5 ? 4 : 0);      // block bytes
  static constexpr int QO = BB - 16;                                // quant bytes offset
  static constexpr int HO = MADD ? 4 : 2;                           // fifth-bit word offset
};

// One thread per block.  Prefill planes: W_int = nib - 8 (Q4_0), q - 16 (Q5_0) or the
// unsigned q (Q4_1, Q5_1); td = d; tm = -m (the min term enters as y -= sum tm * s * S).
template <int TYPE>
__global__ void repack_nib32(const uint8_t *__restrict__ raw, int64_t N, int64_t K, int64_t NP,
                             uint8_t *__restrict__ q, uint16_t *__restrict__ d,
                             uint16_t *__restrict__ dm, uint32_t *__restrict__ qh,
                             __half *__restrict__ mw, float *__restrict__ td,
                             float *__restrict__ tm) {
  using T = Nib32<TYPE>;
  const int64_t nb = K / 32;
  const int nchunk = (int)((K + kChunk - 1) / kChunk);
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nb) return;
  const int64_t n = i / nb, b = i % nb;
  const uint8_t *src = raw + i * T::BB;
  const uint16_t dbits = rd16(src);
  d[q8_0_doff(n, b, nchunk)] = dbits;
  if (T::MADD) dm[q8_0_doff(n, b, nchunk)] = rd16(src + 2);
  uint32_t h = 0;
  if (T::Q5) {
    h = (uint32_t)src[T::HO] | ((uint32_t)src[T::HO + 1] << 8) | ((uint32_t)src[T::HO + 2] << 16) |
        ((uint32_t)src[T::HO + 3] << 24);
    qh[qh_idx(n, b, K)] = qh_regroup(h);
  }
  uint8_t *dst = q + q4_0_off(n, b, K);
  for (int t = 0; t < 4; ++t)
    for (int e = 0; e < 4; ++e) dst[4 * t + e] = src[T::QO + 4 * t + kQ4kPerm[e]];
  if (mw) {
    for (int e = 0; e < 32; ++e) {
      const int nib = (src[T::QO + (e & 15)] >> (4 * (e >> 4))) & 15;
      const int qv = T::Q5 ? nib | (int)(((h >> e) & 1u) << 4) : nib;
      const int wint = T::MADD ? qv : (T::Q5 ? qv - 16 : qv - 8);
      mw[n * K + b * 32 + e] = __int2half_rn(wint);
    }
    td[b * NP + n] = f16bits(dbits);
    if (T::MADD) tm[b * NP + n] = -f16bits(rd16(src + 2));
  }
}

template <int TYPE>
__global__ void unpack_nib32(const uint8_t *__restrict__ q, const uint16_t *__restrict__ d,
                             const uint16_t *__restrict__ dm, const uint32_t *__restrict__ qh,
                             int64_t N, int64_t K, uint8_t *__restrict__ raw) {
  using T = Nib32<TYPE>;
  const int64_t nb = K / 32;
  const int nchunk = (int)((K + kChunk - 1) / kChunk);
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nb) return;
  const int64_t n = i / nb, b = i % nb;
  uint8_t *dst = raw + i * T::BB;
  const uint16_t dv = d[q8_0_doff(n, b, nchunk)];
  dst[0] = dv & 255;
  dst[1] = dv >> 8;
  if (T::MADD) {
    const uint16_t mv = dm[q8_0_doff(n, b, nchunk)];
    dst[2] = mv & 255;
    dst[3] = mv >> 8;
  }
  if (T::Q5) {
    const uint32_t h = qh_restore(qh[qh_idx(n, b, K)]);
    for (int k = 0; k < 4; ++k) dst[T::HO + k] = (uint8_t)(h >> (8 * k));
  }
  const uint8_t *src = q + q4_0_off(n, b, K);
  for (int t = 0; t < 4; ++t)
    for (int e = 0; e < 4; ++e) dst[T::QO + 4 * t + kQ4kPerm[e]] = src[4 * t + e];
}

// F16 / BF16 decode plane: per (row group, chunk), [16-element group j][128 rows][32 bytes],
// the group's elements in their natural order (thread t's elements 4t..4t+3 are bytes
// 8t..8t+7).  One thread per (row, group): 32 bytes, as two 16-byte words.
__device__ __forceinline__ int64_t float_off(int64_t n, int64_t grp, int64_t K) {
  const int64_t g = n / kRowGroup, r = n % kRowGroup, c = grp / 16, j = grp % 16;
  return (g * K + int64_t(kChunk) * c) * kRowGroup * 2 + (j * kRowGroup + r) * 32;
}

__global__ void repack_float(const uint8_t *__restrict__ raw, int64_t N, int64_t K,
                             uint8_t *__restrict__ q) {
  const int64_t ng = K / 16;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * ng) return;
  const uint4 *src = reinterpret_cast<const uint4 *>(raw + i * 32);
  uint4 *dst = reinterpret_cast<uint4 *>(q + float_off(i / ng, i % ng, K));
  dst[0] = src[0];
  dst[1] = src[1];
}

__global__ void unpack_float(const uint8_t *__restrict__ q, int64_t N, int64_t K,
                             uint8_t *__restrict__ raw) {
  const int64_t ng = K / 16;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * ng) return;
  const uint4 *src = reinterpret_cast<const uint4 *>(q + float_off(i / ng, i % ng, K));
  uint4 *dst = reinterpret_cast<uint4 *>(raw + i * 32);
  dst[0] = src[0];
  dst[1] = src[1];
}

// Q5_K decode tile: 128 rows x 176 bytes, row = 16-byte header (d, dmin, scales), the
// 128 quant bytes regrouped as Q4_K's, then the 32 fifth-bit bytes regrouped per
// fragment thread: bytes 8t + 4u + e hold bits byte 16u + 4t + kQ4kPerm[e].
__global__ void repack_q5_k(const uint8_t *__restrict__ raw, int64_t N, int64_t K, int64_t NP,
                            uint8_t *__restrict__ q, __half *__restrict__ mw,
                            float *__restrict__ td, float *__restrict__ tm) {
  const int64_t nsb = K / 256;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nsb) return;
  const uint8_t *src = raw + i * 176;
  uint8_t *dst = q + tile_row(i / nsb, i % nsb, (int)nsb) * 176;
  for (int e = 0; e < 16; ++e) dst[e] = src[e];
  for (int t = 0; t < 4; ++t)
    for (int c = 0; c < 4; ++c)
      for (int u = 0; u < 2; ++u)
        for (int e = 0; e < 4; ++e)
          dst[16 + 32 * t + 4 * (2 * c + u) + e] = src[48 + 32 * c + 16 * u + 4 * t + kQ4kPerm[e]];
  for (int t = 0; t < 4; ++t)
    for (int u = 0; u < 2; ++u)
      for (int e = 0; e < 4; ++e) dst[144 + 8 * t + 4 * u + e] = src[16 + 16 * u + 4 * t + kQ4kPerm[e]];
  if (mw) {
    const int64_t n = i / nsb, s = i % nsb;
    const float dd = f16bits(rd16(src)), dmin = f16bits(rd16(src + 2));
    for (int j = 0; j < 8; ++j) {
      int sc, m;
      q4k_scale_min(src + 4, j, sc, m);
      const int c = j / 2, h = j % 2;
      for (int l = 0; l < 32; ++l) {
        const int q5 = ((src[48 + 32 * c + l] >> (4 * h)) & 15) | (((src[16 + l] >> j) & 1) << 4);
        mw[n * K + s * 256 + 32 * j + l] = __int2half_rn(sc * q5);
      }
      td[(s * 8 + j) * NP + n] = dd;
      tm[(s * 8 + j) * NP + n] = dmin * (float)m;
    }
  }
}

__global__ void unpack_q5_k(const uint8_t *__restrict__ q, int64_t N, int64_t K,
                            uint8_t *__restrict__ raw) {
  const int64_t nsb = K / 256;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nsb) return;
  const uint8_t *src = q + tile_row(i / nsb, i % nsb, (int)nsb) * 176;
  uint8_t *dst = raw + i * 176;
  for (int e = 0; e < 16; ++e) dst[e] = src[e];
  for (int t = 0; t < 4; ++t)
    for (int c = 0; c < 4; ++c)
      for (int u = 0; u < 2; ++u)
        for (int e = 0; e < 4; ++e)
          dst[48 + 32 * c + 16 * u + 4 * t + kQ4kPerm[e]] = src[16 + 32 * t + 4 * (2 * c + u) + e];
  for (int t = 0; t < 4; ++t)
    for (int u = 0; u < 2; ++u)
      for (int e = 0; e < 4; ++e) dst[16 + 16 * u + 4 * t + kQ4kPerm[e]] = src[144 + 8 * t + 4 * u + e];
}

// Byte offset in the raw Q6_K block of word w (0: ql low pair, 1: ql high pair,
// 2: qh) of fragment thread t for half h and 16-element half v.
__device__ __forceinline__ int q6k_src(int t, int h, int v, int w) {
  return w == 0 ? 64 * h + 16 * v + 4 * t
                : (w == 1 ? 64 * h + 32 + 16 * v + 4 * t : 128 + 32 * h + 16 * v + 4 * t);
}

__global__ void repack_q6_k(const uint8_t *__restrict__ raw, int64_t N, int64_t K, int64_t NP,
                            uint8_t *__restrict__ q, __half *__restrict__ mw,
                            __half *__restrict__ mw2, float *__restrict__ td) {
  const int64_t nsb = K / 256;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nsb) return;
  const uint8_t *src = raw + i * 210;
  const int64_t r = (i / nsb) % kRowGroup;
  uint8_t *tile = q + q6k_tile(i / nsb, i % nsb, (int)nsb);
  uint8_t *dst = tile + r * 192;
  for (int t = 0; t < 4; ++t)
    for (int h = 0; h < 2; ++h)
      for (int v = 0; v < 2; ++v)
        for (int w = 0; w < 3; ++w)
          for (int e = 0; e < 4; ++e)
            dst[48 * t + 4 * (3 * (2 * h + v) + w) + e] = src[q6k_src(t, h, v, w) + e];
  for (int e = 0; e < 16; ++e) tile[kRowGroup * 192 + r * 16 + e] = src[192 + e];
  const uint16_t dbits = rd16(src + 208);
  tile[kRowGroup * 208 + 2 * r] = src[208];
  tile[kRowGroup * 208 + 2 * r + 1] = src[209];
  if (mw) {
    const int64_t n = i / nsb, s = i % nsb;
    const float dd = f16bits(dbits);
    for (int e = 0; e < 256; ++e) {
      const int h = e / 128, r = (e / 32) % 4, l = e % 32;
      const int qlb = src[64 * h + 32 * (r % 2) + l];
      const int lo4 = r < 2 ? (qlb & 15) : (qlb >> 4);
      const int hi2 = (src[128 + 32 * h + l] >> (2 * r)) & 3;
      const int v = (int)(int8_t)src[192 + e / 16] * ((lo4 | (hi2 << 4)) - 32);
      const int odd = v & 1;  // v - 2*floor(v/2), two's complement
      mw[n * K + s * 256 + e] = __int2half_rn(v - odd);
      mw2[n * K + s * 256 + e] = __int2half_rn(odd);
    }
    for (int b = 0; b < 8; ++b) td[(s * 8 + b) * NP + n] = dd;
  }
}

__global__ void unpack_q6_k(const uint8_t *__restrict__ q, int64_t N, int64_t K,
                            uint8_t *__restrict__ raw) {
  const int64_t nsb = K / 256;
  const int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (i >= N * nsb) return;
  const int64_t r = (i / nsb) % kRowGroup;
  const uint8_t *tile = q + q6k_tile(i / nsb, i % nsb, (int)nsb);
  const uint8_t *src = tile + r * 192;
  uint8_t *dst = raw + i * 210;
  for (int t = 0; t < 4; ++t)
    for (int h = 0; h < 2; ++h)
      for (int v = 0; v < 2; ++v)
        for (int w = 0; w < 3; ++w)
          for (int e = 0; e < 4; ++e)
            dst[q6k_src(t, h, v, w) + e] = src[48 * t + 4 * (3 * (2 * h + v) + w) + e];
  for (int e = 0; e < 16; ++e) dst[192 + e] = tile[kRowGroup * 192 + r * 16 + e];
  dst[208] = tile[kRowGroup * 208 + 2 * r];
  dst[209] = tile[kRowGroup * 208 + 2 * r + 1];
}

// Q4_K min-term operand (one thread per weight row n): v_n = 2^k with
// max_b |dmin*m_j| / v_n in [2^13, 2^14), and m~ = dmin*m_j / v_n split into
// f16 hi and lo, stored as hi | lo | hi over the blocks (paired with the
// activation side's hi | hi | lo, the three products hi*hi + hi*lo + lo*hi).
__global__ void minplane_q4_k(const float *__restrict__ tm, int64_t N, int64_t nb, int64_t NP,
                              __half *__restrict__ mb, float *__restrict__ vcol) {
  const int64_t n = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (n >= N) return;
  float mx = 0.f;
  for (int64_t b = 0; b < nb; ++b) mx = fmaxf(mx, fabsf(tm[b * NP + n]));
  const int E = (int)((__float_as_uint(mx) >> 23) & 255);
  int k = mx == 0.f ? 0 : E - 140;
  k = min(max(k, -100), 100);
  const float inv_v = __int_as_float((127 - k) << 23);
  vcol[n] = __int_as_float((127 + k) << 23);
  __half *row = mb + n * min_ld(nb);
  for (int64_t b = 0; b < nb; ++b) {
    const float t = tm[b * NP + n] * inv_v;
    const __half hi = __float2half_rn(t);
    const __half lo = __float2half_rn(t - __half2float(hi));
    row[b] = hi;
    row[nb + b] = lo;
    row[2 * nb + b] = hi;
  }
}

inline unsigned grid_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

mq_status repack_weight(mq_weight *w, const uint8_t *raw, bool mmq, cudaStream_t s) {
  const int T = 128;
  const int64_t N = w->N, K = w->K;
  if (float_type(w->type)) {
    repack_float<<<grid_for(N * (K / 16), T), T, 0, s>>>(raw, N, K, w->q);
    MQ_LAUNCH_CHECK("repack_float");
  } else if (w->type == MQ_Q8_0) {
    const int64_t n = N * (K / 32);
    repack_q8_0<<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, w->d, mmq ? w->mw : nullptr,
                                              w->td);
    MQ_LAUNCH_CHECK("repack_q8_0");
  } else if (block_elems(w->type) == 32) {
    const int64_t n = N * (K / 32);
    __half *mw = mmq ? w->mw : nullptr;
    switch (w->type) {
      case MQ_Q4_0:
        repack_nib32<MQ_Q4_0><<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, w->d, w->dm,
                                                           w->qh, mw, w->td, w->tm);
        break;
      case MQ_Q4_1:
        repack_nib32<MQ_Q4_1><<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, w->d, w->dm,
                                                           w->qh, mw, w->td, w->tm);
        break;
      case MQ_Q5_0:
        repack_nib32<MQ_Q5_0><<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, w->d, w->dm,
                                                           w->qh, mw, w->td, w->tm);
        break;
      default:
        repack_nib32<MQ_Q5_1><<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, w->d, w->dm,
                                                           w->qh, mw, w->td, w->tm);
    }
    MQ_LAUNCH_CHECK("repack_nib32");
    if (mmq && w->tm) {
      minplane_q4_k<<<grid_for(N, T), T, 0, s>>>(w->tm, N, K / 32, w->np, w->mb, w->vcol);
      MQ_LAUNCH_CHECK("minplane_q4_k");
    }
  } else if (w->type == MQ_Q4_K || w->type == MQ_Q5_K) {
    const int64_t n = N * (K / 256);
    if (w->type == MQ_Q4_K) {
      // (no f16 integer plane when the MMQ expands the decode-plane tiles itself)
      repack_q4_k<<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, mmq ? w->mw : nullptr,
                                                mmq ? w->td : nullptr, w->tm);
      MQ_LAUNCH_CHECK("repack_q4_k");
    } else {
      repack_q5_k<<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, mmq ? w->mw : nullptr,
                                                w->td, w->tm);
      MQ_LAUNCH_CHECK("repack_q5_k");
    }
    if (mmq) {
      minplane_q4_k<<<grid_for(N, T), T, 0, s>>>(w->tm, N, K / 32, w->np, w->mb, w->vcol);
      MQ_LAUNCH_CHECK("minplane_q4_k");
    }
  } else {
    const int64_t n = N * (K / 256);
    repack_q6_k<<<grid_for(n, T), T, 0, s>>>(raw, N, K, w->np, w->q, mmq ? w->mw : nullptr,
                                              w->mw2, w->td);
    MQ_LAUNCH_CHECK("repack_q6_k");
  }
  return MQ_OK;
}

mq_status unpack_weight(const mq_weight *w, uint8_t *raw, cudaStream_t s) {
  const int T = 128;
  const int64_t N = w->N, K = w->K;
  if (float_type(w->type)) {
    unpack_float<<<grid_for(N * (K / 16), T), T, 0, s>>>(w->q, N, K, raw);
    MQ_LAUNCH_CHECK("unpack_float");
  } else if (w->type == MQ_Q8_0) {
    unpack_q8_0<<<grid_for(N * (K / 32), T), T, 0, s>>>(w->q, w->d, N, K, raw);
    MQ_LAUNCH_CHECK("unpack_q8_0");
  } else if (block_elems(w->type) == 32) {
    const unsigned g = grid_for(N * (K / 32), T);
    switch (w->type) {
      case MQ_Q4_0:
        unpack_nib32<MQ_Q4_0><<<g, T, 0, s>>>(w->q, w->d, w->dm, w->qh, N, K, raw);
        break;
      case MQ_Q4_1:
        unpack_nib32<MQ_Q4_1><<<g, T, 0, s>>>(w->q, w->d, w->dm, w->qh, N, K, raw);
        break;
      case MQ_Q5_0:
        unpack_nib32<MQ_Q5_0><<<g, T, 0, s>>>(w->q, w->d, w->dm, w->qh, N, K, raw);
        break;
      default:
        unpack_nib32<MQ_Q5_1><<<g, T, 0, s>>>(w->q, w->d, w->dm, w->qh, N, K, raw);
    }
    MQ_LAUNCH_CHECK("unpack_nib32");
  } else if (w->type == MQ_Q4_K) {
    unpack_q4_k<<<grid_for(N * (K / 256), T), T, 0, s>>>(w->q, N, K, raw);
    MQ_LAUNCH_CHECK("unpack_q4_k");
  } else if (w->type == MQ_Q5_K) {
    unpack_q5_k<<<grid_for(N * (K / 256), T), T, 0, s>>>(w->q, N, K, raw);
    MQ_LAUNCH_CHECK("unpack_q5_k");
  } else {
    unpack_q6_k<<<grid_for(N * (K / 256), T), T, 0, s>>>(w->q, N, K, raw);
    MQ_LAUNCH_CHECK("unpack_q6_k");
  }
  return MQ_OK;
}

}  // namespace mq
