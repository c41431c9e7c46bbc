// matvec.cu -- decode matvec y[b][n] = sum_k w[n][k] x[b][k] for GGUF Q8_0 /
// Q4_K / Q6_K weights and f32 activations, B <= 8 ("minfer CUDA Backend Design"
// §4.4: the nt == 1 matvec and the _multi variants for nt 2..8).
//
// GB300 design.  The weights are streamed once from HBM with 16-byte loads
// and dequantised in registers straight into tensor-core fragments; the dot
// products run on the legacy warp-level tensor path (mma.sync m16n8k16, f16
// inputs, f32 accumulate).  This keeps the CUDA-core work per weight element
// to a few integer/f16x2 operations, independent of the batch size B:
//
//  * weight side (A operand, 16 rows x 16 K per MMA): the quants of one
//    16-element scale group become exact f16 integers -- Q4_K nibbles through
//    cvt.rn.f16x2.e4m3x2 (a byte n < 16 read as e4m3 is n * 2^-9 exactly),
//    Q6_K and Q8_0 through a byte permute into an f16 whose exponent makes the
//    low mantissa byte the integer, then one f16x2 subtraction.
//  * activation side (B operand, 16 K x 8 columns): x is staged per 256-element
//    chunk in shared memory as two f16 parts per batch row, hi = f16(x*2^e) and
//    lo = f16(x*2^e - hi), with 2^e a per-(row, chunk) power of two that puts
//    max|x| in [2^14, 2^15).  hi + lo carries 22 significant bits, so the
//    product error is ~2^-22 relative, far inside the 1e-4 * sum|w||x| bound.
//    Columns 2b and 2b+1 of an n8 tile hold hi and lo of batch row b, so one
//    thread's two accumulator columns are the two parts of the same row.
//  * per scale group the f32 MMA result is scaled by the group's weight scale
//    (and, for Q4_K, the min term -dmin*m_j*sum(x) is subtracted), then per
//    chunk by 2^-e.
//
// The fragment rule: thread t (of a quad) holds the elements 4t..4t+3 of each
// 16-element group; A register pairs are (4t, 4t+1) and (4t+2, 4t+3), matched
// by B pairs (x[4t], x[4t+1]) and (x[4t+2], x[4t+3]).  The decode planes
// (repack.cu) store each thread's words contiguously.
//
// Data movement: a CTA owns one 64-row group of the decode plane and a K-slice.
// A producer warp streams, per 256-element chunk, the group's weight tile (one
// contiguous run of the tiled decode plane) and the x chunk of every batch row
// into a 4-stage shared-memory ring with 1-D bulk copies (cp.async.bulk,
// mbarrier transaction counts); four compute warps, 16 rows each, read their
// fragment words from shared memory.  When one wave would be short of CTAs, K
// is split over a thread-block cluster of S CTAs whose partial sums are reduced
// through distributed shared memory in rank order (deterministic, and
// independent of B, so every column of a batched call equals the B = 1 call
// bitwise).  All mbarrier waits are bounded.
#include <cooperative_groups.h>

#include "mq_common.cuh"

namespace cg = cooperative_groups;

namespace mq {
namespace {

constexpr int kNS = 4;          // shared-memory ring stages
constexpr int kThreads = 160;   // 4 compute warps + 1 producer warp
constexpr uint64_t kWaitNs = 2000000000ull;

struct MvArgs {
  const uint8_t *q;
  const int8_t *sc;
  const uint16_t *d;
  const float *x;
  float *y;
  int64_t N, K;
  int B;
  int nchunk;  // ceil(K / 256)
  int S;       // K slices (cluster size)
  int *status;
};

// Bytes of one (64-row group, chunk) tile of the decode planes, as laid out in
// shared memory: Q4_K 64 x 144; Q6_K 64 x 192 quants, then 64 x 16 sub-scales,
// then 64 f16 d; Q8_0 64 x 256 quants (64 x chunk width used), then 64 x 8 f16 d.
template <int TYPE>
constexpr int tile_bytes() {
  return TYPE == MQ_Q4_K ? 64 * 144 : (TYPE == MQ_Q6_K ? 64 * 192 + 64 * 16 + 64 * 2
                                                       : 64 * 256 + 64 * 16);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two bytes < 16 -> f16x2 (n0 * 2^-9, n1 * 2^-9), exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)v16));
  return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 ldg16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ldg8(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Per-thread weight words of one chunk for the two rows (g, g+8) of the tile.
template <int TYPE>
struct WRegs;
template <>
struct WRegs<MQ_Q4_K> {  // 8 quant words per row + the decoded row's header
  uint32_t a[8], b[8];
  uint4 hdr;
};
template <>
struct WRegs<MQ_Q6_K> {  // 12 words per row
  uint32_t a[12], b[12];
  uint2 sc8;             // 8 sub-scales of the decoded row
  uint16_t dbits;
};
template <>
struct WRegs<MQ_Q8_0> {  // 2 words per row per block, 8 blocks
  uint32_t a[16], b[16];
  uint16_t da[8], db[8];
};

template <int TYPE, int NT>
struct MvSmem {
  alignas(128) uint8_t w[kNS][tile_bytes<TYPE>()];  // weight tiles
  alignas(128) float x[kNS][4 * NT][kChunk];        // x chunks of the batch rows
  uint2 frag[16][NT][32];      // B fragments of the staged chunk
  float xsum[8][8];            // Q4_K: per sub-block, per batch row sum of scaled x
  unsigned wmax[8 * NT];       // per 32-item slice max |x| bits
  float unscale[8];            // 2^-e per batch row of the chunk
  float tab[4][16][16];        // per-warp decoded scales of the tile's 16 rows
  float part[64][8];           // split-K partial sums
  uint64_t full[kNS], empty[kNS];
};

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
__device__ __forceinline__ void bulk_1d(uint32_t dst, const void *src, uint32_t bytes,
                                        uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The fragment words of one chunk for tile rows ra (g) and ra + 8, from the
// shared-memory tile (nblk = blocks in the chunk, Q8_0 only).
template <int TYPE>
__device__ __forceinline__ void load_words(const uint8_t *tile, WRegs<TYPE> &w, int ra, int t,
                                           int nblk) {
  const int rb = ra + 8;
  if constexpr (TYPE == MQ_Q4_K) {
    const uint4 a0 = *reinterpret_cast<const uint4 *>(tile + ra * 144 + 16 + 32 * t);
    const uint4 a1 = *reinterpret_cast<const uint4 *>(tile + ra * 144 + 32 + 32 * t);
    const uint4 b0 = *reinterpret_cast<const uint4 *>(tile + rb * 144 + 16 + 32 * t);
    const uint4 b1 = *reinterpret_cast<const uint4 *>(tile + rb * 144 + 32 + 32 * t);
    w.a[0] = a0.x; w.a[1] = a0.y; w.a[2] = a0.z; w.a[3] = a0.w;
    w.a[4] = a1.x; w.a[5] = a1.y; w.a[6] = a1.z; w.a[7] = a1.w;
    w.b[0] = b0.x; w.b[1] = b0.y; w.b[2] = b0.z; w.b[3] = b0.w;
    w.b[4] = b1.x; w.b[5] = b1.y; w.b[6] = b1.z; w.b[7] = b1.w;
    w.hdr = *reinterpret_cast<const uint4 *>(tile + ((t & 1) ? rb : ra) * 144);
  } else if constexpr (TYPE == MQ_Q6_K) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint4 va = *reinterpret_cast<const uint4 *>(tile + ra * 192 + 48 * t + 16 * i);
      const uint4 vb = *reinterpret_cast<const uint4 *>(tile + rb * 192 + 48 * t + 16 * i);
      w.a[4 * i] = va.x; w.a[4 * i + 1] = va.y; w.a[4 * i + 2] = va.z; w.a[4 * i + 3] = va.w;
      w.b[4 * i] = vb.x; w.b[4 * i + 1] = vb.y; w.b[4 * i + 2] = vb.z; w.b[4 * i + 3] = vb.w;
    }
    const int row = (t & 1) ? rb : ra;
    w.sc8 = *reinterpret_cast<const uint2 *>(tile + 64 * 192 + row * 16 + 8 * (t >> 1));
    w.dbits = *reinterpret_cast<const uint16_t *>(tile + 64 * 192 + 64 * 16 + row * 2);
  } else {  // Q8_0: [block j][row][32 bytes], then d [row][8]
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = j < nblk;
      const uint2 va = in ? *reinterpret_cast<const uint2 *>(tile + (j * 64 + ra) * 32 + 8 * t)
                          : make_uint2(0, 0);
      const uint2 vb = in ? *reinterpret_cast<const uint2 *>(tile + (j * 64 + rb) * 32 + 8 * t)
                          : make_uint2(0, 0);
      w.a[2 * j] = va.x; w.a[2 * j + 1] = va.y;
      w.b[2 * j] = vb.x; w.b[2 * j + 1] = vb.y;
      const uint16_t *dd = reinterpret_cast<const uint16_t *>(tile + 64 * 256);
      w.da[j] = in ? dd[ra * 8 + j] : (uint16_t)0;
      w.db[j] = in ? dd[rb * 8 + j] : (uint16_t)0;
    }
  }
}

// Split the staged x chunk (shared memory, raw f32) into f16 hi/lo fragments
// (see the file header).  Called by the 128 compute threads together.
template <int TYPE, int NT>
__device__ __forceinline__ void stage_x(MvSmem<TYPE, NT> &sm, int s, int B, int cw) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int kItems = (256 * NT) / 128;
  float4 xv[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int it = tid + k * 128;
    const int b = it >> 6, g = (it >> 2) & 15, t = it & 3;
    xv[k] = (b < B && 16 * g < cw) ? *reinterpret_cast<const float4 *>(&sm.x[s][b][16 * g + 4 * t])
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 v = xv[k];
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
    if (lane == 0) sm.wmax[it >> 5] = mb;
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int it = tid + k * 128;
    const int b = it >> 6, g = (it >> 2) & 15, t = it & 3;
    const unsigned mb = max(sm.wmax[2 * b], sm.wmax[2 * b + 1]);
    const int E = (int)((mb >> 23) & 255);
    int e = mb == 0 ? 0 : 141 - max(E, 1);
    e = min(max(e, -100), 126);
    const float sc = __int_as_float((e + 127) << 23);
    const float4 v = xv[k];
    const float v0 = v.x * sc, v1 = v.y * sc, v2 = v.z * sc, v3 = v.w * sc;
    const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1), h2 = __float2half_rn(v2),
                 h3 = __float2half_rn(v3);
    const uint32_t hi01 = pack_f16x2(__half2float(h0), __half2float(h1));
    const uint32_t hi23 = pack_f16x2(__half2float(h2), __half2float(h3));
    const uint32_t lo01 = pack_f16x2(v0 - __half2float(h0), v1 - __half2float(h1));
    const uint32_t lo23 = pack_f16x2(v2 - __half2float(h2), v3 - __half2float(h3));
    const int col = 2 * (b & 3);
    sm.frag[g][b >> 2][col * 4 + t] = make_uint2(hi01, hi23);
    sm.frag[g][b >> 2][(col + 1) * 4 + t] = make_uint2(lo01, lo23);
    if constexpr (TYPE == MQ_Q4_K) {
      // sum over the 8 consecutive items (32 elements) of sub-block g/2
      float ps = (v0 + v1) + (v2 + v3);
      ps += __shfl_xor_sync(0xffffffffu, ps, 1);
      ps += __shfl_xor_sync(0xffffffffu, ps, 2);
      ps += __shfl_xor_sync(0xffffffffu, ps, 4);
      if ((it & 7) == 0) sm.xsum[g >> 1][b] = ps;
    }
    if ((it & 63) == 0) sm.unscale[b] = __int_as_float((127 - e) << 23);
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int TYPE, int NT>
__global__ void __launch_bounds__(kThreads) matvec_kernel(const MvArgs p) {
  extern __shared__ uint8_t smem_raw[];
  MvSmem<TYPE, NT> &sm = *reinterpret_cast<MvSmem<TYPE, NT> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int rank = blockIdx.x % p.S;
  const int64_t group = blockIdx.x / p.S;
  const int c_begin = (int)((int64_t)rank * p.nchunk / p.S);
  const int c_end = (int)((int64_t)(rank + 1) * p.nchunk / p.S);
  const int nch = c_end - c_begin;

  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.full[s])), "r"(1));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.empty[s])), "r"(4));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  float tot[2][NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) tot[0][i] = tot[1][i] = 0.f;
  const int ra = 16 * warp + g;  // tile row of fragment row g (the other is ra + 8)
  const int64_t rA = group * 64 + ra, rB = rA + 8;
  const bool okA = rA < p.N, okB = rB < p.N;

  if (warp == 4) {  // ---- producer: weight tiles and x chunks into the ring
    if (lane == 0) {
      for (int i = 0; i < nch; ++i) {
        const int c = c_begin + i, s = i % kNS;
        const int cw = chunk_width(p.K, c);
        if (i >= kNS) mbar_wait(sa(&sm.empty[s]), ((i / kNS) - 1) & 1, p.status, 21);
        const int64_t tile = group * p.nchunk + c;
        uint32_t bytes = (uint32_t)(p.B * cw * 4);
        if constexpr (TYPE == MQ_Q4_K) bytes += 64 * 144;
        if constexpr (TYPE == MQ_Q6_K) bytes += 64 * 192 + 64 * 16 + 64 * 2;
        if constexpr (TYPE == MQ_Q8_0) bytes += 64 * cw + 64 * 16;
        const uint32_t bar = sa(&sm.full[s]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"(bytes)
                     : "memory");
        uint8_t *w = sm.w[s];
        if constexpr (TYPE == MQ_Q4_K) {
          bulk_1d(sa(w), p.q + tile * 64 * 144, 64 * 144, bar);
        } else if constexpr (TYPE == MQ_Q6_K) {
          bulk_1d(sa(w), p.q + tile * 64 * 192, 64 * 192, bar);
          bulk_1d(sa(w + 64 * 192), p.sc + tile * 64 * 16, 64 * 16, bar);
          bulk_1d(sa(w + 64 * 192 + 64 * 16), p.d + tile * 64, 64 * 2, bar);
        } else {
          bulk_1d(sa(w), p.q + (group * p.K + int64_t(c) * kChunk) * 64, (uint32_t)(64 * cw), bar);
          bulk_1d(sa(w + 64 * 256), p.d + tile * 64 * 8, 64 * 16, bar);
        }
        for (int b = 0; b < p.B; ++b)
          bulk_1d(sa(sm.x[s][b]), p.x + int64_t(b) * p.K + int64_t(c) * kChunk,
                  (uint32_t)(cw * 4), bar);
      }
    }
  } else {  // ---- compute warps
    float(*tab)[16] = sm.tab[warp];
    for (int i = 0; i < nch; ++i) {
      const int c = c_begin + i, s = i % kNS;
      const int cw = chunk_width(p.K, c);
      mbar_wait(sa(&sm.full[s]), (i / kNS) & 1, p.status, 22);
      stage_x<TYPE, NT>(sm, s, p.B, cw);
      WRegs<TYPE> cur;
      load_words<TYPE>(sm.w[s], cur, ra, t, cw / 32);
    float acc[2][NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[0][i] = acc[1][i] = 0.f;

    if constexpr (TYPE == MQ_Q4_K) {
      // decode 4 scales + 4 mins of row (t&1 ? g+8 : g), sub-blocks 4*(t>>1) .. +3
      {
        const uint4 h = cur.hdr;
        const float dd = __half2float(__ushort_as_half((unsigned short)(h.x & 0xffff)));
        const float dm = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
        uint32_t scw, mw;
        if (t >> 1) {
          scw = (h.w & 0x0f0f0f0fu) | ((h.y >> 2) & 0x30303030u);
          mw = ((h.w >> 4) & 0x0f0f0f0fu) | ((h.z >> 2) & 0x30303030u);
        } else {
          scw = h.y & 0x3f3f3f3fu;
          mw = h.z & 0x3f3f3f3fu;
        }
        const int rl = g + 8 * (t & 1), j0 = 4 * (t >> 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tab[rl][2 * (j0 + i)] = dd * 512.f * (float)((scw >> (8 * i)) & 255u);
          tab[rl][2 * (j0 + i) + 1] = dm * (float)((mw >> (8 * i)) & 255u);
        }
      }
      __syncwarp();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {  // sub-blocks 2cc (low nibbles), 2cc+1 (high)
        float clo[NT][4], chi[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
          for (int r = 0; r < 4; ++r) clo[i][r] = chi[i][r] = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t wa = cur.a[2 * cc + u], wb = cur.b[2 * cc + u];
          const uint32_t la = wa & 0x0f0f0f0fu, ha = (wa >> 4) & 0x0f0f0f0fu;
          const uint32_t lb = wb & 0x0f0f0f0fu, hb = (wb >> 4) & 0x0f0f0f0fu;
          const uint32_t la0 = e4m3x2_to_f16x2(la & 0xffff), la2 = e4m3x2_to_f16x2(la >> 16);
          const uint32_t lb0 = e4m3x2_to_f16x2(lb & 0xffff), lb2 = e4m3x2_to_f16x2(lb >> 16);
          const uint32_t ha0 = e4m3x2_to_f16x2(ha & 0xffff), ha2 = e4m3x2_to_f16x2(ha >> 16);
          const uint32_t hb0 = e4m3x2_to_f16x2(hb & 0xffff), hb2 = e4m3x2_to_f16x2(hb >> 16);
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            const uint2 bl = sm.frag[4 * cc + u][i][lane];      // group 2*(2cc) + u
            const uint2 bh = sm.frag[4 * cc + 2 + u][i][lane];  // group 2*(2cc+1) + u
            mma16816(clo[i], la0, lb0, la2, lb2, bl.x, bl.y);
            mma16816(chi[i], ha0, hb0, ha2, hb2, bh.x, bh.y);
          }
        }
        const int jl = 2 * cc, jh = 2 * cc + 1;
        const float sAl = tab[g][2 * jl], mAl = tab[g][2 * jl + 1];
        const float sBl = tab[g + 8][2 * jl], mBl = tab[g + 8][2 * jl + 1];
        const float sAh = tab[g][2 * jh], mAh = tab[g][2 * jh + 1];
        const float sBh = tab[g + 8][2 * jh], mBh = tab[g + 8][2 * jh + 1];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const float xl = sm.xsum[jl][t + 4 * i], xh = sm.xsum[jh][t + 4 * i];
          acc[0][i] = fmaf(sAl, clo[i][0] + clo[i][1], acc[0][i]);
          acc[1][i] = fmaf(sBl, clo[i][2] + clo[i][3], acc[1][i]);
          acc[0][i] = fmaf(-mAl, xl, acc[0][i]);
          acc[1][i] = fmaf(-mBl, xl, acc[1][i]);
          acc[0][i] = fmaf(sAh, chi[i][0] + chi[i][1], acc[0][i]);
          acc[1][i] = fmaf(sBh, chi[i][2] + chi[i][3], acc[1][i]);
          acc[0][i] = fmaf(-mAh, xh, acc[0][i]);
          acc[1][i] = fmaf(-mBh, xh, acc[1][i]);
        }
      }
    } else if constexpr (TYPE == MQ_Q6_K) {
      {
        const float dd = __half2float(__ushort_as_half(cur.dbits));
        const int rl = g + 8 * (t & 1), s0 = 8 * (t >> 1);
        const uint32_t w0 = cur.sc8.x, w1 = cur.sc8.y;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tab[rl][s0 + i] = dd * (float)(int8_t)((w0 >> (8 * i)) & 255u);
          tab[rl][s0 + 4 + i] = dd * (float)(int8_t)((w1 >> (8 * i)) & 255u);
        }
      }
      __syncwarp();
      const uint32_t magic = 0x64646464u;
      const uint32_t bias = 0x64206420u;  // f16x2 (1056, 1056)
#pragma unroll
      for (int hv = 0; hv < 4; ++hv) {  // (h, v) = (hv >> 1, hv & 1)
        const uint32_t qaA = cur.a[3 * hv], qbA = cur.a[3 * hv + 1], qhA = cur.a[3 * hv + 2];
        const uint32_t qaB = cur.b[3 * hv], qbB = cur.b[3 * hv + 1], qhB = cur.b[3 * hv + 2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          uint32_t loA, loB, hA, hB;
          if (r == 0) { loA = qaA & 0x0f0f0f0fu; loB = qaB & 0x0f0f0f0fu; hA = qhA << 4; hB = qhB << 4; }
          else if (r == 1) { loA = qbA & 0x0f0f0f0fu; loB = qbB & 0x0f0f0f0fu; hA = qhA << 2; hB = qhB << 2; }
          else if (r == 2) { loA = (qaA >> 4) & 0x0f0f0f0fu; loB = (qaB >> 4) & 0x0f0f0f0fu; hA = qhA; hB = qhB; }
          else { loA = (qbA >> 4) & 0x0f0f0f0fu; loB = (qbB >> 4) & 0x0f0f0f0fu; hA = qhA >> 2; hB = qhB >> 2; }
          const uint32_t qA = loA | (hA & 0x30303030u), qB = loB | (hB & 0x30303030u);
          const uint32_t a0 = hsub2(__byte_perm(qA, magic, 0x5140), bias);
          const uint32_t a2 = hsub2(__byte_perm(qA, magic, 0x5342), bias);
          const uint32_t a1 = hsub2(__byte_perm(qB, magic, 0x5140), bias);
          const uint32_t a3 = hsub2(__byte_perm(qB, magic, 0x5342), bias);
          const int sidx = 8 * (hv >> 1) + 2 * r + (hv & 1);
          const float sA = tab[g][sidx], sB = tab[g + 8][sidx];
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            float cacc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint2 bf = sm.frag[sidx][i][lane];
            mma16816(cacc, a0, a1, a2, a3, bf.x, bf.y);
            acc[0][i] = fmaf(sA, cacc[0] + cacc[1], acc[0][i]);
            acc[1][i] = fmaf(sB, cacc[2] + cacc[3], acc[1][i]);
          }
        }
      }
    } else {  // Q8_0
      const uint32_t magic = 0x64646464u;
      const uint32_t bias = 0x64806480u;  // f16x2 (1152, 1152)
#pragma unroll
      for (int blk = 0; blk < 8; ++blk) {
        float cacc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
          for (int r = 0; r < 4; ++r) cacc[i][r] = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t qA = cur.a[2 * blk + u] ^ 0x80808080u;
          const uint32_t qB = cur.b[2 * blk + u] ^ 0x80808080u;
          const uint32_t a0 = hsub2(__byte_perm(qA, magic, 0x5140), bias);
          const uint32_t a2 = hsub2(__byte_perm(qA, magic, 0x5342), bias);
          const uint32_t a1 = hsub2(__byte_perm(qB, magic, 0x5140), bias);
          const uint32_t a3 = hsub2(__byte_perm(qB, magic, 0x5342), bias);
#pragma unroll
          for (int i = 0; i < NT; ++i) {
            const uint2 bf = sm.frag[2 * blk + u][i][lane];
            mma16816(cacc[i], a0, a1, a2, a3, bf.x, bf.y);
          }
        }
        const float dA = __half2float(__ushort_as_half(cur.da[blk]));
        const float dB = __half2float(__ushort_as_half(cur.db[blk]));
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          acc[0][i] = fmaf(dA, cacc[i][0] + cacc[i][1], acc[0][i]);
          acc[1][i] = fmaf(dB, cacc[i][2] + cacc[i][3], acc[1][i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const float us = sm.unscale[t + 4 * i];
      tot[0][i] = fmaf(us, acc[0][i], tot[0][i]);
      tot[1][i] = fmaf(us, acc[1][i], tot[1][i]);
    }
      __syncwarp();
      if (lane == 0)  // this warp is done with stage s
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(&sm.empty[s])) : "memory");
    }
  }

  if (p.S == 1) {
    if (warp < 4) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int b = t + 4 * i;
        if (b < p.B) {
          if (okA) p.y[int64_t(b) * p.N + rA] = tot[0][i];
          if (okB) p.y[int64_t(b) * p.N + rB] = tot[1][i];
        }
      }
    }
    return;
  }
  // split-K over the cluster: rank 0 sums the ranks' partials in rank order
  if (warp < 4) {
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      sm.part[16 * warp + g][t + 4 * i] = tot[0][i];
      sm.part[16 * warp + g + 8][t + 4 * i] = tot[1][i];
    }
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (rank == 0 && warp < 4) {
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int b = t + 4 * i;
      float sA = 0.f, sB = 0.f;
      for (int r = 0; r < p.S; ++r) {
        float(*rp)[8] = cluster.map_shared_rank(sm.part, r);
        sA += rp[16 * warp + g][b];
        sB += rp[16 * warp + g + 8][b];
      }
      if (b < p.B) {
        if (okA) p.y[int64_t(b) * p.N + rA] = sA;
        if (okB) p.y[int64_t(b) * p.N + rB] = sB;
      }
    }
  }
  cluster.sync();
}

template <int TYPE, int NT>
constexpr size_t mv_smem_bytes() {
  return sizeof(MvSmem<TYPE, NT>) + 128;
}

template <int TYPE, int NT>
mq_status launch_one(const MvArgs &a, cudaStream_t s, const char *name) {
  const int64_t groups = (a.N + 63) / 64;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(groups * a.S), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = mv_smem_bytes<TYPE, NT>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.S > 1 ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, matvec_kernel<TYPE, NT>, a);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "launch of %s (grid %u, cluster %d) failed: %s", name,
                cfg.gridDim.x, a.S, cudaGetErrorName(e));
  return MQ_OK;
}

template <int TYPE, int NT>
mq_status optin_mv(const DeviceState *st, const char *name) {
  const size_t smem = mv_smem_bytes<TYPE, NT>();
  if ((int)smem > st->smem_optin)
    return fail(MQ_ERR_LAUNCH, "%s needs %zu bytes of shared memory; the device allows %d", name,
                smem, st->smem_optin);
  cudaError_t e = cudaFuncSetAttribute(matvec_kernel<TYPE, NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "smem opt-in of %s (%zu bytes) refused: %s", name, smem,
                cudaGetErrorName(e));
  return MQ_OK;
}

}  // namespace

mq_status init_matvec(DeviceState *st) {
  mq_status s;
  if ((s = optin_mv<MQ_Q8_0, 1>(st, "matvec_kernel<Q8_0,NT=1>")) != MQ_OK) return s;
  if ((s = optin_mv<MQ_Q8_0, 2>(st, "matvec_kernel<Q8_0,NT=2>")) != MQ_OK) return s;
  if ((s = optin_mv<MQ_Q4_K, 1>(st, "matvec_kernel<Q4_K,NT=1>")) != MQ_OK) return s;
  if ((s = optin_mv<MQ_Q4_K, 2>(st, "matvec_kernel<Q4_K,NT=2>")) != MQ_OK) return s;
  if ((s = optin_mv<MQ_Q6_K, 1>(st, "matvec_kernel<Q6_K,NT=1>")) != MQ_OK) return s;
  if ((s = optin_mv<MQ_Q6_K, 2>(st, "matvec_kernel<Q6_K,NT=2>")) != MQ_OK) return s;
  return MQ_OK;
}

// K-split heuristic: enough CTAs for two per SM.  Depends only on (N, K, type),
// never on B, so batched columns reproduce the B = 1 result bitwise.
static int choose_split(int64_t N, int64_t K, int sms, int rows_per_cta) {
  const int64_t groups = (N + rows_per_cta - 1) / rows_per_cta;
  const int nchunk = (int)((K + kChunk - 1) / kChunk);
  int64_t want = (2 * int64_t(sms) + groups - 1) / groups;
  int S = (int)(want < 8 ? want : 8);
  S = min(S, nchunk);
  return max(S, 1);
}

mq_status launch_matvec(const mq_weight *W, const float *x, float *y, int B, cudaStream_t s,
                        const DeviceState *st) {
  MvArgs a;
  a.q = W->q;
  a.sc = W->sc;
  a.d = W->d;
  a.x = x;
  a.y = y;
  a.N = W->N;
  a.K = W->K;
  a.B = B;
  a.nchunk = (int)((W->K + kChunk - 1) / kChunk);
  a.S = choose_split(W->N, W->K, st->sms, 64);
  a.status = st->status;
  const bool two = B > 4;
  switch (W->type) {
    case MQ_Q4_K:
      return two ? launch_one<MQ_Q4_K, 2>(a, s, "matvec_kernel<Q4_K,NT=2>")
                 : launch_one<MQ_Q4_K, 1>(a, s, "matvec_kernel<Q4_K,NT=1>");
    case MQ_Q6_K:
      return two ? launch_one<MQ_Q6_K, 2>(a, s, "matvec_kernel<Q6_K,NT=2>")
                 : launch_one<MQ_Q6_K, 1>(a, s, "matvec_kernel<Q6_K,NT=1>");
    default:
      return two ? launch_one<MQ_Q8_0, 2>(a, s, "matvec_kernel<Q8_0,NT=2>")
                 : launch_one<MQ_Q8_0, 1>(a, s, "matvec_kernel<Q8_0,NT=1>");
  }
}

}  // namespace mq
