// matvec.cu -- decode matvec y[b][n] = sum_k w[n][k] x[b][k] for GGUF Q4_0 / Q4_1 /
// Q5_0 / Q5_1 / Q8_0 / Q4_K / Q5_K / Q6_K weights and f32 activations, B <= 8
// ("minfer CUDA Backend Design" §4.4: the nt == 1 matvec and the _multi variants for
// nt 2..8).
//
// GB300 design.  The weights are streamed once from HBM and dequantised in
// registers straight into tensor-core fragments; the dot products run on the
// warp-level tensor path (mma.sync m16n8k16, f16 inputs, f32 accumulate), so the
// CUDA-core work per weight element is a fraction of an instruction and does
// not grow with the batch size B:
//
//  * weight side (A operand, 16 rows x 16 K per MMA): quants become exact f16
//    integers.  Q4_K: a nibble masked into the mantissa of 1024 (bits 0-3) or
//    1024/16-scaled (bits 4-7) is turned by one f16x2 fma into sc_j * nib, the
//    6-bit sub-block scale folded in exactly (sc_j * nib <= 945), so a whole
//    256-element super-block accumulates in the MMA and d is applied once.
//    Q6_K and Q8_0: a byte permute into an f16 whose exponent makes the low
//    mantissa byte the integer, then one f16x2 subtraction; the 16-element
//    (Q6_K) or 32-element (Q8_0) scale is applied to the f32 MMA result.
//  * Q4_K min term -dmin * sum_j m_j * sum(x over sub-block j): one more MMA per
//    super-block whose A operand holds the eight 6-bit mins m_j and whose B
//    operand holds the sub-block sums of x.
//  * activation side (B operand, 16 K x 8 columns): x is staged per 256-element
//    chunk as two f16 parts per batch row, hi = f16(x*2^e) and lo =
//    f16(x*2^e - hi), with 2^e a per-(row, chunk) power of two that puts max|x|
//    in [2^14, 2^15).  hi + lo carries 22 significant bits, so the product error
//    is ~2^-22 relative, far inside the 1e-4 * sum|w||x| bound.  Columns 2b and
//    2b+1 of an n8 tile hold hi and lo of batch row b, so one thread's two
//    accumulator columns are the two parts of the same row.
//
// The fragment rule: thread t (of a quad) holds the elements 4t..4t+3 of each
// 16-element group; A register pairs are (4t, 4t+1) and (4t+2, 4t+3), matched
// by B pairs (x[4t], x[4t+1]) and (x[4t+2], x[4t+3]).  The decode planes
// (repack.cu) store each thread's words contiguously.
//
// Data movement and roles.  A CTA owns one 128-row group of the decode plane
// and a K-slice, and runs 10 warps (11 in most kernels for three or more batch rows,
// see x_warps) around a shared-memory ring of chunk stages:
//  * the copy warp (one lane) streams, per 256-element chunk, the group's weight
//    tile (one contiguous run of the tiled decode plane) and the x chunk of every
//    batch row into the stage with 1-D bulk copies (cp.async.bulk, counted by the
//    stage's transaction barrier);
//  * the x warp (or two, each with half of the batch rows) turns the staged x
//    chunk into B fragments (and the sub-block sums for Q4_K) in a second,
//    smaller ring of fragment slots;
//  * eight compute warps, 16 rows each, wait for a weight stage, decode their
//    rows' scales into a warp-private table and copy their quant words into
//    registers, release the weight stage at once (so the next chunk's copy is
//    in flight during the MMAs), then wait for the fragment slot, run the MMAs
//    and release the slot.  They never wait for one another.
// Launches overlap: the kernel is launched with programmatic stream
// serialization and lets the next kernel in the stream launch as soon as all of
// its CTAs are running.  The weight tiles of the first ring stages are
// requested before griddepcontrol.wait (registered weights are never written
// by a kernel), x only after it, and y is written only after x has been read,
// so the tail of the previous kernel overlaps this kernel's first HBM traffic.
// When one wave would be short of CTAs, K is split over a thread-block cluster
// of S CTAs whose partial sums are reduced through distributed shared memory in
// rank order (deterministic, and independent of B, so every column of a batched
// call equals the B = 1 call bitwise).  All mbarrier waits are bounded.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "mv_device.cuh"

namespace cg = cooperative_groups;

namespace mq {
namespace {

using namespace mvd;

constexpr int kRows = kRowGroup;               // rows per CTA
constexpr int kMaxSplit = 16;                  // K slices: a cluster of up to 16 CTAs
constexpr int kCompute = kRows / 16;           // compute warps, 16 rows each
// x-fragment warps: one in the kernel for B <= 2; in the kernels for more batch rows two
// (x warp j converts rows [j * 2NT, (j + 1) * 2NT) of the chunk), except for Q6_K, whose
// single x warp converts all rows step by step over the rows (stage_x_rows); the bulk-copy
// warp comes last.  Measured at B = 4 / 8 against one row-by-row x warp: Q4_K 18944 x 3584
// 15.6 -> 13.8 / 22.0 -> 18.4 us, Q5_K 17.4 -> 15.9 / 25.2 -> 21.4 us, Q4_1 B = 8 26.4 ->
// 23.8 us, Q8_0 B = 8 22.7 -> 21.6 us; Q6_K 3584 x 18944 B = 8 took 23.9 us with two x warps
// (either form) and 23.3 us with the one row-batched warp.
template <int TYPE, bool XE>
__host__ __device__ constexpr int x_warps() {
  return XE && TYPE != MQ_Q6_K ? 2 : 1;
}
template <int TYPE, bool XE>
__host__ __device__ constexpr int copy_warp() {
  return kCompute + x_warps<TYPE, XE>();
}
template <int TYPE, bool XE>
__host__ __device__ constexpr int mv_threads() {
  return 32 * (kCompute + 1 + x_warps<TYPE, XE>());
}

struct MvArgs {
  const uint8_t *q;
  const uint16_t *d;
  const uint16_t *dm;  // Q4_1 / Q5_1 block m
  const uint32_t *qh;  // Q5_0 / Q5_1 fifth-bit words
  const float *x;
  float *y;
  int64_t N, K;
  int B;
  int nchunk;  // ceil(K / 256)
  int S;       // K slices (cluster size)
  int swiglu;  // fused gate/up weight: y[b][n] = silu(gate row) * (its up row), N / 2 wide
  int *status;
};

// The per-32-element-block types, those among them with an additive min m (w = d*q + m),
// and those with a fifth bit per element.
template <int TYPE>
__host__ __device__ constexpr bool q32_type() {
  return TYPE == MQ_Q8_0 || TYPE == MQ_Q4_0 || TYPE == MQ_Q4_1 || TYPE == MQ_Q5_0 ||
         TYPE == MQ_Q5_1;
}
template <int TYPE>
__host__ __device__ constexpr bool addmin_type() {
  return TYPE == MQ_Q4_1 || TYPE == MQ_Q5_1;
}
template <int TYPE>
__host__ __device__ constexpr bool fifth_type() {
  return TYPE == MQ_Q5_0 || TYPE == MQ_Q5_1;
}
// Bytes per 32-element block and tile row of the per-32-block types' quant plane.
template <int TYPE>
__host__ __device__ constexpr int q32_bytes() {
  return TYPE == MQ_Q8_0 ? 32 : 16;
}
// Stage layout of the per-32-block types: quants [8 blocks][128 rows][q32_bytes], then
// the f16 d [128 rows][8 blocks], then (additive-min types) m as d, then (fifth-bit
// types) the fifth-bit words [8 blocks][128 rows].
template <int TYPE>
__host__ __device__ constexpr int q32_off_d() {
  return kRows * 8 * q32_bytes<TYPE>();
}
template <int TYPE>
__host__ __device__ constexpr int q32_off_m() {
  return q32_off_d<TYPE>() + kRows * 16;
}
template <int TYPE>
__host__ __device__ constexpr int q32_off_h() {
  return q32_off_d<TYPE>() + kRows * 16 * (addmin_type<TYPE>() ? 2 : 1);
}
// Unquantised f16 / bf16 weights.
template <int TYPE>
__host__ __device__ constexpr bool float_w() {
  return TYPE == MQ_F16 || TYPE == MQ_BF16;
}
// Bytes of one (128-row group, chunk) tile of the decode plane.
template <int TYPE>
__host__ __device__ constexpr int tile_bytes() {
  return float_w<TYPE>()   ? kRows * kChunk * 2
         : TYPE == MQ_Q4_K ? kRows * 144
         : TYPE == MQ_Q5_K ? kRows * 176
         : TYPE == MQ_Q6_K ? kRows * 210
                           : q32_off_h<TYPE>() + (fifth_type<TYPE>() ? kRows * 32 : 0);
}
// Weight-ring depth: two CTAs per SM must fit in shared memory (checked at each launch
// site for the quantised types; the f16 / bf16 tiles take one CTA per SM); within that,
// the depth that measured fastest (Q4_K B <= 4: 2 stages beat 3 and 4; a third stage for
// the Q4_K / Q5_K two-tile kernel left one CTA per SM and doubled its time; Q6_K 3584 x
// 18944 in clusters of 10, B = 1..4: 2 stages 1.5-2% faster than 3).
template <int TYPE, int NT>
__host__ __device__ constexpr int ring_stages() {
  return 2;
}
// Fragment-ring depth.
template <int TYPE>
__host__ __device__ constexpr int frag_slots() {
  return (TYPE == MQ_Q4_K || TYPE == MQ_Q5_K) ? 3 : 2;
}
// The super-block types with a sub-block min term (their x warp also stages sub-block sums).
template <int TYPE>
__host__ __device__ constexpr bool kmin_type() {
  return TYPE == MQ_Q4_K || TYPE == MQ_Q5_K;
}
// Per-warp tables decoded from the tile headers of the warp's 16 rows.
template <int TYPE>
struct WarpTab;
template <>
struct WarpTab<MQ_Q4_K> {
  uint4 sc[4][2][8];  // [pair c'][lo, hi sub-block][g]: f16x2 (mul A, add A, mul B, add B)
  uint2 mf[4][8];     // [t][g]: min-term A fragment words of rows g, g+8
  float4 dd[8];       // [g]: d_A, 32*dmin_A, d_B, 32*dmin_B
};
template <>
struct WarpTab<MQ_Q6_K> {
  float2 s[16][8];  // [16-element group][g]: d*sc of rows g, g+8
};
template <>
struct WarpTab<MQ_Q8_0> {
  float2 s[8][8];  // [32-element block][g]: d of rows g, g+8
};
template <>
struct WarpTab<MQ_Q4_0> : WarpTab<MQ_Q8_0> {};
template <>
struct WarpTab<MQ_Q5_0> : WarpTab<MQ_Q8_0> {};
template <>
struct WarpTab<MQ_Q4_1> {
  float2 s[8][8];  // [32-element block][g]: d of rows g, g+8
  float2 m[8][8];  // the blocks' m
};
template <>
struct WarpTab<MQ_Q5_1> : WarpTab<MQ_Q4_1> {};
template <>
struct WarpTab<MQ_F16> {
  float unused;  // no scales: the weights are the f16 operand itself
};
template <>
struct WarpTab<MQ_BF16> : WarpTab<MQ_F16> {};
template <>
struct WarpTab<MQ_Q5_K> : WarpTab<MQ_Q4_K> {};

template <int TYPE, int NT>
struct MvSmem {
  static constexpr int NS = ring_stages<TYPE, NT>();
  static constexpr int FS = frag_slots<TYPE>();
  static constexpr int FG = kmin_type<TYPE>() ? 17 : 16;  // 16 groups (+ the min group)
  union {
    alignas(128) uint8_t w[NS][tile_bytes<TYPE>()];  // weight tiles
    float part[kRows][8];  // split-K partial sums (after the ring has drained)
  };
  alignas(128) float xr[NS][4 * NT][kChunk];  // staged x chunks of the batch rows
  // B fragments.  Each group is padded by 8 words (4 uint2 after its one n8 tile, or 2
  // after each of two) so that consecutive groups start 8 banks apart: an x-warp fragment
  // store (8 groups x 4 lanes) then takes 2 wavefronts instead of 8.  Measured 0.7-2.4%
  // faster (Q4_K 18944 x 3584 B = 1 / 4 / 8, Q6_K 3584 x 18944 B = 4, Q8_0 B = 8).
  alignas(16) uint2 frag[FS][FG][NT][32 + (NT == 1 ? 4 : 2)];
  float unscale[FS][8];                       // 2^-e per batch row of the slot's chunk
  WarpTab<TYPE> tab[kCompute];
  float xs[4 * NT][8];  // x-warp scratch: sub-block sums of each batch row
  float xb[addmin_type<TYPE>() ? FS : 1][8][8];  // per slot: [block][batch row] sums of x
  // weight stage: copied (wfull) / read into registers by all warps (wempty);
  // fragment slot: written (ffull) / used by the compute warps (fempty)
  uint64_t wfull[NS], wempty[NS], ffull[FS], fempty[FS];
};

// ---------------------------------------------------------------------------
// Copy warp (one lane): weight tile and x rows of each chunk into its stage.
template <int TYPE, int NT>
__device__ __forceinline__ void issue_copies(MvSmem<TYPE, NT> &sm, const MvArgs &p,
                                             int64_t group, int c_begin, int nch) {
  constexpr int NS = MvSmem<TYPE, NT>::NS;
  auto weights = [&](int i) {
    const int c = c_begin + i, s = i % NS;
    const int cw = chunk_width(p.K, c);
    const uint32_t bar = sa(&sm.wfull[s]);
    constexpr bool Q32 = q32_type<TYPE>();  // per-32-block scales
    constexpr int QB = q32_bytes<TYPE>();  // quant bytes per block row
    constexpr int HB = fifth_type<TYPE>() ? 4 : 0, MB = addmin_type<TYPE>() ? 16 : 0;
    const uint32_t wbytes = Q32            ? (uint32_t)(kRows * (cw / 32) * (QB + HB) + kRows * (16 + MB))
                            : float_w<TYPE>() ? (uint32_t)(kRows * cw * 2)
                                              : (uint32_t)tile_bytes<TYPE>();
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(wbytes + (uint32_t)(p.B * cw * 4))
                 : "memory");
    uint8_t *w = sm.w[s];
    if constexpr (Q32) {
      bulk_1d(sa(w), p.q + (group * (p.K / 32) + int64_t(c) * 8) * kRows * QB,
              (uint32_t)(kRows * (cw / 32) * QB), bar);
      bulk_1d(sa(w + q32_off_d<TYPE>()), p.d + (group * p.nchunk + c) * kRows * 8, kRows * 16,
              bar);
      if constexpr (addmin_type<TYPE>())
        bulk_1d(sa(w + q32_off_m<TYPE>()), p.dm + (group * p.nchunk + c) * kRows * 8, kRows * 16,
                bar);
      if constexpr (fifth_type<TYPE>())
        bulk_1d(sa(w + q32_off_h<TYPE>()), p.qh + (group * (p.K / 32) + int64_t(c) * 8) * kRows,
                (uint32_t)(kRows * (cw / 32) * 4), bar);
    } else if constexpr (float_w<TYPE>()) {  // a partial last chunk is a shorter run
      bulk_1d(sa(w), p.q + (group * p.K + int64_t(c) * kChunk) * kRows * 2, wbytes, bar);
    } else {
      bulk_1d(sa(w), p.q + (group * p.nchunk + c) * int64_t(tile_bytes<TYPE>()),
              (uint32_t)tile_bytes<TYPE>(), bar);
    }
  };
  auto xrows = [&](int i) {
    const int c = c_begin + i, s = i % NS;
    const int cw = chunk_width(p.K, c);
    for (int b = 0; b < p.B; ++b)
      bulk_1d(sa(sm.xr[s][b]), p.x + int64_t(b) * p.K + int64_t(c) * kChunk, (uint32_t)(cw * 4),
              sa(&sm.wfull[s]));
  };
  const int pre = nch < NS ? nch : NS;
  for (int i = 0; i < pre; ++i) weights(i);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
  for (int i = 0; i < pre; ++i) xrows(i);
  for (int i = pre; i < nch; ++i) {
    mbar_wait(sa(&sm.wempty[i % NS]), ((i / NS) - 1) & 1, p.status, 21);
    weights(i);
    xrows(i);
  }
}

// x warp of the Q6_K kernels for three or more batch rows: the chunk's rows are read into
// registers and the weight stage is released first; then each step runs over all rows of
// the kernel's tiles before the next (row maxima; scaled hi/lo parts, fragments and sums;
// min-term fragments), so the rows' dependency chains (warp reductions, shuffles) overlap
// instead of running one row after another.  Rows beyond B are computed on zeros and not
// stored.  Per row the arithmetic is that of stage_x below, so the fragments are the same.
// With one x warp, measured per type at B = 8: Q6_K 3584 x 18944 25.1 -> 23.3 us; Q8_0 and
// Q4_1 2% slower, Q4_0, Q5_0 level, Q4_K and Q5_K 1-9% slower (their min-term sums).  The
// other types take two row-by-row x warps instead.  The function is written for every type.
template <int TYPE, int NT, int XI>
__device__ __forceinline__ void stage_x_rows(MvSmem<TYPE, NT> &sm, const MvArgs &p,
                                             int c_begin, int nch, int lane) {
  constexpr int NS = MvSmem<TYPE, NT>::NS, FS = MvSmem<TYPE, NT>::FS;
  constexpr int R = 4 * NT / x_warps<TYPE, true>(), R0 = XI * R;  // rows R0 .. R0 + R - 1
  for (int i = 0; i < nch; ++i) {
    const int c = c_begin + i, s = i % NS, fs = i % FS;
    const int cw = chunk_width(p.K, c);
    mbar_wait(sa(&sm.wfull[s]), (i / NS) & 1, p.status, 23);
    // lane handles float4 items f = lane and lane + 32 of each batch row
    float4 xv[R][2];
#pragma unroll
    for (int b = 0; b < R; ++b)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k;
        xv[b][k] = R0 + b < p.B && 4 * f < cw
                       ? *reinterpret_cast<const float4 *>(&sm.xr[s][R0 + b][4 * f])
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(sa(&sm.wempty[s]));  // done reading the staged x
    if (i >= FS) mbar_wait(sa(&sm.fempty[fs]), ((i / FS) - 1) & 1, p.status, 25);
    float scale[R];
#pragma unroll
    for (int b = 0; b < R; ++b) {
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(xv[b][k].x), fabsf(xv[b][k].y)),
                           fmaxf(fabsf(xv[b][k].z), fabsf(xv[b][k].w))));
      const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      const int E = (int)((mb >> 23) & 255);
      int e = mb == 0 ? 0 : 141 - max(E, 1);
      e = min(max(e, -100), 126);
      scale[b] = __int_as_float((e + 127) << 23);
      if (lane == 0 && R0 + b < p.B) sm.unscale[fs][R0 + b] = __int_as_float((127 - e) << 23);
    }
#pragma unroll
    for (int bl = 0; bl < R; ++bl) {
      const int b = R0 + bl;  // batch row
      const int col = 2 * (b & 3);
      const bool live = b < p.B;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k, g16 = f >> 2, t = f & 3;
        const float v0 = xv[bl][k].x * scale[bl], v1 = xv[bl][k].y * scale[bl],
                    v2 = xv[bl][k].z * scale[bl], v3 = xv[bl][k].w * scale[bl];
        uint32_t hi01, hi23, lo01, lo23;
        if constexpr (TYPE == MQ_BF16) {  // bf16 parts: 16 significant bits of x
          hi01 = pack_bf16x2(v0, v1);
          hi23 = pack_bf16x2(v2, v3);
          lo01 = pack_bf16x2(v0 - bf16_lo(hi01), v1 - bf16_hi(hi01));
          lo23 = pack_bf16x2(v2 - bf16_lo(hi23), v3 - bf16_hi(hi23));
        } else {
          hi01 = pack_f16x2(v0, v1);
          hi23 = pack_f16x2(v2, v3);
          lo01 = pack_f16x2(v0 - f16_lo(hi01), v1 - f16_hi(hi01));
          lo23 = pack_f16x2(v2 - f16_lo(hi23), v3 - f16_hi(hi23));
        }
        if (live) {
          sm.frag[fs][g16][b >> 2][col * 4 + t] = make_uint2(hi01, hi23);
          sm.frag[fs][g16][b >> 2][(col + 1) * 4 + t] = make_uint2(lo01, lo23);
        }
        if constexpr (addmin_type<TYPE>() || kmin_type<TYPE>()) {
          // sum of the 8 consecutive items of block / sub-block f >> 3, in f32
          float ps = (v0 + v1) + (v2 + v3);
          ps += __shfl_xor_sync(0xffffffffu, ps, 1);
          ps += __shfl_xor_sync(0xffffffffu, ps, 2);
          ps += __shfl_xor_sync(0xffffffffu, ps, 4);
          if (live && (lane & 7) == 0) {
            if constexpr (addmin_type<TYPE>())
              sm.xb[fs][f >> 3][b] = ps;
            else  // scaled by 1/32 so that |sum| < 2^15 fits f16
              sm.xs[b][f >> 3] = ps * 0.03125f;
          }
        }
      }
    }
    if constexpr (kmin_type<TYPE>()) {
      // min-term B fragments: lane (col', t') of row b holds sums 2t', 2t'+1 (hi or lo part)
      __syncwarp();
      if (lane < 8) {
        const int part = lane >> 2, t = lane & 3;
#pragma unroll
        for (int b = R0; b < R0 + R; ++b) {
          if (b < p.B) {
            const float s0 = sm.xs[b][2 * t], s1 = sm.xs[b][2 * t + 1];
            const uint32_t h = pack_f16x2(s0, s1);
            const uint32_t word = part == 0 ? h : pack_f16x2(s0 - f16_lo(h), s1 - f16_hi(h));
            sm.frag[fs][16][b >> 2][(2 * (b & 3) + part) * 4 + t] = make_uint2(word, 0u);
          }
        }
      }
      __syncwarp();
    }
    mbar_arrive(sa(&sm.ffull[fs]));  // each lane, after its own fragment stores
  }
}

// x warp: staged x chunk -> hi/lo B fragments (+ the Q4_K / Q5_K sub-block sums, the
// Q4_1 / Q5_1 block sums).  XE: the chunk's x goes to registers first and the weight stage
// is released before the conversion (the copy warp refills it meanwhile), which pays from
// three batch rows on; otherwise the stage is released after the conversion.
template <int TYPE, int NT, bool XE, int XI>
__device__ __forceinline__ void stage_x(MvSmem<TYPE, NT> &sm, const MvArgs &p, int c_begin,
                                        int nch, int lane) {
  constexpr int NS = MvSmem<TYPE, NT>::NS, FS = MvSmem<TYPE, NT>::FS;
  constexpr int R = 4 * NT / x_warps<TYPE, XE>(), R0 = XI * R;  // rows R0 .. R0 + R - 1
  for (int i = 0; i < nch; ++i) {
    const int c = c_begin + i, s = i % NS, fs = i % FS;
    const int cw = chunk_width(p.K, c);
    mbar_wait(sa(&sm.wfull[s]), (i / NS) & 1, p.status, 23);
    // lane handles float4 items f = lane and lane + 32 of each batch row
    constexpr bool early = XE;
    float4 xv[R][2];
    if (early) {
#pragma unroll
      for (int bl = 0; bl < R; ++bl)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int f = lane + 32 * k;
          xv[bl][k] = R0 + bl < p.B && 4 * f < cw
                          ? *reinterpret_cast<const float4 *>(&sm.xr[s][R0 + bl][4 * f])
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(sa(&sm.wempty[s]));  // done reading the staged x
    }
    if (i >= FS) mbar_wait(sa(&sm.fempty[fs]), ((i / FS) - 1) & 1, p.status, 25);
#pragma unroll
    for (int bl = 0; bl < R; ++bl) {
      const int b = R0 + bl;  // batch row
      if (b >= p.B) break;
      float4 v[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k;
        v[k] = early ? xv[bl][k]
                     : (4 * f < cw ? *reinterpret_cast<const float4 *>(&sm.xr[s][b][4 * f])
                                   : make_float4(0.f, 0.f, 0.f, 0.f));
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
      if (lane == 0) sm.unscale[fs][b] = __int_as_float((127 - e) << 23);
      const int col = 2 * (b & 3);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k, g16 = f >> 2, t = f & 3;
        const float v0 = v[k].x * scale, v1 = v[k].y * scale, v2 = v[k].z * scale,
                    v3 = v[k].w * scale;
        uint32_t hi01, hi23, lo01, lo23;
        if constexpr (TYPE == MQ_BF16) {  // bf16 parts: 16 significant bits of x
          hi01 = pack_bf16x2(v0, v1);
          hi23 = pack_bf16x2(v2, v3);
          lo01 = pack_bf16x2(v0 - bf16_lo(hi01), v1 - bf16_hi(hi01));
          lo23 = pack_bf16x2(v2 - bf16_lo(hi23), v3 - bf16_hi(hi23));
        } else {
          hi01 = pack_f16x2(v0, v1);
          hi23 = pack_f16x2(v2, v3);
          lo01 = pack_f16x2(v0 - f16_lo(hi01), v1 - f16_hi(hi01));
          lo23 = pack_f16x2(v2 - f16_lo(hi23), v3 - f16_hi(hi23));
        }
        sm.frag[fs][g16][b >> 2][col * 4 + t] = make_uint2(hi01, hi23);
        sm.frag[fs][g16][b >> 2][(col + 1) * 4 + t] = make_uint2(lo01, lo23);
        if constexpr (addmin_type<TYPE>()) {
          // block f >> 3 (8 consecutive items) sum of the scaled x, in f32
          float ps = (v0 + v1) + (v2 + v3);
          ps += __shfl_xor_sync(0xffffffffu, ps, 1);
          ps += __shfl_xor_sync(0xffffffffu, ps, 2);
          ps += __shfl_xor_sync(0xffffffffu, ps, 4);
          if ((lane & 7) == 0) sm.xb[fs][f >> 3][b] = ps;
        }
        if constexpr (kmin_type<TYPE>()) {
          // sum of sub-block j = f >> 3 (8 consecutive items), scaled by 1/32 so
          // that |sum| < 2^15 fits f16
          float ps = (v0 + v1) + (v2 + v3);
          ps += __shfl_xor_sync(0xffffffffu, ps, 1);
          ps += __shfl_xor_sync(0xffffffffu, ps, 2);
          ps += __shfl_xor_sync(0xffffffffu, ps, 4);
          if ((lane & 7) == 0) sm.xs[b][f >> 3] = ps * 0.03125f;
        }
      }
      if constexpr (kmin_type<TYPE>()) {
        // min-term B fragment: lane (col', t') holds sums 2t', 2t'+1 (hi or lo part)
        __syncwarp();
        if (lane < 8) {
          const int part = lane >> 2, t = lane & 3;
          const float s0 = sm.xs[b][2 * t], s1 = sm.xs[b][2 * t + 1];
          const uint32_t h = pack_f16x2(s0, s1);
          const uint32_t word = part == 0 ? h : pack_f16x2(s0 - f16_lo(h), s1 - f16_hi(h));
          sm.frag[fs][16][b >> 2][(col + part) * 4 + t] = make_uint2(word, 0u);
        }
        __syncwarp();
      }
    }
    mbar_arrive(sa(&sm.ffull[fs]));  // each lane, after its own fragment stores
    if (!early) {
      __syncwarp();
      if (lane == 0) mbar_arrive(sa(&sm.wempty[s]));  // done reading the staged x
    }
  }
}

// ---------------------------------------------------------------------------
// Compute warps.  After a warp has read its scales and quant words out of a
// weight stage it releases the stage, then waits for the fragment slot.
__device__ __forceinline__ void release_and_wait(uint64_t &wempty, uint64_t &ffull,
                                                 uint32_t fpar, int lane, int *status) {
  __syncwarp();
  if (lane == 0) mbar_arrive(sa(&wempty));
  mbar_wait(sa(&ffull), fpar, status, 24);
}

// ---------------------------------------------------------------------------
// Compute warps.  Thread (g, t) of warp w covers tile rows ra = 16w + g and
// rb = ra + 8; tot[0/1][i] accumulates rows ra/rb for batch row 4i + t.

// Q4_K and Q5_K (rows of RS = 144 / 176 bytes; Q5_K's fifth bits follow the quants).
// For Q5_K the fifth bit of each element goes to bit 4 (low-nibble path: 1024 + q) or
// bit 8 (high-nibble path: 1024 + 16q) of its f16 half before the magic exponent is
// OR-ed in, so q in [0, 31] takes the same exact multiply-add by sc (or sc/16): sc*q is
// at most 63*31 = 1953 < 2048, exact in f16.
template <int TYPE, int NT>
__device__ __forceinline__ void compute_chunk_q4k(MvSmem<TYPE, NT> &sm, int s, int fs,
                                                  uint32_t fpar, int warp, int lane, int *status,
                                                  const int (&fl)[NT], float (&tot)[2][NT]) {
  constexpr bool Q5 = TYPE == MQ_Q5_K;
  constexpr int RS = Q5 ? 176 : 144;
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *tile = sm.w[s];
  WarpTab<MQ_Q4_K> &tb = sm.tab[warp];
  {  // lane c'*8 + r decodes sub-blocks 2c', 2c'+1 of rows r and r+8 (entry = lane)
    const int cp = lane >> 3, r = lane & 7;
    const uint4 ha = *reinterpret_cast<const uint4 *>(tile + (16 * warp + r) * RS);
    const uint4 hb = *reinterpret_cast<const uint4 *>(tile + (16 * warp + r + 8) * RS);
    // 6-bit scales / mins of sub-blocks 4q..4q+3 as bytes (q = cp >> 1)
    uint32_t sa4, sb4, ma4, mb4;
    if (cp < 2) {
      sa4 = ha.y & 0x3f3f3f3fu;
      sb4 = hb.y & 0x3f3f3f3fu;
      ma4 = ha.z & 0x3f3f3f3fu;
      mb4 = hb.z & 0x3f3f3f3fu;
    } else {
      sa4 = (ha.w & 0x0f0f0f0fu) | ((ha.y >> 2) & 0x30303030u);
      sb4 = (hb.w & 0x0f0f0f0fu) | ((hb.y >> 2) & 0x30303030u);
      ma4 = ((ha.w >> 4) & 0x0f0f0f0fu) | ((ha.z >> 2) & 0x30303030u);
      mb4 = ((hb.w >> 4) & 0x0f0f0f0fu) | ((hb.z >> 2) & 0x30303030u);
    }
    // bytes 2(cp&1), 2(cp&1)+1 of each -> f16x2 integers (1024 + v) - 1024
    const uint32_t sel = (cp & 1) ? 0x5342u : 0x5140u, k1024 = 0x64006400u;
    const uint32_t scA = hsub2(__byte_perm(sa4, 0x64646464u, sel), k1024);
    const uint32_t scB = hsub2(__byte_perm(sb4, 0x64646464u, sel), k1024);
    // lo sub-block 2c' multiplies (1024 + n) by sc; hi sub-block 2c'+1 multiplies
    // (1024 + 16n) by sc/16; the addend is -1024 times the multiplier in both
    const uint32_t loA = __byte_perm(scA, scA, 0x1010), loB = __byte_perm(scB, scB, 0x1010);
    const uint32_t hiA = hmul2(__byte_perm(scA, scA, 0x3232), 0x2C002C00u);
    const uint32_t hiB = hmul2(__byte_perm(scB, scB, 0x3232), 0x2C002C00u);
    constexpr uint32_t kNeg1024 = 0xE400E400u;
    tb.sc[cp][0][r] = make_uint4(loA, hmul2(loA, kNeg1024), loB, hmul2(loB, kNeg1024));
    tb.sc[cp][1][r] = make_uint4(hiA, hmul2(hiA, kNeg1024), hiB, hmul2(hiB, kNeg1024));
    tb.mf[cp][r] = make_uint2(hsub2(__byte_perm(ma4, 0x64646464u, sel), k1024),
                              hsub2(__byte_perm(mb4, 0x64646464u, sel), k1024));
    if (cp == 0)
      tb.dd[r] = make_float4(f16_lo(ha.x), 32.f * f16_hi(ha.x), f16_lo(hb.x), 32.f * f16_hi(hb.x));
  }
  __syncwarp();
  const int ra = 16 * warp + g, rb = ra + 8;
  const uint4 a0 = *reinterpret_cast<const uint4 *>(tile + ra * RS + 16 + 32 * t);
  const uint4 a1 = *reinterpret_cast<const uint4 *>(tile + ra * RS + 32 + 32 * t);
  const uint4 b0 = *reinterpret_cast<const uint4 *>(tile + rb * RS + 16 + 32 * t);
  const uint4 b1 = *reinterpret_cast<const uint4 *>(tile + rb * RS + 32 + 32 * t);
  const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  uint2 qha = make_uint2(0u, 0u), qhb = make_uint2(0u, 0u);  // Q5_K fifth-bit words (u = 0, 1)
  if constexpr (Q5) {
    qha = *reinterpret_cast<const uint2 *>(tile + ra * RS + 144 + 8 * t);
    qhb = *reinterpret_cast<const uint2 *>(tile + rb * RS + 144 + 8 * t);
  }
  release_and_wait(sm.wempty[s], sm.ffull[fs], fpar, lane, status);
  // min term first: its MMA latency hides under the main loop
  float cm[NT][4];
  {
    const uint2 mf = tb.mf[t][g];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const uint2 bm = sm.frag[fs][16][i][fl[i]];
      cm[i][0] = cm[i][1] = cm[i][2] = cm[i][3] = 0.f;
      mma16816(cm[i], mf.x, mf.y, 0u, 0u, bm.x, bm.y);
    }
  }
  float acc[2][NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[0][i][r] = acc[1][i][r] = 0.f;
  // nibble n of bits 0-3 (kLo) or 4-7 (kHi) of each half -> f16 1024 + n or 1024 + 16n
  constexpr uint32_t kMagic = 0x64006400u, kLo = 0x000f000fu, kHi = 0x00f000f0u;
#pragma unroll
  for (int cp = 0; cp < 4; ++cp) {
    const uint4 slo = tb.sc[cp][0][g], shi = tb.sc[cp][1][g];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t xa = wa[2 * cp + u], xb = wb[2 * cp + u];
      const uint32_t xa8 = xa >> 8, xb8 = xb >> 8;
      // the OR-ed exponent word of each register: the magic, plus the fifth bits for Q5_K
      // (bit 2c' of bytes 0/2 or 1/3 of the fifth-bit word for the low nibbles, bit
      // 2c' + 1 for the high nibbles)
      uint32_t mla = kMagic, mlb = kMagic, mla8 = kMagic, mlb8 = kMagic;
      uint32_t mha = kMagic, mhb = kMagic, mha8 = kMagic, mhb8 = kMagic;
      if constexpr (Q5) {
        constexpr uint32_t kB4 = 0x00100010u, kB8 = 0x01000100u;
        const uint32_t qa = u ? qha.y : qha.x, qb = u ? qhb.y : qhb.x;
        mla = and_or(shl(qa, 4 - 2 * cp), kB4, kMagic);
        mlb = and_or(shl(qb, 4 - 2 * cp), kB4, kMagic);
        mla8 = and_or(shl(qa, -4 - 2 * cp), kB4, kMagic);
        mlb8 = and_or(shl(qb, -4 - 2 * cp), kB4, kMagic);
        mha = and_or(shl(qa, 7 - 2 * cp), kB8, kMagic);
        mhb = and_or(shl(qb, 7 - 2 * cp), kB8, kMagic);
        mha8 = and_or(shl(qa, -1 - 2 * cp), kB8, kMagic);
        mhb8 = and_or(shl(qb, -1 - 2 * cp), kB8, kMagic);
      }
      const uint32_t l0 = hfma2(and_or(xa, kLo, mla), slo.x, slo.y);
      const uint32_t l1 = hfma2(and_or(xb, kLo, mlb), slo.z, slo.w);
      const uint32_t l2 = hfma2(and_or(xa8, kLo, mla8), slo.x, slo.y);
      const uint32_t l3 = hfma2(and_or(xb8, kLo, mlb8), slo.z, slo.w);
      const uint32_t h0 = hfma2(and_or(xa, kHi, mha), shi.x, shi.y);
      const uint32_t h1 = hfma2(and_or(xb, kHi, mhb), shi.z, shi.w);
      const uint32_t h2 = hfma2(and_or(xa8, kHi, mha8), shi.x, shi.y);
      const uint32_t h3 = hfma2(and_or(xb8, kHi, mhb8), shi.z, shi.w);
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint2 bl = sm.frag[fs][4 * cp + u][i][fl[i]];      // sub-block 2c', K half u
        const uint2 bh = sm.frag[fs][4 * cp + 2 + u][i][fl[i]];  // sub-block 2c'+1
        mma16816(acc[0][i], l0, l1, l2, l3, bl.x, bl.y);
        mma16816(acc[1][i], h0, h1, h2, h3, bh.x, bh.y);
      }
    }
  }
  const float4 dd = tb.dd[g];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float us = sm.unscale[fs][4 * i + t];
    const float yA = dd.x * ((acc[0][i][0] + acc[0][i][1]) + (acc[1][i][0] + acc[1][i][1])) -
                     dd.y * (cm[i][0] + cm[i][1]);
    const float yB = dd.z * ((acc[0][i][2] + acc[0][i][3]) + (acc[1][i][2] + acc[1][i][3])) -
                     dd.w * (cm[i][2] + cm[i][3]);
    tot[0][i] = fmaf(us, yA, tot[0][i]);
    tot[1][i] = fmaf(us, yB, tot[1][i]);
  }
}

template <int NT>
__device__ __forceinline__ void compute_chunk_q6k(MvSmem<MQ_Q6_K, NT> &sm, int s, int fs,
                                                  uint32_t fpar, int warp, int lane, int *status,
                                                  const int (&fl)[NT], float (&tot)[2][NT]) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *tile = sm.w[s];
  WarpTab<MQ_Q6_K> &tb = sm.tab[warp];
  {  // lane (r, h): groups 8h..8h+7 of row r
    const int r = lane & 15, h = lane >> 4, row = 16 * warp + r;
    const uint2 scv = *reinterpret_cast<const uint2 *>(tile + kRows * 192 + row * 16 + 8 * h);
    const float dv =
        __half2float(*reinterpret_cast<const __half *>(tile + kRows * 208 + row * 2));
    float *dst = reinterpret_cast<float *>(&tb.s[8 * h][r & 7]) + (r >> 3);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      dst[k * 16] = dv * (float)(int8_t)((scv.x >> (8 * k)) & 255u);
      dst[(4 + k) * 16] = dv * (float)(int8_t)((scv.y >> (8 * k)) & 255u);
    }
  }
  __syncwarp();
  const int ra = 16 * warp + g, rb = ra + 8;
  uint32_t wa[12], wb[12];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint4 va = *reinterpret_cast<const uint4 *>(tile + ra * 192 + 48 * t + 16 * i);
    const uint4 vb = *reinterpret_cast<const uint4 *>(tile + rb * 192 + 48 * t + 16 * i);
    wa[4 * i] = va.x; wa[4 * i + 1] = va.y; wa[4 * i + 2] = va.z; wa[4 * i + 3] = va.w;
    wb[4 * i] = vb.x; wb[4 * i + 1] = vb.y; wb[4 * i + 2] = vb.z; wb[4 * i + 3] = vb.w;
  }
  release_and_wait(sm.wempty[s], sm.ffull[fs], fpar, lane, status);
  float acc[2][NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[0][i] = acc[1][i] = 0.f;
  const uint32_t magic = 0x64646464u;
  const uint32_t bias = 0x64206420u;  // f16x2 (1056, 1056): 1024 + 32
#pragma unroll
  for (int hv = 0; hv < 4; ++hv) {  // (h, v) = (hv >> 1, hv & 1)
    const uint32_t qaA = wa[3 * hv], qbA = wa[3 * hv + 1], qhA = wa[3 * hv + 2];
    const uint32_t qaB = wb[3 * hv], qbB = wb[3 * hv + 1], qhB = wb[3 * hv + 2];
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
      const float2 sc = tb.s[sidx][g];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        float c4[4] = {0.f, 0.f, 0.f, 0.f};
        const uint2 bf = sm.frag[fs][sidx][i][fl[i]];
        mma16816(c4, a0, a1, a2, a3, bf.x, bf.y);
        acc[0][i] = fmaf(sc.x, c4[0] + c4[1], acc[0][i]);
        acc[1][i] = fmaf(sc.y, c4[2] + c4[3], acc[1][i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float us = sm.unscale[fs][4 * i + t];
    tot[0][i] = fmaf(us, acc[0][i], tot[0][i]);
    tot[1][i] = fmaf(us, acc[1][i], tot[1][i]);
  }
}

// The per-32-block types: one scale d per block, applied after the block's two MMAs.
// A nibble type's word of a (block, row) holds the block's quant bytes 4t..4t+3 (order
// 0, 2, 1, 3): its low nibbles are elements 4t..4t+3 of the first 16-element half, its
// high nibbles those of the second.  A low nibble n masked into the mantissa of 1024
// gives 1024 + n, a high one 1024 + 16n; one f16x2 subtraction or fma (by 1/16) turns
// them into the exact integer weight: n - 8 (Q4_0), n (Q4_1).  For Q5_0 / Q5_1 the
// fifth bit of each element is OR-ed in beside the nibble first (bit 4 of the half:
// 1024 + q, or bit 8: 1024 + 16q), giving q - 16 (Q5_0) or q (Q5_1).  The fifth-bit
// word of a (block, row) holds the pair of elements of register r of thread t at bits
// 4r + t and 16 + 4r + t, so one shift and one mask move both to their halves.  The
// additive min m of Q4_1 / Q5_1 adds m times the block's sum of x (staged by the x warp).
template <int TYPE, int NT>
__device__ __forceinline__ void compute_chunk_q32(MvSmem<TYPE, NT> &sm, int s, int fs,
                                                  uint32_t fpar, int warp, int lane, int *status,
                                                  int nblk, const int (&fl)[NT],
                                                  float (&tot)[2][NT]) {
  constexpr bool NIB = TYPE != MQ_Q8_0, Q5 = fifth_type<TYPE>(), MADD = addmin_type<TYPE>();
  constexpr int QB = q32_bytes<TYPE>();
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *tile = sm.w[s];
  WarpTab<TYPE> &tb = sm.tab[warp];
  {  // lane (r, h): blocks 4h..4h+3 of row r (slots past the chunk's blocks hold 0)
    const int r = lane & 15, h = lane >> 4, row = 16 * warp + r;
    const uint2 dv = *reinterpret_cast<const uint2 *>(tile + q32_off_d<TYPE>() + row * 16 + 8 * h);
    float *dst = reinterpret_cast<float *>(&tb.s[4 * h][r & 7]) + (r >> 3);
    dst[0] = f16_lo(dv.x);
    dst[16] = f16_hi(dv.x);
    dst[32] = f16_lo(dv.y);
    dst[48] = f16_hi(dv.y);
    if constexpr (MADD) {
      const uint2 mv =
          *reinterpret_cast<const uint2 *>(tile + q32_off_m<TYPE>() + row * 16 + 8 * h);
      float *dm = reinterpret_cast<float *>(&tb.m[4 * h][r & 7]) + (r >> 3);
      dm[0] = f16_lo(mv.x);
      dm[16] = f16_hi(mv.x);
      dm[32] = f16_lo(mv.y);
      dm[48] = f16_hi(mv.y);
    }
  }
  __syncwarp();
  const int ra = 16 * warp + g, rb = ra + 8;
  // nibble types: .x the quant word, .y the fifth-bit word (0 without fifth bits)
  uint2 va[8], vb[8];  // blocks past the chunk's end hold stale but finite bytes
#pragma unroll
  for (int blk = 0; blk < 8; ++blk) {
    if constexpr (NIB) {
      va[blk].x = *reinterpret_cast<const uint32_t *>(tile + (blk * kRows + ra) * 16 + 4 * t);
      vb[blk].x = *reinterpret_cast<const uint32_t *>(tile + (blk * kRows + rb) * 16 + 4 * t);
      if constexpr (Q5) {
        va[blk].y = *reinterpret_cast<const uint32_t *>(tile + q32_off_h<TYPE>() +
                                                        (blk * kRows + ra) * 4);
        vb[blk].y = *reinterpret_cast<const uint32_t *>(tile + q32_off_h<TYPE>() +
                                                        (blk * kRows + rb) * 4);
      } else {
        va[blk].y = vb[blk].y = 0u;
      }
    } else {
      va[blk] = *reinterpret_cast<const uint2 *>(tile + (blk * kRows + ra) * QB + 8 * t);
      vb[blk] = *reinterpret_cast<const uint2 *>(tile + (blk * kRows + rb) * QB + 8 * t);
    }
  }
  release_and_wait(sm.wempty[s], sm.ffull[fs], fpar, lane, status);
  float acc[2][NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[0][i] = acc[1][i] = 0.f;
  const uint32_t magic = 0x64646464u;
  const uint32_t bias = 0x64806480u;  // f16x2 (1152, 1152): 1024 + 128
  // nibble types: (1024 + n) - kSub and (1024 + 16n)/16 + kAdd give the integer weight
  constexpr uint32_t kSub = TYPE == MQ_Q4_0   ? 0x64086408u   // 1032: n - 8
                            : TYPE == MQ_Q5_0 ? 0x64106410u   // 1040: q - 16
                                              : 0x64006400u;  // 1024: n or q
  constexpr uint32_t kAdd = TYPE == MQ_Q4_0   ? 0xD480D480u   // -72
                            : TYPE == MQ_Q5_0 ? 0xD500D500u   // -80
                                              : 0xD400D400u;  // -64
#pragma unroll
  for (int blk = 0; blk < 8; ++blk) {
    if (blk < nblk) {
      float c4[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) c4[i][r] = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t a0, a1, a2, a3;
        if constexpr (NIB) {
          constexpr uint32_t kM = 0x64006400u, kLo = 0x000f000fu, kHi = 0x00f000f0u;
          constexpr uint32_t kSixteenth = 0x2C002C00u;  // 1/16
          const uint32_t xA = va[blk].x, xB = vb[blk].x, xA8 = xA >> 8, xB8 = xB >> 8;
          const uint32_t hA = va[blk].y, hB = vb[blk].y;
          // exponent words OR-ed beside the nibbles: the magic, plus the fifth bits
          uint32_t mA0 = kM, mA2 = kM, mB0 = kM, mB2 = kM;
          if (u == 0) {
            if constexpr (Q5) {  // pairs of registers r = 0, 1 to bits 4 and 20
              constexpr uint32_t kB4 = 0x00100010u;
              mA0 = and_or(hA << (4 - t), kB4, kM);
              mB0 = and_or(hB << (4 - t), kB4, kM);
              mA2 = and_or(hA >> t, kB4, kM);
              mB2 = and_or(hB >> t, kB4, kM);
            }
            a0 = hsub2(and_or(xA, kLo, mA0), kSub);
            a2 = hsub2(and_or(xA8, kLo, mA2), kSub);
            a1 = hsub2(and_or(xB, kLo, mB0), kSub);
            a3 = hsub2(and_or(xB8, kLo, mB2), kSub);
          } else {
            if constexpr (Q5) {  // registers r = 2, 3 to bits 8 and 24
              constexpr uint32_t kB8 = 0x01000100u;
              mA0 = and_or(hA >> t, kB8, kM);
              mB0 = and_or(hB >> t, kB8, kM);
              mA2 = and_or(hA >> (4 + t), kB8, kM);
              mB2 = and_or(hB >> (4 + t), kB8, kM);
            }
            a0 = hfma2(and_or(xA, kHi, mA0), kSixteenth, kAdd);
            a2 = hfma2(and_or(xA8, kHi, mA2), kSixteenth, kAdd);
            a1 = hfma2(and_or(xB, kHi, mB0), kSixteenth, kAdd);
            a3 = hfma2(and_or(xB8, kHi, mB2), kSixteenth, kAdd);
          }
        } else {
          const uint32_t qA = (u ? va[blk].y : va[blk].x) ^ 0x80808080u;
          const uint32_t qB = (u ? vb[blk].y : vb[blk].x) ^ 0x80808080u;
          a0 = hsub2(__byte_perm(qA, magic, 0x5140), bias);
          a2 = hsub2(__byte_perm(qA, magic, 0x5342), bias);
          a1 = hsub2(__byte_perm(qB, magic, 0x5140), bias);
          a3 = hsub2(__byte_perm(qB, magic, 0x5342), bias);
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const uint2 bf = sm.frag[fs][2 * blk + u][i][fl[i]];
          mma16816(c4[i], a0, a1, a2, a3, bf.x, bf.y);
        }
      }
      const float2 dv = tb.s[blk][g];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        acc[0][i] = fmaf(dv.x, c4[i][0] + c4[i][1], acc[0][i]);
        acc[1][i] = fmaf(dv.y, c4[i][2] + c4[i][3], acc[1][i]);
      }
      if constexpr (MADD) {
        const float2 mv = tb.m[blk][g];
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const float xs = sm.xb[fs][blk][4 * i + t];
          acc[0][i] = fmaf(mv.x, xs, acc[0][i]);
          acc[1][i] = fmaf(mv.y, xs, acc[1][i]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float us = sm.unscale[fs][4 * i + t];
    tot[0][i] = fmaf(us, acc[0][i], tot[0][i]);
    tot[1][i] = fmaf(us, acc[1][i], tot[1][i]);
  }
}

// F16 / BF16: the weights are the A operand as stored (thread t's 8 bytes of a 16-element
// group and row hold elements 4t..4t+3, the two registers of a row).  Nothing to decode,
// so the warp reads its words straight from the stage inside the MMA loop and releases
// the stage after it.  Against bf16 weights the x warp stages bf16 hi/lo parts.
template <int TYPE, int NT>
__device__ __forceinline__ void compute_chunk_float(MvSmem<TYPE, NT> &sm, int s, int fs,
                                                    uint32_t fpar, int warp, int lane,
                                                    int *status, int ngrp, const int (&fl)[NT],
                                                    float (&tot)[2][NT]) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *tile = sm.w[s];
  const int ra = 16 * warp + g, rb = ra + 8;
  mbar_wait(sa(&sm.ffull[fs]), fpar, status, 24);
  float c4[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) c4[i][r] = 0.f;
#pragma unroll
  for (int grp = 0; grp < 16; ++grp) {
    if (grp < ngrp) {
      const uint2 wa = *reinterpret_cast<const uint2 *>(tile + (grp * kRows + ra) * 32 + 8 * t);
      const uint2 wb = *reinterpret_cast<const uint2 *>(tile + (grp * kRows + rb) * 32 + 8 * t);
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint2 bf = sm.frag[fs][grp][i][fl[i]];
        if constexpr (TYPE == MQ_BF16)
          mma16816_bf16(c4[i], wa.x, wb.x, wa.y, wb.y, bf.x, bf.y);
        else
          mma16816(c4[i], wa.x, wb.x, wa.y, wb.y, bf.x, bf.y);
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(sa(&sm.wempty[s]));
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float us = sm.unscale[fs][4 * i + t];
    tot[0][i] = fmaf(us, c4[i][0] + c4[i][1], tot[0][i]);
    tot[1][i] = fmaf(us, c4[i][2] + c4[i][3], tot[1][i]);
  }
}

// Results of the thread's row pair (rA, rA + 8) for batch row b.  A fused gate/up
// weight has rows in units of 16 (8 gate rows, then the same 8 rows of the up
// weight), so rA is a gate row and rA + 8 its up row: one SwiGLU output,
// silu(g) * u with silu(v) = v / (1 + e^-v), at output row 8 * (rA / 16) + rA % 8.
__device__ __forceinline__ void store_rows(const MvArgs &p, int b, int64_t rA, float vA,
                                           float vB) {
  if (p.swiglu) {
    if (rA < p.N) {
      const int64_t nout = p.N >> 1;
      p.y[int64_t(b) * nout + (rA >> 4) * 8 + (rA & 7)] = vA / (1.f + expf(-vA)) * vB;
    }
    return;
  }
  if (rA < p.N) p.y[int64_t(b) * p.N + rA] = vA;
  if (rA + 8 < p.N) p.y[int64_t(b) * p.N + rA + 8] = vB;
}

template <int TYPE, int NT, bool XE>
__global__ void __launch_bounds__(mv_threads<TYPE, XE>(), 2) matvec_kernel(const MvArgs p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = MvSmem<TYPE, NT>;
  constexpr int NS = Smem::NS;
  // aligned by an offset into the __shared__ array, so the compiler keeps knowing that
  // every member lives in shared memory (plain loads become LDS, addresses stay 32-bit)
  Smem &sm = *reinterpret_cast<Smem *>(
      smem_raw + ((128u - (uint32_t)__cvta_generic_to_shared(smem_raw)) & 127u));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int rank = blockIdx.x % p.S;
  const int64_t group = blockIdx.x / p.S;
  const int c_begin = (int)((int64_t)rank * p.nchunk / p.S);
  const int c_end = (int)((int64_t)(rank + 1) * p.nchunk / p.S);
  const int nch = c_end - c_begin;

  // fragment columns of absent batch rows stay zero (never read for stored outputs)
  {
    uint4 *f = reinterpret_cast<uint4 *>(&sm.frag[0][0][0][0]);
    constexpr int n16 = (int)(sizeof(sm.frag) / 16);
    for (int i = tid; i < n16; i += mv_threads<TYPE, XE>()) f[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < Smem::FS * 8) (&sm.unscale[0][0])[tid] = 0.f;
    constexpr int nxb = (int)(sizeof(sm.xb) / 4);
    for (int i = tid; i < nxb; i += mv_threads<TYPE, XE>()) (&sm.xb[0][0][0])[i] = 0.f;
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.wfull[s])), "r"(1));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.wempty[s])),
                   "r"(kCompute + x_warps<TYPE, XE>()));
    }
    for (int f = 0; f < Smem::FS; ++f) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.ffull[f])),
                   "r"(32 * x_warps<TYPE, XE>()));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.fempty[f])),
                   "r"(kCompute));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  float tot[2][NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) tot[0][i] = tot[1][i] = 0.f;

  if (warp == copy_warp<TYPE, XE>()) {
    if (lane == 0) issue_copies<TYPE, NT>(sm, p, group, c_begin, nch);
  } else if (warp == kCompute) {
    if constexpr (XE && TYPE == MQ_Q6_K)
      stage_x_rows<TYPE, NT, 0>(sm, p, c_begin, nch, lane);
    else
      stage_x<TYPE, NT, XE, 0>(sm, p, c_begin, nch, lane);
  } else if (x_warps<TYPE, XE>() == 2 && warp == kCompute + 1) {
    if constexpr (x_warps<TYPE, XE>() == 2) stage_x<TYPE, NT, XE, 1>(sm, p, c_begin, nch, lane);
  } else {
    // Lane (g, t) feeds column g of each n8 tile, i.e. batch row 4i + g/2.  Lanes
    // of absent batch rows read lane (g mod 2, t)'s fragment instead: the copy
    // only feeds accumulator columns that are never stored, and the shared
    // reads then touch fewer distinct words.
    int fl[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) fl[i] = 4 * i + (g >> 1) < p.B ? lane : (lane & 7);
    for (int i = 0; i < nch; ++i) {
      const int s = i % NS, fs = i % Smem::FS;
      const uint32_t fpar = (i / Smem::FS) & 1;
      mbar_wait(sa(&sm.wfull[s]), (i / NS) & 1, p.status, 22);
      if constexpr (kmin_type<TYPE>())
        compute_chunk_q4k<TYPE, NT>(sm, s, fs, fpar, warp, lane, p.status, fl, tot);
      else if constexpr (TYPE == MQ_Q6_K)
        compute_chunk_q6k<NT>(sm, s, fs, fpar, warp, lane, p.status, fl, tot);
      else if constexpr (float_w<TYPE>())
        compute_chunk_float<TYPE, NT>(sm, s, fs, fpar, warp, lane, p.status,
                                      chunk_width(p.K, c_begin + i) / 16, fl, tot);
      else
        compute_chunk_q32<TYPE, NT>(sm, s, fs, fpar, warp, lane, p.status,
                                    chunk_width(p.K, c_begin + i) / 32, fl, tot);
      __syncwarp();
      if (lane == 0) mbar_arrive(sa(&sm.fempty[fs]));  // this warp is done with the slot
    }
  }

  const int64_t rA = group * kRows + 16 * warp + g;
  if (p.S == 1) {
    if (warp < kCompute) {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int b = t + 4 * i;
        if (b < p.B) store_rows(p, b, rA, tot[0][i], tot[1][i]);
      }
    }
    return;
  }
  // split-K over the cluster: the ranks' partials are summed in rank order (the rows of
  // compute warp w by rank w mod S).
  // part overlays the ring, so every warp must be past its last ring access.
  __syncthreads();
  if (warp < kCompute) {
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      sm.part[16 * warp + g][t + 4 * i] = tot[0][i];
      sm.part[16 * warp + g + 8][t + 4 * i] = tot[1][i];
    }
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (warp < kCompute && warp % p.S == rank) {
    // the rows of compute warp w are summed by rank w mod S (the ranks share the reads);
    // all ranks' partials are loaded first (the distributed-shared-memory loads overlap),
    // then added in rank order
    float pa[kMaxSplit][NT], pb[kMaxSplit][NT];
#pragma unroll
    for (int r = 0; r < kMaxSplit; ++r) {
      if (r < p.S) {
        float(*rp)[8] = cluster.map_shared_rank(sm.part, r);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          pa[r][i] = rp[16 * warp + g][t + 4 * i];
          pb[r][i] = rp[16 * warp + g + 8][t + 4 * i];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const int b = t + 4 * i;
      float sA = 0.f, sB = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxSplit; ++r) {
        if (r < p.S) {
          sA += pa[r][i];
          sB += pb[r][i];
        }
      }
      if (b < p.B) store_rows(p, b, rA, sA, sB);
    }
  }
  cluster.sync();
}

template <int TYPE, int NT>
constexpr size_t mv_smem_bytes() {
  return sizeof(MvSmem<TYPE, NT>) + 128;
}

// Shared memory of two CTAs on one SM: 228 KB, less 1 KB reserved per CTA.
constexpr size_t kSmemTwoPerSm = 233472 / 2 - 1024;

template <int TYPE, int NT, bool XE>
mq_status launch_one(const MvArgs &a, cudaStream_t s, const char *name) {
  static_assert(float_w<TYPE>() || mv_smem_bytes<TYPE, NT>() <= kSmemTwoPerSm,
                "a quantised-type matvec CTA must leave room for a second one on its SM");
  const int64_t groups = (a.N + kRows - 1) / kRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(test_fail_launch() ? 0u : (unsigned)(groups * a.S), 1, 1);
  cfg.blockDim = dim3(mv_threads<TYPE, XE>(), 1, 1);
  cfg.dynamicSmemBytes = mv_smem_bytes<TYPE, NT>();
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.S > 1 ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, matvec_kernel<TYPE, NT, XE>, a);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // the refused launch leaves no error behind for later calls
    return fail(MQ_ERR_LAUNCH, "launch of %s (grid %u, cluster %d) failed: %s", name,
                cfg.gridDim.x, a.S, cudaGetErrorName(e));
  }
  return MQ_OK;
}

template <int TYPE, int NT, bool XE>
mq_status optin_mv(const DeviceState *st, const char *name) {
  const size_t smem = mv_smem_bytes<TYPE, NT>();
  if ((int)smem > st->smem_optin)
    return fail(MQ_ERR_LAUNCH, "%s needs %zu bytes of shared memory; the device allows %d", name,
                smem, st->smem_optin);
  cudaError_t e = cudaFuncSetAttribute(matvec_kernel<TYPE, NT, XE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)  // clusters of up to 16 CTAs (above the portable 8)
    e = cudaFuncSetAttribute(matvec_kernel<TYPE, NT, XE>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "smem / cluster opt-in of %s (%zu bytes) refused: %s", name, smem,
                cudaGetErrorName(e));
  return MQ_OK;
}

// The most clusters of S CTAs of this kernel that the device holds at once (0 if none).
template <int TYPE, int NT, bool XE>
int max_clusters(int S) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S, 1, 1);
  cfg.blockDim = dim3(mv_threads<TYPE, XE>(), 1, 1);
  cfg.dynamicSmemBytes = mv_smem_bytes<TYPE, NT>();
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = S;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, matvec_kernel<TYPE, NT, XE>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

// The three kernels of a type: one n8 tile (B <= 2; B = 3, 4 with the early x release) and
// two tiles (B = 5..8, early x release).
// Also records, per cluster size, the most clusters resident at once for every kernel of
// the type (the least over the three).
template <int TYPE>
mq_status optin_type(DeviceState *st, const char *name) {
  mq_status s;
  if ((s = optin_mv<TYPE, 1, false>(st, name)) != MQ_OK) return s;
  if ((s = optin_mv<TYPE, 1, true>(st, name)) != MQ_OK) return s;
  if ((s = optin_mv<TYPE, 2, true>(st, name)) != MQ_OK) return s;
  st->mv_clusters[TYPE][1] = 1 << 30;  // no cluster
  for (int S = 2; S <= kMaxSplit; ++S)
    st->mv_clusters[TYPE][S] = min(max_clusters<TYPE, 1, false>(S),
                                   min(max_clusters<TYPE, 1, true>(S),
                                       max_clusters<TYPE, 2, true>(S)));
  return MQ_OK;
}

mq_status init_matvec(DeviceState *st) {
  mq_status s;
  if ((s = init_matvec_kq(st)) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q8_0>(st, "matvec_kernel<Q8_0>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q4_K>(st, "matvec_kernel<Q4_K>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q6_K>(st, "matvec_kernel<Q6_K>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q5_K>(st, "matvec_kernel<Q5_K>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q4_0>(st, "matvec_kernel<Q4_0>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q4_1>(st, "matvec_kernel<Q4_1>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q5_0>(st, "matvec_kernel<Q5_0>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_Q5_1>(st, "matvec_kernel<Q5_1>")) != MQ_OK) return s;
  if ((s = optin_type<MQ_F16>(st, "matvec_kernel<F16>")) != MQ_OK) return s;
  return optin_type<MQ_BF16>(st, "matvec_kernel<BF16>");
}

// K-split: as many slices as keep every CTA of the grid resident in one wave of cps CTAs
// per SM, at most one per chunk; up to 8 (a portable cluster) by that count alone, and up to
// 16 where the device also reports every cluster of that size co-resident for each of the
// type's kernels (its count of resident clusters covers how clusters fit into the GPCs).
// Depends only on (N, K), the type and the device, never on B, so batched columns
// reproduce the B = 1 result bitwise.  Measured on Q6_K 3584 x 18944 (28 row groups, 74
// chunks): S = 8 / 9 / 10 took 16.3 / 15.5 / 15.0 us at B = 1 and 23.3 / 22.0 / 23.1 us at
// B = 8; 11 to 16 need two waves (20.6-22.9 us at B = 1).  The counts check alone would
// lower f16 weights' 5-way split (whose clusters it does not count as all co-resident),
// which measured slower at B = 8, so it only decides sizes above 8.
static int choose_split(int64_t N, int64_t K, int type, const DeviceState *st, int cps) {
  const int64_t groups = (N + kRows - 1) / kRows;
  const int nchunk = (int)((K + kChunk - 1) / kChunk);
  const int64_t fit = cps * int64_t(st->sms) / groups;
  int top = fit < kMaxSplit ? (int)fit : kMaxSplit;
  if (top > nchunk) top = nchunk;
  for (int S = top; S > 8; --S)
    if (groups <= st->mv_clusters[type][S]) return S;
  return top < 8 ? (top > 1 ? top : 1) : 8;
}

template <int TYPE>
mq_status launch_type(const MvArgs &a, int B, cudaStream_t s, const char *name) {
  if (B > 4) return launch_one<TYPE, 2, true>(a, s, name);
  if (B > 2) return launch_one<TYPE, 1, true>(a, s, name);
  return launch_one<TYPE, 1, false>(a, s, name);
}

mq_status launch_matvec(const mq_weight *W, const float *x, float *y, int B, cudaStream_t s,
                        const DeviceState *st) {
  MvArgs a;
  a.q = W->q;
  a.d = W->d;
  a.dm = W->dm;
  a.qh = W->qh;
  a.x = x;
  a.y = y;
  a.N = W->N;
  a.K = W->K;
  a.B = B;
  a.nchunk = (int)((W->K + kChunk - 1) / kChunk);
  // the f16 / bf16 stages (64 KB) leave room for one CTA per SM, the others for two
  a.S = choose_split(W->N, W->K, W->type, st, float_type(W->type) ? 1 : 2);
  a.swiglu = W->ffn_gu;
  a.status = st->status;
  const bool kq = W->type == MQ_Q4_K || W->type == MQ_Q5_K || W->type == MQ_Q6_K;
  if (kq && matvec_kq_applies(W->N, st->sms)) return launch_matvec_kq(W, x, y, B, s, st);
  switch (W->type) {
    case MQ_Q4_K: return launch_type<MQ_Q4_K>(a, B, s, "matvec_kernel<Q4_K>");
    case MQ_Q6_K: return launch_type<MQ_Q6_K>(a, B, s, "matvec_kernel<Q6_K>");
    case MQ_Q5_K: return launch_type<MQ_Q5_K>(a, B, s, "matvec_kernel<Q5_K>");
    case MQ_Q4_0: return launch_type<MQ_Q4_0>(a, B, s, "matvec_kernel<Q4_0>");
    case MQ_Q4_1: return launch_type<MQ_Q4_1>(a, B, s, "matvec_kernel<Q4_1>");
    case MQ_Q5_0: return launch_type<MQ_Q5_0>(a, B, s, "matvec_kernel<Q5_0>");
    case MQ_Q5_1: return launch_type<MQ_Q5_1>(a, B, s, "matvec_kernel<Q5_1>");
    case MQ_F16: return launch_type<MQ_F16>(a, B, s, "matvec_kernel<F16>");
    case MQ_BF16: return launch_type<MQ_BF16>(a, B, s, "matvec_kernel<BF16>");
    default: return launch_type<MQ_Q8_0>(a, B, s, "matvec_kernel<Q8_0>");
  }
}

}  // namespace mq
