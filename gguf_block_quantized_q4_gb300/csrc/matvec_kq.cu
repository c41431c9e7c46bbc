// matvec_kq.cu -- persistent decode matvec y[b][n] = sum_k w[n][k] x[b][k] for the
// super-block types Q4_K, Q5_K and Q6_K, B <= 8, for weights of at least SMs / 2 row groups
// of 128 ("minfer CUDA Backend Design" §4.4: the nt == 1 matvec and the _multi variants for
// nt 2..8; "minfer Architecture Execution Plan" A6: the decode loop is weight-streaming
// bound).  Narrower weights need a K split and run matvec.cu's kernel.
//
// The arithmetic follows matvec.cu (weights dequantised in registers into exact f16
// tensor-core fragments, x carried as f16 hi + lo parts under a power-of-two scale per
// chunk, mma.sync m16n8k16 with f32 accumulation).  For Q4_K / Q5_K the operand is formed
// differently: a quant masked into the low mantissa bits of an f16 half is the exact
// subnormal q * 2^-24 (or 16q * 2^-24 for a high nibble), so one LOP3 forms each A register,
// and the 6-bit sub-block scale and d are applied to each sub-block's f32 MMA result
// (d * sc * 2^24, or / 16 for high nibbles: exact powers of two).
//
// Data movement.  One persistent CTA per SM, 21 warps:
//  * warp 18, one lane: streams the weight tiles (one contiguous 1-D bulk copy per 128-row
//    group and 256-element chunk, the decode-plane tiles of repack.cu) through a ring of NS
//    stages.  Registered weights are never written by a kernel, so it does not wait for the
//    previous kernel in the stream: a launch's first HBM traffic overlaps the previous
//    kernel's end (programmatic dependent launch);
//  * warps 16, 17, 19, 20: x warps (row slice, chunk parity).  After griddepcontrol.wait each
//    reads its rows of x for its chunks from global memory two chunks ahead (cp.async into
//    a staging ring) and converts them into B fragments in a ring of FS slots, so x never
//    waits on a weight stage and a weight stage is released as soon as the compute warps
//    have read it;
//  * warps 0-15: two teams of eight; team t computes the chunks whose index in the CTA's
//    chunk sequence has parity t (those converted by the x warps of parity t), warp w of a
//    team rows 16w..16w+15 of the group.  At the end of a group the
//    team-1 warp hands its partial sums to the team-0 warp of the same rows through shared
//    memory (an mbarrier pair), which adds them to its own (a fixed order) and stores y.
// CTA b takes groups b, b + grid, ... (grid = min(groups, SMs)), and the ring runs on
// across its groups, so there is no ramp between them.  The per-row arithmetic does not
// depend on B, so every column of a batched call equals the B = 1 call bitwise.  All
// mbarrier waits are bounded (2 s by %globaltimer; expiry writes the status word).
#include "mv_device.cuh"

namespace mq {
namespace {

using namespace mvd;

constexpr int kRows = kRowGroup;   // rows per group (128)
constexpr int kTeam = 8;           // compute warps per team
constexpr int kCompute = 2 * kTeam;
constexpr int kFS = 4;             // fragment slots
constexpr int kXS = 3;             // x staging slots per x warp (its chunks read 2 ahead)

template <int NT>
__host__ __device__ constexpr int kq_xrows() { return NT == 1 ? 2 : 4; }  // rows per x warp
// x warps: (row slice of kq_xrows rows, chunk parity); 4 in both kernels
template <int NT>
__host__ __device__ constexpr int kq_xwarps() { return 2 * (4 * NT / kq_xrows<NT>()); }
template <int NT>
__host__ __device__ constexpr int kq_threads() { return 32 * (kCompute + kq_xwarps<NT>() + 1); }
// The copy warp (warp 18, the third warp scheduler) sits between the x warps of the first
// row slice (warps 16, 17) and the others, so with B <= kq_xrows it shares its scheduler
// with no busy x warp: its next bulk copy goes out as soon as a stage is released.
template <int NT>
__host__ __device__ constexpr int kq_copy_warp() { return kCompute + 2; }
// x warp index (0 .. kq_xwarps - 1) of warp w >= kCompute, w != the copy warp
__device__ __forceinline__ int kq_xwarp_index(int w) {
  return w < kCompute + 2 ? w - kCompute : w - kCompute - 1;
}

template <int TYPE>
__host__ __device__ constexpr int kq_row_bytes() {
  return TYPE == MQ_Q4_K ? 144 : TYPE == MQ_Q5_K ? 176 : 210;
}
template <int TYPE>
__host__ __device__ constexpr int kq_tile_bytes() { return kRows * kq_row_bytes<TYPE>(); }
template <int TYPE>
__host__ __device__ constexpr bool kq_kmin() { return TYPE != MQ_Q6_K; }
// Weight-ring depth.  It must be even, and so must the fragment ring's: chunk i goes to
// stage i % NS and slot i % FS and is consumed by team i % 2, so with even depths every
// stage and slot belongs to one team, which uses it in order; with an odd depth a stage
// alternates between the teams, and a team running a round ahead would find the parity of
// a phase two ahead already "complete".  Four stages measured faster than six and eight
// (Q4_K 18944 x 3584, B = 1 and 2: 10.1 against 10.5 and 11.7 us), and the same for the
// Q6_K LM head.
template <int TYPE, int NT>
__host__ __device__ constexpr int kq_stages() {
  return 4;
}
static_assert(kFS % 2 == 0, "each fragment slot must belong to one team (see kq_stages)");

struct KqArgs {
  const uint8_t *q;
  const float *x;
  float *y;
  int64_t N, K;
  int B;
  int nchunk;   // K / 256
  int64_t groups;
  int swiglu;
  int *status;
  // the activation fragment plane of this call (xplane.cu), or nullptr: the x warps convert
  // x themselves
  const uint8_t *xp;
};

template <int TYPE>
struct KqTab;
template <>
struct KqTab<MQ_Q4_K> {
  float4 s[4][8];  // [pair c'][r]: d*sc (low-nibble sub-block 2c') of rows r, r+8, then
                   // d*sc/16 (high-nibble sub-block 2c'+1) of rows r, r+8
  uint2 mf[4][8];  // [t][r]: min-term A fragment words of rows r, r+8
  float2 dm[8];    // [r]: 32*dmin of rows r, r+8
};
template <>
struct KqTab<MQ_Q5_K> : KqTab<MQ_Q4_K> {};
template <>
struct KqTab<MQ_Q6_K> {
  float2 s[16][8];  // [16-element group][r]: d*sc of rows r, r+8
};

template <int TYPE, int NT>
struct KqSmem {
  static constexpr int NS = kq_stages<TYPE, NT>();
  static_assert(NS % 2 == 0, "each weight stage must belong to one team (see kq_stages)");
  static constexpr int FG = kq_kmin<TYPE>() ? 17 : 16;  // 16 groups (+ the min group)
  alignas(128) uint8_t w[NS][kq_tile_bytes<TYPE>()];  // weight tiles
  // B fragments, each group padded by 8 words (consecutive groups 8 banks apart)
  alignas(16) uint2 frag[kFS][FG][NT][32 + (NT == 1 ? 4 : 2)];
  alignas(16) float unscale[kFS][8];      // 2^-e per batch row of the slot's chunk
  alignas(16) float xr[kq_xwarps<NT>()][kXS][kq_xrows<NT>()][kChunk];  // x staging rings
  KqTab<TYPE> tab[kCompute];
  float xs[kq_xwarps<NT>()][kq_xrows<NT>()][8];  // x-warp scratch: sub-block sums
  float xch[2][kTeam][32][2 * NT];         // team 1 -> team 0 partial sums, by unit parity
  uint64_t wfull[NS], wempty[NS], ffull[kFS], fempty[kFS], pfull[kTeam][2], pempty[kTeam][2];
  static_assert(sizeof(frag[0]) == FG * xp_group_bytes(NT),
                "a fragment slot must have the activation fragment plane's layout");
};

template <int TYPE, int NT>
constexpr size_t kq_smem_bytes() {
  return sizeof(KqSmem<TYPE, NT>) + 128;
}

// The units of this CTA: groups blockIdx.x, + gridDim.x, ..., each over all chunks.
struct Unit {
  int64_t group;
  int cb, ce;
};
__device__ __forceinline__ bool unit_at(const KqArgs &p, int u, Unit &out) {
  const int64_t g = blockIdx.x + int64_t(u) * gridDim.x;
  if (g >= p.groups) return false;
  out.group = g;
  out.cb = 0;
  out.ce = p.nchunk;
  return true;
}

// ---------------------------------------------------------------------------
// Copy warp (one lane): the weight tile of every chunk of every unit, in order.
template <int TYPE, int NT>
__device__ __forceinline__ void kq_copies(KqSmem<TYPE, NT> &sm, const KqArgs &p) {
  constexpr int NS = KqSmem<TYPE, NT>::NS;
  constexpr uint32_t TB = kq_tile_bytes<TYPE>();
  // registered weights are never written by a kernel, so the copies need not wait for the
  // previous kernel in the stream (griddepcontrol.wait): only x does
  int i = 0;
  Unit un;
  for (int u = 0; unit_at(p, u, un); ++u) {
    for (int c = un.cb; c < un.ce; ++c, ++i) {
      const int s = i % NS;
      if (i >= NS) mbar_wait(sa(&sm.wempty[s]), ((i / NS) - 1) & 1, p.status, 31);
      // ramp: the launch's first two tiles go out at once, each later one of the first ring
      // round when the tile two before it has landed, so that every SM's first tile is not
      // queued behind the whole first round of all SMs (Q6_K 18944 x 3584 B = 1 / 2 / 8:
      // 12.63 / 13.27 / 18.68 -> 12.44 / 12.92 / 18.14 us, Q5_K B = 1 12.90 -> 12.67 us;
      // Q4_K and the Q6_K LM head within 0.5%)
      else if (i >= 2) mbar_wait(sa(&sm.wfull[i - 2]), 0u, p.status, 30);
      const uint32_t bar = sa(&sm.wfull[s]);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(TB)
                   : "memory");
      bulk_1d(sa(sm.w[s]), p.q + (un.group * p.nchunk + c) * int64_t(TB), TB, bar);
    }
  }
}

// ---------------------------------------------------------------------------
// x warp (xi, par): batch rows R xi .. R xi + R - 1 (R = kq_xrows) of the chunks whose index in this CTA's
// chunk sequence has parity par (one out-of-line copy of the code for all x warps), read from global memory kXS - 1 chunks ahead, into B
// fragments (hi / lo f16 parts under a power-of-two scale that puts the chunk's max |x| in
// [2^14, 2^15)) and, for Q4_K / Q5_K, the min-term fragments of the sub-block sums.  The
// arithmetic per row is that of matvec.cu's x warp; rows past B are skipped.
template <int TYPE, int NT>
__device__ __noinline__ void kq_stage_x(KqSmem<TYPE, NT> &sm, const KqArgs &p, int lane, int xi,
                                        int par) {
  constexpr int R = kq_xrows<NT>();
  const int r0 = R * xi;
  const int nr = min(max(p.B - r0, 0), R);  // live rows of this warp
  if (nr == 0) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Lane handles float4 items f = lane and lane + 32 of each row.  Each lane copies its own
  // items (16-byte cp.async, one commit group per chunk) into the warp's staging ring, so
  // only its own copies need waiting for.
  float(*xr)[R][kChunk] = sm.xr[2 * xi + par];
  // cursor over this warp's chunks: global index i (parity par), unit u, chunk c
  struct Cur {
    Unit un;
    int u, c, i;
    bool alive;
  };
  auto start = [&](Cur &q) {
    q.u = 0;
    q.i = 0;
    q.alive = unit_at(p, 0, q.un);
    q.c = q.alive ? q.un.cb : 0;
    if (q.alive && par == 1) {  // to the second chunk of the sequence
      if (++q.c >= q.un.ce) {
        q.alive = unit_at(p, ++q.u, q.un);
        q.c = q.alive ? q.un.cb : 0;
      }
      q.i = 1;
    }
  };
  auto advance = [&](Cur &q) {  // two chunks on
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (!q.alive) return;
      if (++q.c >= q.un.ce) {
        q.alive = unit_at(p, ++q.u, q.un);
        q.c = q.alive ? q.un.cb : 0;
      }
    }
    q.i += 2;
  };
  Cur iq, cq;
  start(iq);
  start(cq);
  auto issue = [&](int slot) {
    if (iq.alive) {
      for (int b = 0; b < nr; ++b)
#pragma unroll
        for (int k = 0; k < 2; ++k)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                           sa(&xr[slot][b][4 * (lane + 32 * k)])),
                       "l"(p.x + int64_t(r0 + b) * p.K + int64_t(iq.c) * kChunk +
                           4 * (lane + 32 * k))
                       : "memory");
      advance(iq);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int k = 0; k < kXS - 1; ++k) issue(k);
  for (int n = 0; cq.alive; ++n) {
    issue((n + kXS - 1) % kXS);  // the slot of this warp's previous chunk
    asm volatile("cp.async.wait_group %0;" ::"n"(kXS - 1) : "memory");
    const int i = cq.i, fs = i % kFS;
    if (i >= kFS) mbar_wait(sa(&sm.fempty[fs]), ((i / kFS) - 1) & 1, p.status, 35);
    float4 cur[R][2];
    float scale[R];
#pragma unroll
    for (int b = 0; b < R; ++b) {
      if (b >= nr) break;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        cur[b][k] = *reinterpret_cast<const float4 *>(&xr[n % kXS][b][4 * (lane + 32 * k)]);
      float m = 0.f;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(cur[b][k].x), fabsf(cur[b][k].y)),
                           fmaxf(fabsf(cur[b][k].z), fabsf(cur[b][k].w))));
      const unsigned mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
      const int E = (int)((mb >> 23) & 255);
      int e = mb == 0 ? 0 : 141 - max(E, 1);
      e = min(max(e, -100), 126);
      scale[b] = __int_as_float((e + 127) << 23);
      if (lane == 0) sm.unscale[fs][r0 + b] = __int_as_float((127 - e) << 23);
    }
#pragma unroll
    for (int bl = 0; bl < R; ++bl) {
      if (bl >= nr) break;
      const int b = r0 + bl;
      const int col = 2 * (b & 3);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = lane + 32 * k, g16 = f >> 2, t = f & 3;
        const float v0 = cur[bl][k].x * scale[bl], v1 = cur[bl][k].y * scale[bl],
                    v2 = cur[bl][k].z * scale[bl], v3 = cur[bl][k].w * scale[bl];
        const uint32_t hi01 = pack_f16x2(v0, v1), hi23 = pack_f16x2(v2, v3);
        const uint32_t lo01 = pack_f16x2(v0 - f16_lo(hi01), v1 - f16_hi(hi01));
        const uint32_t lo23 = pack_f16x2(v2 - f16_lo(hi23), v3 - f16_hi(hi23));
        sm.frag[fs][g16][b >> 2][col * 4 + t] = make_uint2(hi01, hi23);
        sm.frag[fs][g16][b >> 2][(col + 1) * 4 + t] = make_uint2(lo01, lo23);
        if constexpr (kq_kmin<TYPE>()) {
          // sum of sub-block f >> 3 (8 consecutive items), scaled by 1/32 so that
          // |sum| < 2^15 fits f16
          float ps = (v0 + v1) + (v2 + v3);
          ps += __shfl_xor_sync(0xffffffffu, ps, 1);
          ps += __shfl_xor_sync(0xffffffffu, ps, 2);
          ps += __shfl_xor_sync(0xffffffffu, ps, 4);
          if ((lane & 7) == 0) sm.xs[2 * xi + par][bl][f >> 3] = ps * 0.03125f;
        }
      }
    }
    if constexpr (kq_kmin<TYPE>()) {
      // min-term B fragments: lane (col', t') of row b holds sums 2t', 2t'+1 (hi or lo part)
      __syncwarp();
      if (lane < 8) {
        const int part = lane >> 2, t = lane & 3;
        for (int bl = 0; bl < nr; ++bl) {
          const int b = r0 + bl;
          const float s0 = sm.xs[2 * xi + par][bl][2 * t], s1 = sm.xs[2 * xi + par][bl][2 * t + 1];
          const uint32_t h = pack_f16x2(s0, s1);
          const uint32_t word = part == 0 ? h : pack_f16x2(s0 - f16_lo(h), s1 - f16_hi(h));
          sm.frag[fs][16][b >> 2][(2 * (b & 3) + part) * 4 + t] = make_uint2(word, 0u);
        }
      }
      __syncwarp();
    }
    mbar_arrive(sa(&sm.ffull[fs]));  // each lane, after its own fragment stores
    advance(cq);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// With an activation fragment plane: lane 0 of the x warp of row slice 0 and chunk parity
// par copies the fragments and unscale factors of this parity's chunks into their fragment
// slots (one bulk-copy transaction per slot), once the team is done with the slot.
template <int TYPE, int NT>
__device__ __noinline__ void kq_copy_plane(KqSmem<TYPE, NT> &sm, const KqArgs &p, int par) {
  constexpr uint32_t FB = KqSmem<TYPE, NT>::FG * xp_group_bytes(NT);
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the plane comes from the previous kernel
  int i = 0;
  Unit un;
  for (int u = 0; unit_at(p, u, un); ++u) {
    for (int c = un.cb; c < un.ce; ++c, ++i) {
      if ((i & 1) != par) continue;
      const int fs = i % kFS;
      if (i >= kFS) mbar_wait(sa(&sm.fempty[fs]), ((i / kFS) - 1) & 1, p.status, 38);
      const uint32_t bar = sa(&sm.ffull[fs]);
      mbar_arrive_tx(bar, FB + 32u);
      const uint8_t *src = p.xp + int64_t(c) * xp_chunk_bytes(NT);
      bulk_1d(sa(&sm.frag[fs][0][0][0]), src, FB, bar);
      bulk_1d(sa(&sm.unscale[fs][0]), src + xp_off_unscale(NT), 32u, bar);
    }
  }
}

// Every lane releases the weight stage after its own reads of it (the stage's "empty"
// barrier counts all 256 lanes of the team), then waits for the fragment slot.
__device__ __forceinline__ void kq_release_and_wait(uint64_t &wempty, uint64_t &ffull,
                                                    uint32_t fpar, int lane, int *status) {
  mbar_arrive(sa(&wempty));
  mbar_wait(sa(&ffull), fpar, status, 34);
}

// Position in a ring of N slots: slot and phase parity, advanced without division.
template <int N>
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void advance(int d) {  // d < N
    s += d;
    if (s >= N) {
      s -= N;
      ph ^= 1u;
    }
  }
};

// Q4_K / Q5_K chunk of one compute warp (rows 16 wq .. 16 wq + 15 of the tile).  A quant
// q masked into the low mantissa bits of an f16 half is the exact subnormal q * 2^-24
// (bits 0-4: low nibble, with Q5_K's fifth bit at bit 4) or 16q * 2^-24 (bits 4-8: high
// nibble, fifth bit at bit 8), so one LOP3 forms each A register; the tensor cores take f16
// subnormals exactly, every product q * x is exact in f32, and one MMA accumulator per
// 32-element sub-block (two K halves) is scaled after the MMA by d * sc_j (d * sc_j / 16
// for the high nibbles) from the warp's table.  The min term -dmin * m_j * sum(x over the
// sub-block) is one more MMA per super-block (exact integer mins m_j, sub-block sums of x).
template <int TYPE, int NT>
__device__ __forceinline__ void kq_chunk_q4k(KqSmem<TYPE, NT> &sm, int s, int fs, uint32_t fpar,
                                             int warp, int wq, int lane, int *status,
                                             const int (&fl)[NT], float (&tot)[2][NT]) {
  constexpr bool Q5 = TYPE == MQ_Q5_K;
  constexpr int RS = Q5 ? 176 : 144;
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *tile = sm.w[s];
  KqTab<MQ_Q4_K> &tb = sm.tab[warp];
  {  // lane c'*8 + r: sub-blocks 2c', 2c'+1 of rows r and r+8
    const int cp = lane >> 3, r = lane & 7;
    const uint4 ha = *reinterpret_cast<const uint4 *>(tile + (16 * wq + r) * RS);
    const uint4 hb = *reinterpret_cast<const uint4 *>(tile + (16 * wq + r + 8) * RS);
    // 6-bit scales / mins of sub-blocks 4q..4q+3 as bytes (q = cp >> 1)
    const bool low = cp < 2;
    const uint32_t sa4 = low ? ha.y & 0x3f3f3f3fu
                             : (ha.w & 0x0f0f0f0fu) | ((ha.y >> 2) & 0x30303030u);
    const uint32_t sb4 = low ? hb.y & 0x3f3f3f3fu
                             : (hb.w & 0x0f0f0f0fu) | ((hb.y >> 2) & 0x30303030u);
    const uint32_t ma4 = low ? ha.z & 0x3f3f3f3fu
                             : ((ha.w >> 4) & 0x0f0f0f0fu) | ((ha.z >> 2) & 0x30303030u);
    const uint32_t mb4 = low ? hb.z & 0x3f3f3f3fu
                             : ((hb.w >> 4) & 0x0f0f0f0fu) | ((hb.z >> 2) & 0x30303030u);
    const int sh = 16 * (cp & 1);  // bytes 2(cp&1), 2(cp&1)+1: sub-blocks 2c', 2c'+1
    // d * sc * 2^24 for the low-nibble sub-block (its A registers carry q * 2^-24); the same
    // / 16 for the high-nibble one (16q * 2^-24); powers of two, so the products stay exact
    const float dA = f16_lo(ha.x) * 16777216.f, dB = f16_lo(hb.x) * 16777216.f;
    tb.s[cp][r] = make_float4(dA * (float)((sa4 >> sh) & 255u), dB * (float)((sb4 >> sh) & 255u),
                              dA * 0.0625f * (float)((sa4 >> (sh + 8)) & 255u),
                              dB * 0.0625f * (float)((sb4 >> (sh + 8)) & 255u));
    // min-term A fragment: the exact integer mins as f16, (1024 + m) - 1024
    const uint32_t sel = (cp & 1) ? 0x5342u : 0x5140u, k1024 = 0x64006400u;
    tb.mf[cp][r] = make_uint2(hsub2(__byte_perm(ma4, 0x64646464u, sel), k1024),
                              hsub2(__byte_perm(mb4, 0x64646464u, sel), k1024));
    if (cp == 0) tb.dm[r] = make_float2(32.f * f16_hi(ha.x), 32.f * f16_hi(hb.x));
  }
  __syncwarp();
  const int ra = 16 * wq + g, rb = ra + 8;
  const uint4 a0 = *reinterpret_cast<const uint4 *>(tile + ra * RS + 16 + 32 * t);
  const uint4 a1 = *reinterpret_cast<const uint4 *>(tile + ra * RS + 32 + 32 * t);
  const uint4 b0 = *reinterpret_cast<const uint4 *>(tile + rb * RS + 16 + 32 * t);
  const uint4 b1 = *reinterpret_cast<const uint4 *>(tile + rb * RS + 32 + 32 * t);
  const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  uint2 qha = make_uint2(0u, 0u), qhb = make_uint2(0u, 0u);  // Q5_K fifth-bit words
  if constexpr (Q5) {
    qha = *reinterpret_cast<const uint2 *>(tile + ra * RS + 144 + 8 * t);
    qhb = *reinterpret_cast<const uint2 *>(tile + rb * RS + 144 + 8 * t);
  }
  kq_release_and_wait(sm.wempty[s], sm.ffull[fs], fpar, lane, status);
  float cm[NT][4];
  {
    const uint2 mf = tb.mf[t][g];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const uint2 bm = sm.frag[fs][16][i][fl[i]];
      mma16816_z(cm[i], mf.x, mf.y, 0u, 0u, bm.x, bm.y);
    }
  }
  float yA[NT], yB[NT];
  constexpr uint32_t kLo = 0x000f000fu, kHi = 0x00f000f0u;
#pragma unroll
  for (int cp = 0; cp < 4; ++cp) {
    float cL[NT][4], cH[NT][4];  // sub-blocks 2c' (low nibbles) and 2c'+1 (high nibbles)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t xa = wa[2 * cp + u], xb = wb[2 * cp + u];
      const uint32_t xa8 = xa >> 8, xb8 = xb >> 8;
      // Q5_K: the fifth bits (bit 2c' of bytes 0/2 or 1/3 of the fifth-bit word for the
      // low nibbles, bit 2c' + 1 for the high nibbles) beside the quant
      uint32_t mla = 0u, mlb = 0u, mla8 = 0u, mlb8 = 0u, mha = 0u, mhb = 0u, mha8 = 0u, mhb8 = 0u;
      if constexpr (Q5) {
        constexpr uint32_t kB4 = 0x00100010u, kB8 = 0x01000100u;
        const uint32_t qa = u ? qha.y : qha.x, qb = u ? qhb.y : qhb.x;
        mla = shl(qa, 4 - 2 * cp) & kB4;
        mlb = shl(qb, 4 - 2 * cp) & kB4;
        mla8 = shl(qa, -4 - 2 * cp) & kB4;
        mlb8 = shl(qb, -4 - 2 * cp) & kB4;
        mha = shl(qa, 7 - 2 * cp) & kB8;
        mhb = shl(qb, 7 - 2 * cp) & kB8;
        mha8 = shl(qa, -1 - 2 * cp) & kB8;
        mhb8 = shl(qb, -1 - 2 * cp) & kB8;
      }
      const uint32_t l0 = and_or(xa, kLo, mla), l1 = and_or(xb, kLo, mlb);
      const uint32_t l2 = and_or(xa8, kLo, mla8), l3 = and_or(xb8, kLo, mlb8);
      const uint32_t h0 = and_or(xa, kHi, mha), h1 = and_or(xb, kHi, mhb);
      const uint32_t h2 = and_or(xa8, kHi, mha8), h3 = and_or(xb8, kHi, mhb8);
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const uint2 bl = sm.frag[fs][4 * cp + u][i][fl[i]];      // sub-block 2c', K half u
        const uint2 bh = sm.frag[fs][4 * cp + 2 + u][i][fl[i]];  // sub-block 2c'+1
        if (u == 0) {
          mma16816_z(cL[i], l0, l1, l2, l3, bl.x, bl.y);
          mma16816_z(cH[i], h0, h1, h2, h3, bh.x, bh.y);
        } else {
          mma16816(cL[i], l0, l1, l2, l3, bl.x, bl.y);
          mma16816(cH[i], h0, h1, h2, h3, bh.x, bh.y);
        }
      }
    }
    const float4 sc = tb.s[cp][g];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      const float a = fmaf(sc.z, cH[i][0] + cH[i][1], sc.x * (cL[i][0] + cL[i][1]));
      const float b = fmaf(sc.w, cH[i][2] + cH[i][3], sc.y * (cL[i][2] + cL[i][3]));
      yA[i] = cp == 0 ? a : yA[i] + a;
      yB[i] = cp == 0 ? b : yB[i] + b;
    }
  }
  const float2 dm = tb.dm[g];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float us = sm.unscale[fs][4 * i + t];
    tot[0][i] = fmaf(us, fmaf(-dm.x, cm[i][0] + cm[i][1], yA[i]), tot[0][i]);
    tot[1][i] = fmaf(us, fmaf(-dm.y, cm[i][2] + cm[i][3], yB[i]), tot[1][i]);
  }
}

// Q6_K chunk of one compute warp: 6-bit quants (4 low bits from ql, 2 high from qh) as
// exact f16 q - 32, one MMA per 16-element group, the group's d * sc applied to the f32
// result.
template <int NT>
__device__ __forceinline__ void kq_chunk_q6k(KqSmem<MQ_Q6_K, NT> &sm, int s, int fs,
                                             uint32_t fpar, int warp, int wq, int lane,
                                             int *status, const int (&fl)[NT],
                                             float (&tot)[2][NT]) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *tile = sm.w[s];
  KqTab<MQ_Q6_K> &tb = sm.tab[warp];
  {  // lane (r, h): groups 8h..8h+7 of row r
    const int r = lane & 15, h = lane >> 4, row = 16 * wq + r;
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
  const int ra = 16 * wq + g, rb = ra + 8;
  uint32_t wa[12], wb[12];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const uint4 va = *reinterpret_cast<const uint4 *>(tile + ra * 192 + 48 * t + 16 * i);
    const uint4 vb = *reinterpret_cast<const uint4 *>(tile + rb * 192 + 48 * t + 16 * i);
    wa[4 * i] = va.x; wa[4 * i + 1] = va.y; wa[4 * i + 2] = va.z; wa[4 * i + 3] = va.w;
    wb[4 * i] = vb.x; wb[4 * i + 1] = vb.y; wb[4 * i + 2] = vb.z; wb[4 * i + 3] = vb.w;
  }
  kq_release_and_wait(sm.wempty[s], sm.ffull[fs], fpar, lane, status);
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

// Results of the thread's row pair (rA, rA + 8) for batch row b; a fused gate/up weight
// (rows in units of 16: 8 gate rows, then the same 8 rows of the up weight) stores
// silu(g) * u with silu(v) = v / (1 + e^-v) at output row 8 * (rA / 16) + rA % 8.
__device__ __forceinline__ void kq_store(const KqArgs &p, int b, int64_t rA, float vA,
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

template <int TYPE, int NT>
__global__ void __launch_bounds__(kq_threads<NT>(), 1) matvec_kq_kernel(const KqArgs p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = KqSmem<TYPE, NT>;
  constexpr int NS = Smem::NS;
  Smem &sm = *reinterpret_cast<Smem *>(
      smem_raw + ((128u - (uint32_t)__cvta_generic_to_shared(smem_raw)) & 127u));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;

  // fragment columns of absent batch rows stay zero (never read for stored outputs); with an
  // activation fragment plane the slots are filled by bulk copies alone (zeros included)
  if (!p.xp) {
    uint4 *f = reinterpret_cast<uint4 *>(&sm.frag[0][0][0][0]);
    constexpr int n16 = (int)(sizeof(sm.frag) / 16);
    for (int i = tid; i < n16; i += kq_threads<NT>()) f[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < kFS * 8) (&sm.unscale[0][0])[tid] = 0.f;
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.wfull[s])), "r"(1));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.wempty[s])),
                   "r"(32 * kTeam));  // every lane of the consuming team
    }
    // a slot is filled by the x warps of its chunk parity that have batch rows (the others
    // return at once); with a plane, by one bulk-copy transaction
    const int xlive = min((p.B + kq_xrows<NT>() - 1) / kq_xrows<NT>(), kq_xwarps<NT>() / 2);
    for (int f = 0; f < kFS; ++f) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.ffull[f])),
                   "r"(p.xp ? 1 : 32 * xlive));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.fempty[f])),
                   "r"(32 * kTeam));
    }
    for (int w = 0; w < kTeam; ++w)
      for (int k = 0; k < 2; ++k) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.pfull[w][k])), "r"(1));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(&sm.pempty[w][k])),
                     "r"(1));
      }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kq_copy_warp<NT>()) {
    if (lane == 0) kq_copies<TYPE, NT>(sm, p);
  } else if (warp >= kCompute) {  // x warp (row slice, chunk parity)
    const int xw = kq_xwarp_index(warp);
    if (!p.xp)
      kq_stage_x<TYPE, NT>(sm, p, lane, xw >> 1, xw & 1);
    else if ((xw >> 1) == 0 && lane == 0)
      kq_copy_plane<TYPE, NT>(sm, p, xw & 1);
  } else {
    const int team = warp / kTeam, wq = warp % kTeam;
    // Lane (g, t) feeds column g of each n8 tile, i.e. batch row 4i + g/2.  Lanes of absent
    // batch rows read lane (g mod 2, t)'s fragment instead: the copy only feeds accumulator
    // columns that are never stored.
    int fl[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) fl[i] = 4 * i + (g >> 1) < p.B ? lane : (lane & 7);
    // ring positions of global chunk index `at` (this team's chunks of each unit)
    RingPos<NS> wpos;
    RingPos<kFS> fpos;
    int at = 0;
    int base = 0;
    Unit un;
    for (int u = 0; unit_at(p, u, un); ++u) {
      const int nch = un.ce - un.cb;
      float tot[2][NT];
#pragma unroll
      for (int i = 0; i < NT; ++i) tot[0][i] = tot[1][i] = 0.f;
      // chunks of global index parity `team`: exactly the chunks that the x warps of that
      // parity convert, so each team and its x warps form one in-order pipeline (with the
      // unit-local parity, odd chunk counts let the two pipelines wait on each other)
      for (int j = (team + base) & 1; j < nch; j += 2) {
        wpos.advance(base + j - at);
        fpos.advance(base + j - at);
        at = base + j;
        const int s = wpos.s, fs = fpos.s;
        mbar_wait(sa(&sm.wfull[s]), wpos.ph, p.status, 32);
        if constexpr (TYPE == MQ_Q6_K)
          kq_chunk_q6k<NT>(sm, s, fs, fpos.ph, warp, wq, lane, p.status, fl, tot);
        else
          kq_chunk_q4k<TYPE, NT>(sm, s, fs, fpos.ph, warp, wq, lane, p.status, fl, tot);
        mbar_arrive(sa(&sm.fempty[fs]));  // each lane: done with the slot
      }
      base += nch;
      // team 1 hands its partial sums to the team-0 warp of the same rows
      const int par = u & 1;
      if (team == 1) {
        if (u >= 2) mbar_wait(sa(&sm.pempty[wq][par]), ((u >> 1) - 1) & 1, p.status, 36);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          sm.xch[par][wq][lane][2 * i] = tot[0][i];
          sm.xch[par][wq][lane][2 * i + 1] = tot[1][i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sa(&sm.pfull[wq][par]));
        continue;
      }
      mbar_wait(sa(&sm.pfull[wq][par]), (u >> 1) & 1, p.status, 37);
      float res[2][NT];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        res[0][i] = tot[0][i] + sm.xch[par][wq][lane][2 * i];
        res[1][i] = tot[1][i] + sm.xch[par][wq][lane][2 * i + 1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(sa(&sm.pempty[wq][par]));
      const int64_t rA = un.group * kRows + 16 * wq + g;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        const int b = t + 4 * i;
        if (b < p.B) kq_store(p, b, rA, res[0][i], res[1][i]);
      }
    }
  }
}

template <int TYPE, int NT>
mq_status kq_launch_one(const KqArgs &a, unsigned grid, cudaStream_t s, const char *name) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(test_fail_launch() ? 0u : grid, 1, 1);
  cfg.blockDim = dim3(kq_threads<NT>(), 1, 1);
  cfg.dynamicSmemBytes = kq_smem_bytes<TYPE, NT>();
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, matvec_kq_kernel<TYPE, NT>, a);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // the refused launch leaves no error behind for later calls
    return fail(MQ_ERR_LAUNCH, "launch of %s (grid %u) failed: %s", name, cfg.gridDim.x,
                cudaGetErrorName(e));
  }
  return MQ_OK;
}

template <int TYPE, int NT>
mq_status kq_optin(const DeviceState *st, const char *name) {
  constexpr size_t smem = kq_smem_bytes<TYPE, NT>();
  static_assert(smem <= 227 * 1024, "matvec_kq shared memory exceeds the per-CTA limit");
  if ((int)smem > st->smem_optin)
    return fail(MQ_ERR_LAUNCH, "%s needs %zu bytes of shared memory; the device allows %d", name,
                smem, st->smem_optin);
  cudaError_t e = cudaFuncSetAttribute(matvec_kq_kernel<TYPE, NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "smem opt-in of %s (%zu bytes) refused: %s", name, smem,
                cudaGetErrorName(e));
  return MQ_OK;
}

}  // namespace

mq_status init_matvec_kq(DeviceState *st) {
  mq_status s;
  if ((s = kq_optin<MQ_Q4_K, 1>(st, "matvec_kq_kernel<Q4_K>")) != MQ_OK) return s;
  if ((s = kq_optin<MQ_Q4_K, 2>(st, "matvec_kq_kernel<Q4_K>")) != MQ_OK) return s;
  if ((s = kq_optin<MQ_Q5_K, 1>(st, "matvec_kq_kernel<Q5_K>")) != MQ_OK) return s;
  if ((s = kq_optin<MQ_Q5_K, 2>(st, "matvec_kq_kernel<Q5_K>")) != MQ_OK) return s;
  if ((s = kq_optin<MQ_Q6_K, 1>(st, "matvec_kq_kernel<Q6_K>")) != MQ_OK) return s;
  return kq_optin<MQ_Q6_K, 2>(st, "matvec_kq_kernel<Q6_K>");
}

// The persistent kernel takes weights of at least SMs / 2 row groups (its grid: one CTA per
// group up to one per SM); narrower weights need a K split, which matvec.cu's kernel does.
// The choice depends on N and the device only, never on B.
bool matvec_kq_applies(int64_t N, int sms) { return (N + kRows - 1) / kRows * 2 >= sms; }

mq_status launch_matvec_kq(const mq_weight *W, const float *x, float *y, int B, cudaStream_t s,
                           const DeviceState *st) {
  KqArgs a;
  a.xp = nullptr;
  a.q = W->q;
  a.x = x;
  a.y = y;
  a.N = W->N;
  a.K = W->K;
  a.B = B;
  a.nchunk = (int)(W->K / kChunk);
  a.groups = (W->N + kRows - 1) / kRows;
  const unsigned grid = (unsigned)(a.groups < st->sms ? a.groups : st->sms);
  a.swiglu = W->ffn_gu;
  a.status = st->status;
  const bool two = B > 4;
  if (!two) {
    switch (W->type) {
      case MQ_Q4_K: return kq_launch_one<MQ_Q4_K, 1>(a, grid, s, "matvec_kq_kernel<Q4_K>");
      case MQ_Q5_K: return kq_launch_one<MQ_Q5_K, 1>(a, grid, s, "matvec_kq_kernel<Q5_K>");
      default: return kq_launch_one<MQ_Q6_K, 1>(a, grid, s, "matvec_kq_kernel<Q6_K>");
    }
  }
  // Q4_K / Q5_K with two tiles (B = 5..8): x converted once into the activation fragment
  // plane, a per-call buffer from the device's stream-ordered pool (freed in stream order
  // after the matvec; in a captured graph, an allocation node and a free node), instead of by
  // the four x warps of every CTA, which also form the min-term sums of these types.
  // Measured at 18944 x 3584: Q4_K B = 5 / 8 16.6 / 17.9 -> 15.0 / 15.0 us, Q5_K 18.9 / 20.3
  // -> 17.9 / 18.0 us.  Where the x warps' work is lighter, the plane's extra launch costs
  // more than it saves: Q6_K B = 5 / 8 17.5 / 18.6 -> 19.0 / 19.0 us; with one tile (B <= 4)
  // Q4_K B = 3 / 4 11.9 / 12.6 -> 13.4 / 13.0 us; the split-K kernel of narrow weights
  // (Q6_K 3584 x 18944) B = 3..5 1.5-1.9 us slower, B = 8 23.6 -> 23.3 us.  Without the
  // pool, or if the allocation is refused, the x warps convert x themselves (the same
  // fragments).
  uint8_t *xp = nullptr;
  if (st->xpool && W->type != MQ_Q6_K && !test_no_xplane()) {
    if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&xp), xplane_bytes(B, W->K), st->xpool,
                                s) != cudaSuccess) {
      (void)cudaGetLastError();
      xp = nullptr;
    } else {
      const mq_status r = launch_xplane(x, B, W->K, xp, s);
      if (r != MQ_OK) {
        (void)cudaFreeAsync(xp, s);
        return r;
      }
    }
  }
  a.xp = xp;
  mq_status r;
  switch (W->type) {
    case MQ_Q4_K: r = kq_launch_one<MQ_Q4_K, 2>(a, grid, s, "matvec_kq_kernel<Q4_K>"); break;
    case MQ_Q5_K: r = kq_launch_one<MQ_Q5_K, 2>(a, grid, s, "matvec_kq_kernel<Q5_K>"); break;
    default: r = kq_launch_one<MQ_Q6_K, 2>(a, grid, s, "matvec_kq_kernel<Q6_K>"); break;
  }
  if (xp) {
    const cudaError_t e = cudaFreeAsync(xp, s);
    if (e != cudaSuccess && r == MQ_OK)
      r = fail(MQ_ERR_CUDA, "release of the activation fragment plane failed: %s",
               cudaGetErrorName(e));
  }
  return r;
}

}  // namespace mq
