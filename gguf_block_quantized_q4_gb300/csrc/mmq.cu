// mmq.cu -- prefill MMQ on the 5th-generation tensor cores (tcgen05):
//   y[m][n] = sum_b s[m][b] * (d[n][b] * D[m][n][b] - dmin_term[n][b] * S[m][b])
// with D the exact integer dot of 32-element block b ("minfer CUDA Backend
// Design" §4.4: the int8 MMQ path for prefill; §4.7: decoded f32 scale planes
// for the per-block epilogue).
//
// Exactness.  Both operands are integers carried in f16 (q in [-127, 127];
// W_int = Q8_0 q, Q4_0 n - 8, Q5_0 q - 16, Q4_1 / Q5_1 q, Q4_K sc_j*nib <= 945,
// Q5_K sc_j*q <= 1953, Q6_K v = sc*(q-32) as even part + odd part, each exact).  Every product is exact and every partial sum of a
// block stays below 2^24 (|D| <= 32*127*4097 < 16.7M), so tcgen05.mma kind::f16
// accumulating one block in f32 yields the integer dot exactly.  sm_103a has
// no integer tcgen05 kind, and f16 integers are exact, so this is the int8
// contraction on the tensor pipe.
//
// Structure.  Output tiles of 128 x 128; one persistent CTA per SM takes tiles
// blockIdx.x, + gridDim.x, ... (m-tiles fastest, so CTAs running together share
// each weight tile through L2 and the weights stream from HBM about once).  The K
// loop runs over pairs of 32-element blocks (64 K per pipeline stage).  20 warps:
//   warpgroup 0 (registers lowered to 32 with setmaxnreg):
//     warp 0    TMA producer: per pair, the activation tile (128 x 64 f16) and the
//               weight tile(s) (128 x 64 f16; Q6_K also the odd part) into a
//               shared-memory ring (128-byte swizzle), mbarrier tx-count; per 8
//               blocks, one 2-D box each of the tile's row scales s and column
//               scales d (8 blocks x 128) into a 2-slot ring.
//     warps 1,2 MMA issuers (warp 1 also owns TMEM: 512 columns = two pairs of
//               128-column f32 accumulators).  The accumulator uses alternate
//               between them (issuer i, accumulator pair i): per pair of blocks
//               4 (Q6_K: 8) tcgen05.mma M=128 N=128 K=16, one block per
//               accumulator, then tcgen05.commit to the stage's "empty" and the
//               accumulator pair's "full" barrier.  Two issuers keep the tensor
//               pipe fed while the other one waits.  Each issuer owns half of the
//               ring (stages i, i+2, ...) and the producer fills the stages in the
//               order of the uses, so every stage is consumed by one issuer, round
//               after round: a parity wait never sees a phase two rounds old.
//   warpgroups 1-4 (registers raised to 112): 16 epilogue warps.  Warp w reads
//               TMEM lanes 32*(w%4).. (its 32 rows) and 32 of the 128 columns;
//               per block it loads the accumulator (tcgen05.ld) and promotes it
//               in registers with packed f32x2 multiply-adds:
//                 Q8_0, Q4_1: y += (s_m * d_n) * D
//                 Q4_K, Q6_K: a = s_m * D (first block of a super-block), then
//                             a += s_m * D; per super-block y += d_n * a
//               and frees the accumulator pair after its second block.
//   Q4_K weights registered without the f16 plane (MQ_REG_MMQ_FROM_DECODE_PLANE) run a
//   24-warp form: the producer bulk-copies the decode plane's 128-row x 144-byte tiles (one
//   per 256-K chunk, two chunks ahead, three slots) instead of the weight tiles, and a sixth
//   warpgroup of four decoder warps writes each stage's weight tile, the same f16 integers
//   sc_j*nib, into the ring in the layout TMA gives the plane's tiles; 4 ring stages; registers
//   80 at launch, 32 / 104 / 32 after setmaxnreg.
// Min term (Q4_K: dmin*m_j per sub-block, subtracted; Q4_1: the block min m, added, so
// its plane holds -m).  sum_b (s*S)_m,b * (dmin*m_j)_n,b is a product of rank K/32;
// the tensor cores form it once per tile, after the main loop, from three f16
// products per block (row side hi | hi | lo of (s*S)/u_m, column side
// hi | lo | hi of (dmin*m_j)/v_n, u and v powers of two that keep both in f16
// range; 22 significant bits), staged through the same ring as two accumulator
// uses, one per issuer.  The epilogue adds y -= u_m * v_n * C_min before the
// store, so the per-block work is a single multiply-add.
// All mbarrier waits are bounded (2 s by %globaltimer); an expired wait writes
// MQ_ERR_TIMEOUT into the device status word read by mq_stream_status.
#include <cstddef>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "quant_row.cuh"

namespace mq {
namespace {

constexpr int TM = 128, TN = 128, TK = 32;
constexpr int PK = 2 * TK;              // K per pipeline stage (a pair of blocks)
constexpr int NEPI = 16;                // epilogue warps: 4 per TMEM lane quarter
constexpr int EC = TN * 4 / NEPI;       // accumulator columns per epilogue thread (32)
constexpr int NTHR = 32 * (4 + NEPI);   // 640 threads
// Q4_K from its decode-plane tiles: a sixth warpgroup of four weight decoders, 768 threads
constexpr int NTHR_PW = NTHR + 128;
template <bool PW>
__host__ __device__ constexpr int nthr() {
  return PW ? NTHR_PW : NTHR;
}
constexpr int kPkBytes = 128 * 144;     // one Q4_K decode-plane tile: 128 rows, one 256-K chunk
constexpr int kPkSlots = 3;             // chunk slots: copies run two chunks ahead
constexpr uint32_t TMEM_COLS = 512;     // accumulator pair i at columns 256*i .. +256
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kTestWaitNs = 1000000ull;
constexpr int kTileBytes = TM * PK * 2;  // 16 KB per operand tile and stage
// launch: 640 threads x 96 registers = 61440; after setmaxnreg the control
// warpgroup holds 128 x 32 and the four epilogue warpgroups 512 x 112 = 61440.
// With the decoder warpgroup: 768 x 80 = 61440 = 128 x 32 (control) + 512 x 104
// (epilogue) + 128 x 32 (decoders).  setmaxnreg.inc waits until the registers are free, so
// the split must fit the launch exactly as compiled: the host checks the kernel's register
// count against reg_launch before the first launch.
constexpr int kRegCtl = 32;
template <bool PW>
__host__ __device__ constexpr int reg_launch() {
  return PW ? 80 : 96;
}
template <bool PW>
__host__ __device__ constexpr int reg_epi() {
  return PW ? 104 : 112;
}
static_assert(128 * kRegCtl + 512 * reg_epi<false>() <= NTHR * reg_launch<false>(),
              "register split exceeds the launch");
static_assert(128 * kRegCtl + 512 * reg_epi<true>() + 128 * kRegCtl <=
                  NTHR_PW * reg_launch<true>(),
              "register split exceeds the launch");
static_assert(NTHR * reg_launch<false>() <= 65536 && NTHR_PW * reg_launch<true>() <= 65536,
              "launch registers exceed the SM");

template <int TYPE, bool PW = false>
constexpr int stages() {  // 192 KB of operand ring (128 KB beside the decode-plane tiles)
  return (TYPE == MQ_Q6_K || PW) ? 4 : 6;
}

struct TcArgs {
  const float *urow;    // [mt] min-term row factors u_m
  const float *vcol;    // [np] min-term column factors v_n
  float *y;             // [M][N]
  int32_t *D;           // [M][N][nb] (block-dot mode)
  int64_t M, N, mt, np;
  int nb;
  int ntm, ntiles;      // output tiles: ntm along M (fastest), ntiles in all
  int mt0;              // first M-tile (a call over M-tiles mt0 .. mt0 + ntm - 1)
  int nms;              // ring stages of the min-term GEMM (3*nb/64 rounded up), or 0
  int *status;
  int debug_expire;
  int swiglu;           // fused gate/up weight: y[m][n'] = silu(gate col) * (its up col), N / 2 wide
  const uint8_t *wq;    // Q4_K decode plane (tiles of 128 rows x 144 bytes per 256-K chunk)
  int nchk;             // its chunks per row group (K / 256)
};

// Fused quantisation (x non-null): the CTAs first quantise the rows of x into xq.
struct QfArgs {
  const float *x;
  uint8_t *xq;
  unsigned *sync;       // the grid barrier's two words inside xq
};

// Arrays that some block types do not need take (almost) no space; every slot
// array starts on a 128-byte boundary (bulk-copy destinations and float4 reads).
template <class T, int N, int W>
struct __align__(128) Slots {
  T v[N][W];
};
template <class T, int W>
struct __align__(128) Slots<T, 0, W> {
  T v[1][1];  // never indexed
};

template <int TYPE, bool PW = false>
struct __align__(1024) TcSmem {
  static constexpr int NST = stages<TYPE, PW>();
  static constexpr bool ODD = TYPE == MQ_Q6_K;
  static constexpr bool MIN = TYPE == MQ_Q4_K || TYPE == MQ_Q4_1;
  __half a[NST][TM * PK];
  __half b[NST][TN * PK];
  Slots<__half, ODD ? NST : 0, TN * PK> b2;
  alignas(128) float gsx[2][8][TM];     // per group slot: row scales s
  alignas(128) float gd[2][8][TN];      // column scales d
  Slots<uint8_t, PW ? kPkSlots : 0, kPkBytes> pk;  // Q4_K decode-plane tiles (chunk slots)
  uint64_t full[NST], empty[NST], tfull[2], tempty[2], gfull[2], gempty[2], pfull[kPkSlots],
      pempty[kPkSlots], never;
  uint32_t tmem;
};

template <int TYPE, bool PW = false>
constexpr bool smem_layout_ok() {
  using S = TcSmem<TYPE, PW>;
  return offsetof(S, a) % 1024 == 0 && offsetof(S, b) % 1024 == 0 &&
         offsetof(S, b2) % 1024 == 0 && offsetof(S, gsx) % 128 == 0 &&
         offsetof(S, gd) % 128 == 0 && offsetof(S, pk) % 128 == 0 && offsetof(S, full) % 8 == 0;
}
static_assert(smem_layout_ok<MQ_Q8_0>() && smem_layout_ok<MQ_Q4_K>() &&
                  smem_layout_ok<MQ_Q6_K>() && smem_layout_ok<MQ_Q4_1>() &&
                  smem_layout_ok<MQ_Q4_K, true>(),
              "TMA tiles need 1024-byte, bulk copies and float4 reads 16-byte alignment");

__device__ __forceinline__ uint32_t sa(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// A probe that may suspend the thread for the system-dependent time limit while
// the phase is incomplete.
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
// Bounded wait on an mbarrier phase.  On expiry: record (timeout, site) in the
// status word and return false; the caller carries on so the kernel ends.  A wait that has
// lasted kAbandonNs while the status word already holds an error gives up at once, so that
// after one expiry the kernel's remaining waits do not each run to the limit (no wait of a
// working pipeline lasts that long; the test hook's 1 ms expiry delays the others by about
// 1 ms, and they still complete).
constexpr uint64_t kAbandonNs = 10000000ull;
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, int *status, int site,
                                          uint64_t limit_ns) {
  if (mbar_try(a, parity)) return true;
  const uint64_t t0 = gtime();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      if (mbar_try(a, parity)) return true;
    }
    const uint64_t dt = gtime() - t0;
    if (dt > limit_ns) {
      if (atomicCAS(status, 0, kStatusTimeout) == 0) atomicExch(status + 1, site);
      return false;
    }
    if (dt > kAbandonNs && *reinterpret_cast<volatile int *>(status) != 0) return false;
  }
}
// Grid-wide barrier of the fused quantise + MMQ (all CTAs co-resident: cooperative launch),
// run by one thread per CTA after the CTA's writers have fenced their writes and met at a
// CTA barrier.  sync[0] counts arrivals, sync[1] is the generation; the last CTA to arrive
// resets the count and advances the generation, so the count is zero again when the
// barrier opens.  The wait is bounded (expiry: status site 8, and the kernel carries on).
__device__ __forceinline__ void grid_wait(unsigned *sync, unsigned G, int *status) {
  unsigned *cnt = sync, *gen = sync + 1;
  unsigned g;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(gen) : "memory");
  __threadfence();
  if (atomicAdd(cnt, 1u) == G - 1) {
    atomicExch(cnt, 0u);
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(gen), "r"(g + 1u) : "memory");
  } else {
    const uint64_t t0 = gtime();
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(gen) : "memory");
      if (v != g) break;
      if (gtime() - t0 > kWaitNs) {
        if (atomicCAS(status, 0, kStatusTimeout) == 0) atomicExch(status + 1, 8);
        break;
      }
    }
  }
  __threadfence();
}

// Fused prologue: the 512 epilogue threads form kQGroups groups of kQThreads, each
// quantising its own rows (row group * gridDim.x + blockIdx.x, then + gridDim.x * kQGroups,
// ...: the rows are dealt to the CTAs first); named barriers: 1..kQGroups per group,
// kBarEpi among the epilogue threads, kBarAll for the whole CTA (the control warps wait
// there until the grid barrier has opened).
constexpr int kQThreads = 128, kQGroups = 4;
constexpr int kBarEpi = 14, kBarAll = 15;

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// One integer weight pair sc * n_lo, sc * n_hi from the nibbles at bits sh and sh + 16 of
// w: 1024 + n is an f16 formed by one bit operation, and fma(1024 + n, sc, -1024 sc) rounds
// once, to the exact sc * n (<= 945).
__device__ __forceinline__ uint32_t q4k_pair(uint32_t w, int sh, __half2 sc, __half2 msc) {
  const uint32_t v = ((w >> sh) & 0x000F000Fu) | 0x64006400u;
  const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&v), sc, msc);
  return *reinterpret_cast<const uint32_t *>(&r);
}
// (sc, sc) and (-1024 sc, -1024 sc) as f16 pairs, sc the byte of scp at selector sel
__device__ __forceinline__ void q4k_scale_pair(uint32_t scp, uint32_t sel, __half2 &sc,
                                               __half2 &msc) {
  const uint32_t v = __byte_perm(scp, 0u, sel) | 0x64006400u;  // 1024 + sc in both halves
  sc = __hsub2(*reinterpret_cast<const __half2 *>(&v), __half2half2(__ushort_as_half(0x6400)));
  msc = __hmul2(sc, __half2half2(__ushort_as_half(0xE400)));  // * -1024
}
// Weight tile of one pipeline stage from a Q4_K decode-plane tile in shared memory: quarter
// qt of the 256-element chunk (elements 64 qt .. 64 qt + 63, sub-blocks 2 qt and 2 qt + 1)
// for rows r0 .. r0 + 31, as the f16 integers sc_j * nib in the K-major 128-byte-swizzled
// layout the MMA reads (the layout a TMA box of the f16 plane lands in: row r at 128 r,
// 16-byte unit j of the row at unit j ^ (r % 8)).  A decode-plane row is the 16-byte block
// header (d, dmin, 12 scale bytes), then four 32-byte groups t whose word 2 qt + u holds qs
// bytes 32 qt + 16 u + 4 t + (0, 2, 1, 3): low nibbles are elements 16 u + 4 t .. + 3 of
// the quarter (sub-block 2 qt), high nibbles the same + 32 (sub-block 2 qt + 1).
// Lane (r8, u, rh): rows r0 + 8 (rh + 2 k) + r8 for k < 2; the 8 lanes of each store phase
// write 8 rows' same unit, distinct banks after the swizzle.
__device__ __forceinline__ void q4k_stage_decode(const uint8_t *pk, __half *b, int qt, int r0,
                                                 int lane) {
  const int r8 = lane & 7, u = (lane >> 3) & 1, rh = lane >> 4;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = r0 + 8 * (rh + 2 * k) + r8;
    const uint8_t *row = pk + r * 144;
    // the quarter's two 6-bit sub-block scales (scale bytes s0..s11 at row + 4): for
    // j < 4, s_j & 63; for j >= 4, (s_{j+4} & 15) | (s_{j-4} >> 6) << 4
    const uint32_t s03 = *reinterpret_cast<const uint32_t *>(row + 4);
    uint32_t scp;
    if (qt < 2) {
      scp = (s03 >> (16 * qt)) & 0x3F3Fu;
    } else {
      const int sh = 16 * (qt - 2);
      const uint32_t s811 = *reinterpret_cast<const uint32_t *>(row + 12);
      scp = ((s811 >> sh) & 0x0F0Fu) | (((s03 >> sh) & 0xC0C0u) >> 2);
    }
    __half2 slo, mlo, shi, mhi;
    q4k_scale_pair(scp, 0x4040u, slo, mlo);
    q4k_scale_pair(scp, 0x4141u, shi, mhi);
    const uint8_t *wp = row + 16 + 8 * qt + 4 * u;
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) w[t] = *reinterpret_cast<const uint32_t *>(wp + 32 * t);
    uint8_t *brow = reinterpret_cast<uint8_t *>(b) + r * 128;
    const int sw = r & 7;
#pragma unroll
    for (int tp = 0; tp < 2; ++tp) {
      const uint32_t wa = w[2 * tp], wb = w[2 * tp + 1];
      // elements 16 u + 8 tp .. + 7 (unit 2 u + tp), then the same + 32 (unit 4 + 2 u + tp)
      *reinterpret_cast<uint4 *>(brow + (((2 * u + tp) ^ sw) << 4)) =
          make_uint4(q4k_pair(wa, 0, slo, mlo), q4k_pair(wa, 8, slo, mlo),
                     q4k_pair(wb, 0, slo, mlo), q4k_pair(wb, 8, slo, mlo));
      *reinterpret_cast<uint4 *>(brow + (((4 + 2 * u + tp) ^ sw) << 4)) =
          make_uint4(q4k_pair(wa, 4, shi, mhi), q4k_pair(wa, 12, shi, mhi),
                     q4k_pair(wb, 4, shi, mhi), q4k_pair(wb, 12, shi, mhi));
    }
  }
}
// K-major operand in the 128-byte swizzle layout TMA writes: 8-row groups of
// 1024 bytes (SBO), leading offset unused (16), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3fff) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// columns j, j+1 of a tcgen05.ld result as an f32 pair
__device__ __forceinline__ float2 pair(const uint32_t *r, int j) {
  return make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define TC_LD32(taddr, r)                                                                     \
  asm volatile(                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"     \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),         \
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),         \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),         \
        "=r"(r[31])                                                                           \
      : "r"(taddr))

template <int TYPE, bool DOTS, bool QF = false, bool PW = false>
__global__ void __launch_bounds__(nthr<PW>(), 1)
    mmq_tc_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tW,
                  const __grid_constant__ CUtensorMap tW2, const __grid_constant__ CUtensorMap tAm,
                  const __grid_constant__ CUtensorMap tBm, const __grid_constant__ CUtensorMap tSx,
                  const __grid_constant__ CUtensorMap tD, const TcArgs p, const QfArgs qf) {
  using Sm = TcSmem<TYPE, PW>;
  static_assert(!PW || TYPE == MQ_Q4_K, "decode-plane weight tiles are Q4_K's");
  constexpr int NT = nthr<PW>();
  constexpr int NST = Sm::NST, SR = NST / 2;  // SR ring stages per MMA issuer
  static_assert(NST % 2 == 0, "the ring is split between two issuers");
  constexpr bool ODD = Sm::ODD, MIN = Sm::MIN;
  // per-block epilogue (a scale d per 32-element block): Q8_0, and Q4_1 with its min term
  constexpr bool PB = TYPE == MQ_Q8_0 || TYPE == MQ_Q4_1;
  extern __shared__ uint8_t smem_raw[];
  // aligned by an offset into the __shared__ array, so the compiler keeps knowing that
  // every member lives in shared memory (plain loads become LDS, addresses stay 32-bit)
  Sm &sm = *reinterpret_cast<Sm *>(
      smem_raw + ((1024u - (uint32_t)__cvta_generic_to_shared(smem_raw)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = p.nb, npairs = (nb + 1) / 2, ngroups = (nb + 7) >> 3;
  // Accumulator uses of a tile, in order: pair pr = use pr, then the min-term GEMM
  // as two uses (npairs + j, j < 2), one per issuer, use j taking min-term stages j,
  // j + 2, ... (use 1 has none when there is one stage).  The CTA is persistent: it
  // takes tiles blockIdx.x, + gridDim.x, ... and every ring, accumulator and group phase
  // counts on across its tiles (global use U = tl * nuse + u, global group
  // G = tl * ngroups + g for the CTA's tl-th tile).  For the K-quants npairs is a
  // multiple of 4, so nuse is even and pair pr of every tile uses accumulator pr % 2.
  const int nms = (MIN && !DOTS) ? p.nms : 0, nmu = nms > 0 ? 2 : 0, nuse = npairs + nmu;


  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      // with decode-plane weights a stage is full when its activation tile has landed and
      // the four decoder warps have written its weight tile
      mbar_init(sa(&sm.full[s]), PW ? 5 : 1);
      mbar_init(sa(&sm.empty[s]), 1);
    }
    for (int t = 0; t < kPkSlots; ++t) {
      mbar_init(sa(&sm.pfull[t]), 1);
      mbar_init(sa(&sm.pempty[t]), 4);  // one arrival per decoder warp
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(sa(&sm.tfull[t]), 1);
      // every epilogue thread arrives on its own: no election or warp sync on the way
      mbar_init(sa(&sm.tempty[t]), 32 * NEPI);
      mbar_init(sa(&sm.gfull[t]), 1);
      mbar_init(sa(&sm.gempty[t]), 32 * NEPI);
    }
    mbar_init(sa(&sm.never), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     sa(&sm.tmem)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  // (launched with programmatic stream serialisation outside the fused form) a following
  // kernel may launch at once; the producer waits for the previous grid before its first
  // load, and everything that reads xq or writes the outputs follows its loads
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- weight decoders (Q4_K from its decode plane): decoder warp dw writes rows
  // 32 dw .. 32 dw + 31 of every stage's weight tile.  They follow the producer's fill order;
  // a stage's tile is written once the MMA has released the stage (its previous round), and
  // the chunk slot is released after the chunk's fourth quarter.  Min-term fills (TMA only)
  // get the decoders' arrivals too, so that every fill completes the same count.
  auto decode_weights = [&](int dw) {
    int c0 = 0, c1 = 0;
    for (int t = blockIdx.x, tl = 0; t < p.ntiles; t += gridDim.x, ++tl) {
      for (int f = 0; f < npairs + nms; ++f) {
        const int pr = f < npairs ? f : -1;
        const int i = (tl * nuse + (f < npairs ? f : npairs + ((f - npairs) & 1))) & 1;
        const int c = i ? c1++ : c0++, s = i + 2 * (c % SR), q = c / SR;
        if (q >= 1) mbar_wait(sa(&sm.empty[s]), (q - 1) & 1, p.status, 11, kWaitNs);
        const int cg = tl * p.nchk + (pr >> 2);  // chunk in this CTA's sequence
        const int ps = cg % kPkSlots;            // its slot, round cg / kPkSlots
        if (pr >= 0) {
          if ((pr & 3) == 0)
            mbar_wait(sa(&sm.pfull[ps]), (cg / kPkSlots) & 1, p.status, 12, kWaitNs);
          q4k_stage_decode(sm.pk.v[PW ? ps : 0], sm.b[s], pr & 3, 32 * dw, lane);
          // the MMA (async proxy) reads what these generic stores wrote
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(sa(&sm.full[s]));
          if (pr >= 0 && (pr & 3) == 3) mbar_arrive(sa(&sm.pempty[ps]));
        }
      }
    }
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegCtl));
    if constexpr (QF) {  // wait until every CTA's rows are in xq (epilogue warps, below)
      asm volatile("bar.sync %0, %1;" ::"n"(kBarAll), "n"(NT) : "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");  // before the TMA reads of xq
    }
    if (warp == 0 && lane == 0) {  // ---- TMA producer (operands and group scales)
      const uint32_t bytes = (PW ? 1 : ODD ? 3 : 2) * kTileBytes;
      // Decode-plane weights: chunk cg of this CTA's sequence (its tile cg / nchk, chunk
      // cg % nchk of that tile's row group) goes to slot cg % kPkSlots with one bulk copy; the
      // first kPkSlots go out before the wait for the previous kernel, chunk cg + 2 when the
      // producer starts chunk cg, once chunk cg - 1 (the slot's previous chunk) is decoded.
      const int nchunks = PW && (int)blockIdx.x < p.ntiles
                              ? ((p.ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) * p.nchk
                              : 0;
      auto chunk_copy = [&](int cg) {
        const int tt = (int)blockIdx.x + (cg / p.nchk) * (int)gridDim.x;
        const uint8_t *src = p.wq + (int64_t(tt / p.ntm) * p.nchk + cg % p.nchk) * kPkBytes;
        const int ps = cg % kPkSlots;
        mbar_expect_tx(sa(&sm.pfull[ps]), kPkBytes);
        bulk_copy(sa(sm.pk.v[PW ? ps : 0]), src, kPkBytes, sa(&sm.pfull[ps]));
      };
      if constexpr (PW) {
        for (int cg = 0; cg < kPkSlots && cg < nchunks; ++cg) chunk_copy(cg);
      }
      // Registered weights are never written by a kernel: the weight tiles of the first
      // tile's first kRamp fills (fill f of the first tile uses ring stage f) go out before
      // the wait for the previous kernel, the activation tiles of those stages after it.
      // The rest of the first ring round is ramped: stage s is filled once stage s - kRamp
      // has landed, so that every SM's first stages are not queued behind the whole first
      // round of all SMs (Q4_K 512 x 18944 x 3584: 109.5 -> 108.9 us; a ramp of 2 109.3).
      constexpr int kRamp = 3;
      int pre = 0;
      if constexpr (!QF && !PW) {
        if (blockIdx.x < p.ntiles) {
          const int n0 = (blockIdx.x / p.ntm) * TN;
          pre = npairs < kRamp ? npairs : kRamp;
          for (int f = 0; f < pre; ++f) {
            mbar_expect_tx(sa(&sm.full[f]), bytes);
            tma_2d(sa(sm.b[f]), &tW, f * PK, n0, sa(&sm.full[f]));
            if constexpr (ODD) tma_2d(sa(sm.b2.v[ODD ? f : 0]), &tW2, f * PK, n0, sa(&sm.full[f]));
          }
        }
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");  // xq comes from the previous kernel
      // Fills in the order of the accumulator uses.  Global use U belongs to issuer U % 2,
      // whose c-th stage is ring stage (U % 2) + 2 * (c % SR), round c / SR.
      int c0 = 0, c1 = 0;
      for (int t = blockIdx.x, tl = 0; t < p.ntiles; t += gridDim.x, ++tl) {
        const int m0 = (p.mt0 + t % p.ntm) * TM, n0 = (t / p.ntm) * TN;
        for (int f = 0; f < npairs + nms; ++f) {
          const int pr = f < npairs ? f : -1;
          const int i = (tl * nuse + (f < npairs ? f : npairs + ((f - npairs) & 1))) & 1;
          const int c = i ? c1++ : c0++, s = i + 2 * (c % SR), q = c / SR;
          if (!DOTS && pr >= 0 && (pr & 3) == 0) {  // group of 8 blocks
            const int g = pr >> 2, G = tl * ngroups + g, slot = G & 1;
            if (G >= 2)
              mbar_wait(sa(&sm.gempty[slot]), ((G >> 1) - 1) & 1, p.status, 5, kWaitNs);
            // the group's 8 x 128 row scales and 8 x 128 column scales, one box each
            // (blocks past the last read as 0)
            mbar_expect_tx(sa(&sm.gfull[slot]), 2u * 8u * 128u * 4u);
            tma_2d(sa(sm.gsx[slot][0]), &tSx, m0, 8 * g, sa(&sm.gfull[slot]));
            tma_2d(sa(sm.gd[slot][0]), &tD, n0, 8 * g, sa(&sm.gfull[slot]));
          }
          if (q >= 1) mbar_wait(sa(&sm.empty[s]), (q - 1) & 1, p.status, 1, kWaitNs);
          else if (tl == 0 && s >= kRamp)  // first round: after stage s - kRamp has landed
            mbar_wait(sa(&sm.full[s - kRamp]), 0u, p.status, 10, kWaitNs);
          if (pr < 0) {  // min-term operands: 64 columns of the [hi|hi|lo] x [hi|lo|hi] planes
            mbar_expect_tx(sa(&sm.full[s]), 2 * kTileBytes);
            tma_2d(sa(sm.a[s]), &tAm, (f - npairs) * PK, m0, sa(&sm.full[s]));
            tma_2d(sa(sm.b[s]), &tBm, (f - npairs) * PK, n0, sa(&sm.full[s]));
            continue;
          }
          if (tl == 0 && f < pre) {  // its weight tiles are in flight already
            tma_2d(sa(sm.a[s]), &tA, pr * PK, m0, sa(&sm.full[s]));
            continue;
          }
          mbar_expect_tx(sa(&sm.full[s]), bytes);
          tma_2d(sa(sm.a[s]), &tA, pr * PK, m0, sa(&sm.full[s]));
          if constexpr (PW) {
            // chunk cg + 2 into the slot of chunk cg - 1
            const int cg = tl * p.nchk + (pr >> 2), cn = cg + kPkSlots - 1;
            if ((pr & 3) == 0 && cg >= 1 && cn < nchunks) {
              mbar_wait(sa(&sm.pempty[cn % kPkSlots]), (cn / kPkSlots - 1) & 1, p.status, 13,
                        kWaitNs);
              chunk_copy(cn);
            }
          } else {
            tma_2d(sa(sm.b[s]), &tW, pr * PK, n0, sa(&sm.full[s]));
          }
          if constexpr (ODD) tma_2d(sa(sm.b2.v[ODD ? s : 0]), &tW2, pr * PK, n0, sa(&sm.full[s]));
        }
      }
    } else if ((warp == 1 || warp == 2) && lane == 0) {  // ---- MMA issuers
      const int i = warp - 1;
      const uint32_t idesc = (1u << 4) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
      const uint32_t acc0 = tmem + (uint32_t)(256 * i);
      int c = 0;  // this issuer's stage count (its half of the ring)
      for (int t = blockIdx.x, tl = 0; t < p.ntiles; t += gridDim.x, ++tl) {
        // this issuer's uses of the tile: U = tl * nuse + u with U % 2 == i
        for (int u = (i - tl * nuse) & 1; u < nuse; u += 2) {
          const int use = (tl * nuse + u) >> 1;  // this issuer's use count
          if (use >= 1) mbar_wait(sa(&sm.tempty[i]), (use - 1) & 1, p.status, 3, kWaitNs);
          if (u >= npairs) {  // min-term use j: stages j, j + nmu, ... into columns acc0 .. +128
            const int ks = (nms - (u - npairs) + 1) >> 1;
            for (int k = 0; k < ks; ++k, ++c) {
              const int s = i + 2 * (c % SR);
              mbar_wait(sa(&sm.full[s]), (c / SR) & 1, p.status, 2, kWaitNs);
              tc_fence_after();
              const uint64_t ad = sdesc(sa(sm.a[s])), bd = sdesc(sa(sm.b[s]));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16(acc0, ad + 2 * kk, bd + 2 * kk, idesc, (k > 0 || kk > 0) ? 1u : 0u);
              mma_commit(sa(&sm.empty[s]));
            }
            mma_commit(sa(&sm.tfull[i]));
            continue;
          }
          const int s = i + 2 * (c % SR);
          mbar_wait(sa(&sm.full[s]), (c / SR) & 1, p.status, 2, kWaitNs);
          ++c;
          tc_fence_after();
          const uint64_t ad = sdesc(sa(sm.a[s])), bd = sdesc(sa(sm.b[s]));
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // block 2*pr + h -> columns acc0 + 128*h
            const uint32_t dt = acc0 + (uint32_t)(128 * h);
            // +2 in the descriptor = +32 bytes = the next 16-element K slice
            mma_f16(dt, ad + 4 * h, bd + 4 * h, idesc, 0u);
            mma_f16(dt, ad + 4 * h + 2, bd + 4 * h + 2, idesc, 1u);
            if constexpr (ODD) {
              const uint64_t od = sdesc(sa(sm.b2.v[ODD ? s : 0]));
              mma_f16(dt, ad + 4 * h, od + 4 * h, idesc, 1u);
              mma_f16(dt, ad + 4 * h + 2, od + 4 * h + 2, idesc, 1u);
            }
          }
          mma_commit(sa(&sm.empty[s]));
          mma_commit(sa(&sm.tfull[i]));
        }
      }
    }
  } else if (PW && warp >= 4 + NEPI) {  // ---- weight decoders (warpgroup 5)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegCtl));
    if constexpr (QF) asm volatile("bar.sync %0, %1;" ::"n"(kBarAll), "n"(NT) : "memory");
    decode_weights(warp - (4 + NEPI));
  } else {  // ---- epilogue warps
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(reg_epi<PW>()));
    if constexpr (QF) {
      // Fused quantisation, with the activation ring (not in use yet) as scratch, then the
      // grid barrier: every row of x is in xq before any CTA's producer reads it.
      static_assert(sizeof(sm.a) >= (kQGroups * kTtCache + NEPI) * sizeof(float),
                    "prologue scratch fits in the activation ring");
      const int et = threadIdx.x - 128, grp = et / kQThreads, tid = et % kQThreads;
      float *scratch = reinterpret_cast<float *>(&sm.a[0][0]);
      float *ttc = scratch + grp * kTtCache, *wmax = scratch + kQGroups * kTtCache + grp * 4;
      const int64_t K = int64_t(nb) * 32;
      const ActLayout L = act_layout(p.M, K);
      for (int64_t m = int64_t(grp) * gridDim.x + blockIdx.x; m < p.M;
           m += int64_t(gridDim.x) * kQGroups) {
        // four passes of loads in flight (eight measured 126.0 against 119.0 us for the
        // Q4_K 512 x 18944 x 3584 call with the pair-arithmetic codes; two 120.0 us)
        quantize_row<kQThreads, 4>(qf.x + m * K, qf.xq, m, K, L, ttc, wmax, tid, 1 + grp);
        asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kQThreads) : "memory");
      }
      // the scratch in the activation ring is overwritten by the producer's TMA next
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __threadfence();
      asm volatile("bar.sync %0, %1;" ::"n"(kBarEpi), "n"(32 * NEPI) : "memory");
      if (et == 0) grid_wait(qf.sync, gridDim.x, p.status);
      asm volatile("bar.sync %0, %1;" ::"n"(kBarAll), "n"(NT) : "memory");
    }
    const int e = warp - 4, q = warp & 3, hcol = e >> 2;  // rows 32q.., columns EC*hcol..
    const int rl = 32 * q + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(EC * hcol);
    // Scale reads are plain C++ shared loads (ordered after the group's mbarrier wait,
    // whose asm clobbers memory), so the compiler folds their constant offsets.
    const float *gsx0 = &sm.gsx[0][0][rl], *gd0 = &sm.gd[0][0][EC * hcol];
    // test hook: a wait that never completes, before the first accumulator use
    if (p.debug_expire) mbar_wait(sa(&sm.never), 0, p.status, 9, kTestWaitNs);
    for (int t = blockIdx.x, tl = 0; t < p.ntiles; t += gridDim.x, ++tl) {
    const int64_t m0 = int64_t(p.mt0 + t % p.ntm) * TM, n0 = int64_t(t / p.ntm) * TN;
    const int64_t m = m0 + rl;
    const bool mok = m < p.M;
    // accumulators as f32 pairs: one packed fma.rn.f32x2 per two columns
    float2 acc[EC / 2], y[EC / 2];
#pragma unroll
    for (int j = 0; j < EC / 2; ++j) acc[j] = y[j] = make_float2(0.f, 0.f);
    // Groups of 8 blocks (4 pairs; a Q4_K / Q6_K super-block), unrolled so that the
    // block's place in the group and every shared-memory offset are compile-time
    // constants.
    const uint32_t ub = (uint32_t)(tl * nuse) >> 1;  // accumulator uses per issuer before this tile
    for (int g = 0; g < ngroups; ++g) {
      const int G = tl * ngroups + g, slot = G & 1;
      if (!DOTS) mbar_wait(sa(&sm.gfull[slot]), (G >> 1) & 1, p.status, 6, kWaitNs);
      const float *gsx = gsx0 + slot * 8 * TM, *gd = gd0 + slot * 8 * TN;
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int pr = 4 * g + pp;
        if (PB && pr >= npairs) break;  // K % 256 == 0 for the K-quants
        // accumulator i and its phase; compile-time i for the K-quants (even nuse)
        const int U = tl * nuse + pr;
        const int i = PB ? U & 1 : pp & 1;
        const uint32_t par = PB ? (U >> 1) & 1 : (ub + (pp >> 1)) & 1;
        mbar_wait(sa(&sm.tfull[i]), par, p.status, 4, kWaitNs);
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int bi = 2 * pp + h, b = 8 * g + bi;
          if (PB && b >= nb) break;
          uint32_t r[EC];
          TC_LD32(trow + (uint32_t)(256 * i + 128 * h), r);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          if (h == 1 || (PB && b == nb - 1)) {  // accumulators in registers: free them
            tc_fence_before();
            mbar_arrive(sa(&sm.tempty[i]));
          }
          if constexpr (DOTS) {
            if (mok) {
#pragma unroll
              for (int j = 0; j < EC; ++j) {
                const int64_t n = n0 + EC * hcol + j;
                if (n < p.N) p.D[(m * p.N + n) * nb + b] = __float2int_rn(__uint_as_float(r[j]));
              }
            }
          } else {
            const float sxv = gsx[bi * TM];
            const float2 sx2 = make_float2(sxv, sxv);
            if constexpr (PB) {  // y += (s_m * d_n) * D per block
#pragma unroll
              for (int j4 = 0; j4 < EC / 4; ++j4) {
                const float4 c = *reinterpret_cast<const float4 *>(gd + bi * TN + 4 * j4);
                y[2 * j4] = __ffma2_rn(__fmul2_rn(sx2, make_float2(c.x, c.y)), pair(r, 4 * j4),
                                       y[2 * j4]);
                y[2 * j4 + 1] = __ffma2_rn(__fmul2_rn(sx2, make_float2(c.z, c.w)),
                                           pair(r, 4 * j4 + 2), y[2 * j4 + 1]);
              }
            } else {
              if (bi == 0) {  // first block of the super-block
#pragma unroll
                for (int j = 0; j < EC / 2; ++j) acc[j] = __fmul2_rn(sx2, pair(r, 2 * j));
              } else {
#pragma unroll
                for (int j = 0; j < EC / 2; ++j) acc[j] = __ffma2_rn(sx2, pair(r, 2 * j), acc[j]);
              }
              if (bi == 7) {  // end of the super-block: y += d * a
#pragma unroll
                for (int j4 = 0; j4 < EC / 4; ++j4) {
                  const float4 c = *reinterpret_cast<const float4 *>(gd + 7 * TN + 4 * j4);
                  y[2 * j4] = __ffma2_rn(make_float2(c.x, c.y), acc[2 * j4], y[2 * j4]);
                  y[2 * j4 + 1] = __ffma2_rn(make_float2(c.z, c.w), acc[2 * j4 + 1], y[2 * j4 + 1]);
                }
              }
            }
          }
        }
      }
      if (!DOTS) {
        mbar_arrive(sa(&sm.gempty[slot]));
      }
    }
    for (int j = 0; j < nmu; ++j) {  // y -= u_m * v_n * C_min, C_min summed over the min uses
      const int U = tl * nuse + npairs + j, i = U & 1;
      mbar_wait(sa(&sm.tfull[i]), (U >> 1) & 1, p.status, 7, kWaitNs);
      tc_fence_after();
      if (nms - j <= 0) {  // an empty use (one min-term stage): nothing to read
        mbar_arrive(sa(&sm.tempty[i]));
        continue;
      }
      uint32_t r[EC];
      TC_LD32(trow + (uint32_t)(256 * i), r);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      mbar_arrive(sa(&sm.tempty[i]));
      const float um = mok ? -p.urow[m] : 0.f;
      const float4 *v4 = reinterpret_cast<const float4 *>(p.vcol + n0 + EC * hcol);
      const float2 um2 = make_float2(um, um);
#pragma unroll
      for (int j4 = 0; j4 < EC / 4; ++j4) {
        const float4 v = __ldg(v4 + j4);
        y[2 * j4] = __ffma2_rn(__fmul2_rn(um2, make_float2(v.x, v.y)), pair(r, 4 * j4), y[2 * j4]);
        y[2 * j4 + 1] =
            __ffma2_rn(__fmul2_rn(um2, make_float2(v.z, v.w)), pair(r, 4 * j4 + 2), y[2 * j4 + 1]);
      }
    }
    if constexpr (!DOTS) {
      if (mok && p.swiglu) {
        // columns in units of 16: 8 gate columns, then the same 8 columns of the up
        // weight; the thread's 32 columns give 16 outputs silu(g) * u
        const int64_t nout = p.N >> 1, c0 = n0 + EC * hcol, left = p.N - c0;
        float h[EC / 2];
#pragma unroll
        for (int v = 0; v < 2; ++v)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int cg = 16 * v + j, cu = cg + 8;
            const float gv = (cg & 1) ? y[cg >> 1].y : y[cg >> 1].x;
            const float uv = (cu & 1) ? y[cu >> 1].y : y[cu >> 1].x;
            h[8 * v + j] = gv / (1.f + expf(-gv)) * uv;
          }
        float *dst = p.y + m * nout + (c0 >> 1);
#pragma unroll
        for (int v = 0; v < 2; ++v)
          if (left >= 16 * (v + 1))
#pragma unroll
            for (int j = 0; j < 8; j += 4)
              *reinterpret_cast<float4 *>(dst + 8 * v + j) =
                  make_float4(h[8 * v + j], h[8 * v + j + 1], h[8 * v + j + 2], h[8 * v + j + 3]);
      } else if (mok) {
        float *dst = p.y + m * p.N + n0 + EC * hcol;
        const int64_t left = p.N - (n0 + EC * hcol);
        if (left >= EC && (p.N & 3) == 0) {
#pragma unroll
          for (int j = 0; j < EC / 2; j += 2)
            *reinterpret_cast<float4 *>(dst + 2 * j) =
                make_float4(y[j].x, y[j].y, y[j + 1].x, y[j + 1].y);
        } else {
#pragma unroll
          for (int j = 0; j < EC; ++j)
            if (j < left) dst[j] = (j & 1) ? y[j >> 1].y : y[j >> 1].x;
        }
      }
    }
    }  // tiles
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
}

// ---- host side -------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

mq_status get_encode() {
  if (g_encode) return MQ_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e =
      cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return fail(MQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver (%s)",
                cudaGetErrorName(e));
  g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  return MQ_OK;
}

// f16 [rows][K] K-major with row stride ld elements (K when 0), box 64 x 128, 128-byte
// swizzle (rows beyond the tensor and columns beyond K read as 0).
mq_status encode_f16_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t K,
                         const char *what, int64_t ld = 0) {
  mq_status s = get_encode();
  if (s != MQ_OK) return s;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld ? ld : K) * 2};
  cuuint32_t box[2] = {PK, 128};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MQ_ERR_CUDA, "TMA descriptor for the %s operand (%lld x %lld f16 at %p) refused: %d",
                what, (long long)rows, (long long)K, ptr, (int)r);
  return MQ_OK;
}

// f32 [rows][cols] row-major (a transposed block-scale plane: row = block, column =
// matrix row), box 128 columns x 8 rows, no swizzle; rows past the plane read as 0.
mq_status encode_scale_map(CUtensorMap *map, const void *ptr, int64_t cols, int64_t rows,
                           const char *what) {
  mq_status s = get_encode();
  if (s != MQ_OK) return s;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {128, 8};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MQ_ERR_CUDA, "TMA descriptor for the %s plane (%lld x %lld f32 at %p) refused: %d",
                what, (long long)rows, (long long)cols, ptr, (int)r);
  return MQ_OK;
}

template <int TYPE, bool PW = false>
constexpr size_t smem_bytes() {
  return sizeof(TcSmem<TYPE, PW>) + 1024;
}

template <int TYPE, bool DOTS, bool QF = false, bool PW = false>
mq_status optin_t(const DeviceState *st, const char *name) {
  const size_t smem = smem_bytes<TYPE, PW>();
  if ((int)smem > st->smem_optin)
    return fail(MQ_ERR_LAUNCH, "%s needs %zu bytes of shared memory; the device allows %d", name,
                smem, st->smem_optin);
  cudaError_t e = cudaFuncSetAttribute(mmq_tc_kernel<TYPE, DOTS, QF, PW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "smem opt-in of %s (%zu bytes) refused: %s", name, smem,
                cudaGetErrorName(e));
  // the warpgroups' setmaxnreg split assumes this launch register count; with another one
  // the epilogue's increase could never be granted, so the kernel is refused instead
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, mmq_tc_kernel<TYPE, DOTS, QF, PW>);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "attributes of %s: %s", name, cudaGetErrorName(e));
  if (fa.numRegs != reg_launch<PW>())
    return fail(MQ_ERR_LAUNCH, "%s was compiled with %d registers per thread; its register "
                "split needs %d", name, fa.numRegs, reg_launch<PW>());
  return MQ_OK;
}

template <int TYPE, bool DOTS, bool PW = false>
mq_status launch_t(const mq_weight *W, const CUtensorMap &tA, const CUtensorMap &tAm,
                   const CUtensorMap &tSx, const TcArgs &a, const QfArgs &qf, cudaStream_t s,
                   int sms, const char *name) {
  // persistent: one CTA per SM (shared memory allows no more), tiles strided over them
  dim3 grid(test_fail_launch() ? 0u : (unsigned)(a.ntiles < sms ? a.ntiles : sms));
  const CUtensorMap &tW = *reinterpret_cast<const CUtensorMap *>(W->tmap_w);
  const CUtensorMap &tW2 = *reinterpret_cast<const CUtensorMap *>(
      TYPE == MQ_Q6_K ? W->tmap_w2 : W->tmap_w);
  const CUtensorMap &tBm = *reinterpret_cast<const CUtensorMap *>(
      TcSmem<TYPE>::MIN && !DOTS ? W->tmap_mb : W->tmap_w);
  const CUtensorMap &tD = *reinterpret_cast<const CUtensorMap *>(DOTS ? W->tmap_w : W->tmap_td);
  if (DOTS || qf.x == nullptr) {
    // programmatic stream serialisation: the CTAs' set-up (barriers, tensor memory) overlaps
    // the previous kernel's tail; the producer waits for that kernel before its first load
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(nthr<PW>(), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<TYPE, PW>();
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mmq_tc_kernel<TYPE, DOTS, false, PW>, tA, tW,
                                             tW2, tAm, tBm, tSx, tD, a, qf);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // the refused launch leaves no error behind for later calls
      return fail(MQ_ERR_LAUNCH, "launch of %s (grid %u) failed: %s", name, grid.x,
                  cudaGetErrorName(e));
    }
    return MQ_OK;
  }
  // fused quantisation: a cooperative launch, so that every CTA of the grid barrier is
  // resident (the runtime refuses the launch otherwise)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(nthr<PW>(), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<TYPE, PW>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, mmq_tc_kernel<TYPE, false, true, PW>, tA, tW, tW2, tAm, tBm, tSx, tD,
                         a, qf);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // the refused launch leaves no error behind for later calls
    return fail(MQ_ERR_LAUNCH, "cooperative launch of %s (grid %u) failed: %s", name, grid.x,
                cudaGetErrorName(e));
  }
  return MQ_OK;
}

}  // namespace

mq_status encode_weight_maps(mq_weight *w) {
  static_assert(sizeof(CUtensorMap) <= sizeof(w->tmap_w), "tensor map storage");
  // (a Q4_K weight registered with MQ_REG_MMQ_FROM_DECODE_PLANE has no f16 plane)
  mq_status s = w->mw ? encode_f16_map(reinterpret_cast<CUtensorMap *>(w->tmap_w), w->mw, w->N,
                                       w->K, "weight")
                      : MQ_OK;
  if (s != MQ_OK) return s;
  if (w->mw2)
    s = encode_f16_map(reinterpret_cast<CUtensorMap *>(w->tmap_w2), w->mw2, w->N, w->K,
                       "weight odd-part");
  if (s == MQ_OK && w->mb)
    s = encode_f16_map(reinterpret_cast<CUtensorMap *>(w->tmap_mb), w->mb, w->np,
                       3 * (w->K / 32), "weight min-term", min_ld(w->K / 32));
  if (s == MQ_OK)
    s = encode_scale_map(reinterpret_cast<CUtensorMap *>(w->tmap_td), w->td, w->np, w->K / 32,
                         "weight block scale");
  // a valid (unused) map in the weight slot of the kernels that take none
  if (s == MQ_OK && !w->mw) memcpy(w->tmap_w, w->tmap_td, sizeof(w->tmap_w));
  return s;
}

mq_status init_kernels(DeviceState *st) {
  mq_status s;
  if ((s = get_encode()) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q8_0, false>(st, "mmq_tc_kernel<Q8_0>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_K, false>(st, "mmq_tc_kernel<Q4_K>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q6_K, false>(st, "mmq_tc_kernel<Q6_K>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_1, false>(st, "mmq_tc_kernel<Q4_1>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q8_0, true>(st, "mmq_tc_kernel<Q8_0,dots>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_K, true>(st, "mmq_tc_kernel<Q4_K,dots>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q6_K, true>(st, "mmq_tc_kernel<Q6_K,dots>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q8_0, false, true>(st, "mmq_tc_kernel<Q8_0,fused>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_K, false, true>(st, "mmq_tc_kernel<Q4_K,fused>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q6_K, false, true>(st, "mmq_tc_kernel<Q6_K,fused>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_1, false, true>(st, "mmq_tc_kernel<Q4_1,fused>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_K, false, false, true>(st, "mmq_tc_kernel<Q4_K,plane>")) != MQ_OK)
    return s;
  if ((s = optin_t<MQ_Q4_K, true, false, true>(st, "mmq_tc_kernel<Q4_K,plane,dots>")) != MQ_OK)
    return s;
  if ((s = optin_t<MQ_Q4_K, false, true, true>(st, "mmq_tc_kernel<Q4_K,plane,fused>")) != MQ_OK)
    return s;
  return MQ_OK;
}

mq_status launch_mmq(const mq_weight *W, const void *xq, float *y, int32_t *D, int64_t M,
                     cudaStream_t s, const DeviceState *st, int debug_expire, const float *x,
                     unsigned *sync, int64_t mt_begin, int64_t mt_count) {
  const ActLayout L = act_layout(M, W->K);
  const uint8_t *base = reinterpret_cast<const uint8_t *>(xq);
  alignas(64) CUtensorMap tA, tAm;
  mq_status r = encode_f16_map(&tA, base + L.op, M, W->K, "activation");
  if (r != MQ_OK) return r;
  // Q5_K runs the Q4_K kernel (integer weight sc*q, same min term); Q4_0 and Q5_0 the
  // Q8_0 kernel (integer weight n - 8 / q - 16, one scale per 32-element block); Q5_1 the
  // Q4_1 kernel (one scale per block plus the min term of m)
  const bool mins = (W->type == MQ_Q4_K || W->type == MQ_Q5_K || W->type == MQ_Q4_1 ||
                     W->type == MQ_Q5_1) &&
                    D == nullptr;
  if (mins && (r = encode_f16_map(&tAm, base + L.amin, M, 3 * (W->K / 32), "activation min-term",
                                  min_ld(W->K / 32))) != MQ_OK)
    return r;
  if (!mins) tAm = tA;
  alignas(64) CUtensorMap tSx;
  if (D == nullptr) {
    if ((r = encode_scale_map(&tSx, base + L.st, L.mt, W->K / 32, "activation block scale")) !=
        MQ_OK)
      return r;
  } else {
    tSx = tA;  // unused by the block-dot kernels
  }
  TcArgs a;
  a.urow = reinterpret_cast<const float *>(base + L.urow);
  a.vcol = W->vcol;
  a.nms = mins ? (int)((3 * (W->K / 32) + PK - 1) / PK) : 0;
  a.y = y;
  a.D = D;
  a.M = M;
  a.N = W->N;
  a.mt = L.mt;
  a.np = W->np;
  a.nb = (int)(W->K / 32);
  const int64_t mt_all = (M + TM - 1) / TM, ntn = (W->N + TN - 1) / TN;
  const int64_t ntm = mt_count < 0 ? mt_all : mt_count;
  if (mt_begin < 0 || ntm < 1 || mt_begin + ntm > mt_all || (x != nullptr && ntm != mt_all))
    return fail(MQ_ERR_ARG, "mq_mmq: M-tiles %lld .. %lld outside the %lld of M=%lld",
                (long long)mt_begin, (long long)(mt_begin + ntm), (long long)mt_all,
                (long long)M);
  a.mt0 = (int)mt_begin;
  if (ntm * ntn > 0x7fffffff / 2)
    return fail(MQ_ERR_SHAPE, "mq_mmq: %lld x %lld output tiles are too many", (long long)ntm,
                (long long)ntn);
  a.ntm = (int)ntm;
  a.ntiles = (int)(ntm * ntn);
  a.status = st->status;
  a.debug_expire = debug_expire;
  a.swiglu = W->ffn_gu;
  a.wq = W->q;
  a.nchk = W->nchunk;
  QfArgs qf;
  qf.x = D == nullptr ? x : nullptr;  // the block-dot export is never fused
  qf.xq = const_cast<uint8_t *>(base);
  qf.sync = sync ? sync : reinterpret_cast<unsigned *>(const_cast<uint8_t *>(base) + L.sync);
  const bool dots = D != nullptr;
  switch (W->type) {
    case MQ_Q4_K:
      if (!W->mw)  // registered without the f16 plane: the weight tiles come from the decode plane
        return dots ? launch_t<MQ_Q4_K, true, true>(W, tA, tAm, tSx, a, qf, s, st->sms,
                                                    "mmq_tc_kernel<Q4_K,plane,dots>")
                    : launch_t<MQ_Q4_K, false, true>(W, tA, tAm, tSx, a, qf, s, st->sms,
                                                     "mmq_tc_kernel<Q4_K,plane>");
      [[fallthrough]];
    case MQ_Q5_K:
      return dots ? launch_t<MQ_Q4_K, true>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q4_K,dots>")
                  : launch_t<MQ_Q4_K, false>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q4_K>");
    case MQ_Q4_1:
    case MQ_Q5_1:  // block dots need no min term: the Q8_0 block-dot kernel
      return dots ? launch_t<MQ_Q8_0, true>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q8_0,dots>")
                  : launch_t<MQ_Q4_1, false>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q4_1>");
    case MQ_Q6_K:
      return dots ? launch_t<MQ_Q6_K, true>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q6_K,dots>")
                  : launch_t<MQ_Q6_K, false>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q6_K>");
    default:
      return dots ? launch_t<MQ_Q8_0, true>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q8_0,dots>")
                  : launch_t<MQ_Q8_0, false>(W, tA, tAm, tSx, a, qf, s, st->sms, "mmq_tc_kernel<Q8_0>");
  }
}

}  // namespace mq
