// mmq.cu -- prefill MMQ: y[m][n] = sum_b s[m][b] * (d[n][b] * D[m][n][b] -
// dmin_term[n][b] * S[m][b]) with D the exact integer dot of block b
// ("minfer CUDA Backend Design" §4.4: the int8 MMQ path for prefill; the
// per-block scale epilogue uses decoded f32 scale planes, §4.7 W_dsc).
//
// The contraction is exact: both operands are integers held in f16 (q in
// [-127, 127]; W_int = Q8_0 q, Q4_K sc_j*nib <= 945, Q6_K q-32 in [-32, 31]),
// every product is exact and every partial sum of one 32-element block stays
// below 2^24, so the f32 tensor-core accumulation of a block equals the
// integer dot.  (sm_103a has no integer tcgen05 kind and its legacy int8
// mma.sync runs at a quarter of the f16 rate, so f16 with integer values is the
// exact and fast encoding here.)
//
// This kernel: CTA tile 64 (m) x 128 (n), 8 warps of 32 x 32, one 32-K block
// per pipeline stage, a 4-stage cp.async ring, mma.sync m16n8k16 with
// ldmatrix fragments from an XOR-swizzled tile.  Per block and element the
// epilogue is
//   Q8_0: y += (s_m * d_n) * D
//   Q4_K: a += s_m * D,  y -= (s_m * S_m) * (dmin*m_j)_n,  per super-block y += d_n * a
//   Q6_K: D = sc_lo_n * D_lo + sc_hi_n * D_hi (exact), a += s_m * D, per super-block y += d_n * a
// In blockdots mode the per-block D is written out instead (test export).
// Grid: m-tiles fastest, so the CTAs in flight share each weight tile through L2
// and the weights stream from HBM about once.
#include "mq_common.cuh"

namespace mq {
namespace {

constexpr int BM = 64, BN = 128, BK = 32, STAGES = 4, THREADS = 256;

struct MmqArgs {
  const __half *A;       // activation operand f16 [M][K]
  const float *sx;       // [M][K/32]
  const int32_t *ssum;   // [M][K/32]
  const __half *W;       // weight operand f16 [N][K]
  const float *bd;       // [N][K/32]
  const float *bm;       // [N][K/32] (Q4_K)
  const float *bs;       // [N][K/16] (Q6_K)
  float *y;              // [M][N]
  int32_t *D;            // [M][N][K/32] (blockdots mode)
  int64_t M, N, K;
};

struct Stage {
  __half a[BM * BK];
  __half b[BN * BK];
  float sx[BM];
  int32_t ss[BM];
  float bd[BN];
  float bx[2 * BN];  // Q4_K: bm[n]; Q6_K: bs lo [n], bs hi [BN + n]
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp16(void *s, const void *g, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(s)), "l"(g),
               "r"(ok ? 16 : 0));
}
__device__ __forceinline__ void cp4(void *s, const void *g, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(s)), "l"(g),
               "r"(ok ? 4 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Row r of a 32-K tile is 64 bytes = 4 chunks of 16; chunk c lives at c ^ ((r>>1)&3).
__device__ __forceinline__ int swz(int r, int c) { return r * BK + 8 * (c ^ ((r >> 1) & 3)); }

template <int TYPE>
__device__ __forceinline__ void load_stage(const MmqArgs &p, Stage &st, int64_t m0, int64_t n0,
                                           int64_t kb) {
  const int tid = threadIdx.x;
  const int64_t nb = p.K / 32;
  {  // A: 64 rows x 4 chunks
    const int r = tid >> 2, c = tid & 3;
    const int64_t m = m0 + r;
    const bool ok = m < p.M;
    cp16(&st.a[swz(r, c)], p.A + (ok ? m : 0) * p.K + kb * BK + 8 * c, ok);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // B: 128 rows x 4 chunks
    const int idx = tid + i * THREADS, r = idx >> 2, c = idx & 3;
    const int64_t n = n0 + r;
    const bool ok = n < p.N;
    cp16(&st.b[swz(r, c)], p.W + (ok ? n : 0) * p.K + kb * BK + 8 * c, ok);
  }
  if (tid < BM) {
    const int64_t m = m0 + tid;
    const bool ok = m < p.M;
    cp4(&st.sx[tid], p.sx + (ok ? m : 0) * nb + kb, ok);
    cp4(&st.ss[tid], p.ssum + (ok ? m : 0) * nb + kb, ok);
  } else if (tid < BM + BN) {
    const int r = tid - BM;
    const int64_t n = n0 + r;
    const bool ok = n < p.N;
    cp4(&st.bd[r], p.bd + (ok ? n : 0) * nb + kb, ok);
    if constexpr (TYPE == MQ_Q4_K) cp4(&st.bx[r], p.bm + (ok ? n : 0) * nb + kb, ok);
    if constexpr (TYPE == MQ_Q6_K) {
      cp4(&st.bx[r], p.bs + (ok ? n : 0) * (2 * nb) + 2 * kb, ok);
      cp4(&st.bx[BN + r], p.bs + (ok ? n : 0) * (2 * nb) + 2 * kb + 1, ok);
    }
  }
}

template <int TYPE, bool DOTS>
__global__ void __launch_bounds__(THREADS, 1) mmq_kernel(const MmqArgs p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Stage *stages = reinterpret_cast<Stage *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile (32 m) x (32 n)
  const int g = lane >> 2, t = lane & 3;
  const int64_t m0 = int64_t(blockIdx.x) * BM, n0 = int64_t(blockIdx.y) * BN;
  const int64_t nb = p.K / 32;

  // fragment-owned rows/cols: rows wm*32 + mi*16 + g (+8), cols wn*32 + ni*8 + 2t (+1)
  float y[2][4][4], a[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int v = 0; v < 4; ++v) y[mi][ni][v] = a[mi][ni][v] = 0.f;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nb) load_stage<TYPE>(p, stages[s], m0, n0, s);
    cp_commit();
  }

  for (int64_t kb = 0; kb < nb; ++kb) {
    cp_wait<STAGES - 2>();
    __syncthreads();
    {
      const int64_t nk = kb + STAGES - 1;
      if (nk < nb) load_stage<TYPE>(p, stages[nk % STAGES], m0, n0, nk);
      cp_commit();
    }
    const Stage &st = stages[kb % STAGES];
    float c0[2][4][4], c1[2][4][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int v = 0; v < 4; ++v) c0[mi][ni][v] = c1[mi][ni][v] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {  // two k16 halves of the block
      uint32_t af[2][4], bf[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int r = wm * 32 + mi * 16 + (lane & 15);
        ldsm_x4(af[mi], &st.a[swz(r, 2 * ks + (lane >> 4))]);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int r = wn * 32 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(bf[np], &st.b[swz(r, 2 * ks + ((lane >> 3) & 1))]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const uint32_t b0 = bf[ni >> 1][2 * (ni & 1)], b1 = bf[ni >> 1][2 * (ni & 1) + 1];
          if (TYPE == MQ_Q6_K && ks == 1)
            mma16816(c1[mi][ni], af[mi], b0, b1);
          else
            mma16816(c0[mi][ni], af[mi], b0, b1);
        }
    }
    // epilogue of block kb
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // rows g, g+8
        const int rl = wm * 32 + mi * 16 + g + 8 * h;
        const float sxm = st.sx[rl];
        const float tm = sxm * (float)st.ss[rl];
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cl = wn * 32 + ni * 8 + 2 * t + e;
            const int v = 2 * h + e;
            float dv = c0[mi][ni][v];
            if constexpr (TYPE == MQ_Q6_K) dv = fmaf(st.bx[BN + cl], c1[mi][ni][v], st.bx[cl] * dv);
            if constexpr (DOTS) {
              const int64_t m = m0 + rl, n = n0 + cl;
              if (m < p.M && n < p.N) p.D[(m * p.N + n) * nb + kb] = __float2int_rn(dv);
            } else if constexpr (TYPE == MQ_Q8_0) {
              y[mi][ni][v] = fmaf(sxm * st.bd[cl], dv, y[mi][ni][v]);
            } else {
              a[mi][ni][v] = fmaf(sxm, dv, a[mi][ni][v]);
              if constexpr (TYPE == MQ_Q4_K) y[mi][ni][v] = fmaf(-tm, st.bx[cl], y[mi][ni][v]);
              if ((kb & 7) == 7) {
                y[mi][ni][v] = fmaf(st.bd[cl], a[mi][ni][v], y[mi][ni][v]);
                a[mi][ni][v] = 0.f;
              }
            }
          }
        }
      }
    }
  }
  cp_wait<0>();
  if constexpr (!DOTS) {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t m = m0 + wm * 32 + mi * 16 + g + 8 * h;
        if (m >= p.M) continue;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const int64_t n = n0 + wn * 32 + ni * 8 + 2 * t;
          float *dst = p.y + m * p.N + n;
          const float v0 = y[mi][ni][2 * h], v1 = y[mi][ni][2 * h + 1];
          if (n + 1 < p.N && ((p.N & 1) == 0)) {
            *reinterpret_cast<float2 *>(dst) = make_float2(v0, v1);
          } else {
            if (n < p.N) dst[0] = v0;
            if (n + 1 < p.N) dst[1] = v1;
          }
        }
      }
  }
}

template <int TYPE, bool DOTS>
mq_status launch_t(const MmqArgs &a, cudaStream_t s, const char *name) {
  const size_t smem = sizeof(Stage) * STAGES;
  dim3 grid((unsigned)((a.M + BM - 1) / BM), (unsigned)((a.N + BN - 1) / BN));
  if (grid.y > 65535)
    return fail(MQ_ERR_SHAPE, "%s: N=%lld needs more than 65535 column tiles", name,
                (long long)a.N);
  mmq_kernel<TYPE, DOTS><<<grid, THREADS, smem, s>>>(a);
  MQ_LAUNCH_CHECK(name);
  return MQ_OK;
}

template <int TYPE, bool DOTS>
mq_status optin_t(const DeviceState *st, const char *name) {
  const size_t smem = sizeof(Stage) * STAGES;
  if ((int)smem > st->smem_optin)
    return fail(MQ_ERR_LAUNCH, "%s needs %zu bytes of shared memory; the device allows %d", name,
                smem, st->smem_optin);
  cudaError_t e = cudaFuncSetAttribute(mmq_kernel<TYPE, DOTS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess)
    return fail(MQ_ERR_LAUNCH, "smem opt-in of %s (%zu bytes) refused: %s", name, smem,
                cudaGetErrorName(e));
  return MQ_OK;
}

}  // namespace

mq_status init_kernels(DeviceState *st) {
  mq_status s;
  if ((s = optin_t<MQ_Q8_0, false>(st, "mmq_kernel<Q8_0>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_K, false>(st, "mmq_kernel<Q4_K>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q6_K, false>(st, "mmq_kernel<Q6_K>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q8_0, true>(st, "mmq_kernel<Q8_0,dots>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q4_K, true>(st, "mmq_kernel<Q4_K,dots>")) != MQ_OK) return s;
  if ((s = optin_t<MQ_Q6_K, true>(st, "mmq_kernel<Q6_K,dots>")) != MQ_OK) return s;
  return MQ_OK;
}

mq_status launch_mmq(const mq_weight *W, const void *xq, float *y, int32_t *D, int64_t M,
                     cudaStream_t s, const DeviceState *) {
  const ActLayout L = act_layout(M, W->K);
  const uint8_t *base = reinterpret_cast<const uint8_t *>(xq);
  MmqArgs a;
  a.A = reinterpret_cast<const __half *>(base + L.op);
  a.sx = reinterpret_cast<const float *>(base + L.scale);
  a.ssum = reinterpret_cast<const int32_t *>(base + L.bsum);
  a.W = W->mw;
  a.bd = W->mbd;
  a.bm = W->mbm;
  a.bs = W->mbs;
  a.y = y;
  a.D = D;
  a.M = M;
  a.N = W->N;
  a.K = W->K;
  const bool dots = D != nullptr;
  switch (W->type) {
    case MQ_Q4_K:
      return dots ? launch_t<MQ_Q4_K, true>(a, s, "mmq_kernel<Q4_K,dots>")
                  : launch_t<MQ_Q4_K, false>(a, s, "mmq_kernel<Q4_K>");
    case MQ_Q6_K:
      return dots ? launch_t<MQ_Q6_K, true>(a, s, "mmq_kernel<Q6_K,dots>")
                  : launch_t<MQ_Q6_K, false>(a, s, "mmq_kernel<Q6_K>");
    default:
      return dots ? launch_t<MQ_Q8_0, true>(a, s, "mmq_kernel<Q8_0,dots>")
                  : launch_t<MQ_Q8_0, false>(a, s, "mmq_kernel<Q8_0>");
  }
}

}  // namespace mq
