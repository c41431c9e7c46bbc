/*
 * mq.h -- C ABI of libmq: GGUF block-quantised weight x f32 activation matmul
 * on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the quantised MatMul of the minfer engine ("minfer CUDA
 * Backend Design", §4.4 Execution dispatch): weights stay in their GGUF block
 * encoding (Q8_0 / Q4_K / Q6_K, and Q4_0, Q4_1, Q5_0, Q5_1, Q5_K; unquantised F16 and
 * BF16 for the matvec), activations and outputs are f32 ("CUDA Backend Design" §1.3:
 * activations stay f32).  Two forms:
 *
 *   decode matvec   y[b][n] = sum_k w[n][k] * x[b][k],  b < B <= 8
 *                   ("CUDA Backend Design" §4.4: nt == 1 and the _multi
 *                   variants for nt 2..8), weights dequantised in registers.
 *   prefill MMQ     activations quantised per 32-element block to int8 with an
 *                   f32 scale (mq_quantize_act), then an exact integer
 *                   contraction per block and a per-block scale epilogue
 *                   (mq_mmq) ("CUDA Backend Design" §4.4: the int8 MMQ path);
 *                   mq_mmq_fused does both in one kernel.
 *
 * Conventions ("CUDA Backend Design" §4.9 GPU safety; "GPU Safety" CUDA
 * rules): every invariant violation returns an error status and never falls
 * back to another kernel or to the CPU; every launch is checked at its site;
 * device limits are queried at run time; waits inside kernels are bounded.
 *
 * Threading: calls may come from several host threads.  mq_last_error() is
 * per thread.  A weight handle may be used concurrently from several streams
 * (kernels only read it).  mq_weight_free must not race with calls using the
 * handle.
 *
 * Pointers: "device pointer" means memory the current CUDA device can access
 * as global memory (cudaMalloc, torch CUDA tensors, managed memory).  Host
 * pointers passed where a device pointer is required are rejected with
 * MQ_ERR_ARG (checked with cudaPointerGetAttributes).  All hot-path calls are
 * asynchronous on the given stream.  They allocate nothing, with one exception:
 * mq_matvec with B = 5..8 on a Q4_K / Q5_K weight of at least SMs / 2 row
 * groups of 128 takes a per-call buffer of 36 bytes per element of K
 * (the activation fragment plane) from a stream-ordered pool that mq_init
 * creates for the device, and frees it in stream order after its kernels (in
 * a captured graph: an allocation node and a free node).  If the pool cannot
 * give it, the call computes the same result without it.
 */
#ifndef MQ_H
#define MQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GGUF tensor type ids of the supported block formats.
 *   MQ_Q4_0: 32-element blocks of 18 bytes: f16 d, 16 bytes of 4-bit quants
 *            (element j < 16 the low nibble of byte j, element 16 + j its high
 *            nibble);  w = d*(q - 8).
 *   MQ_Q4_1: 32-element blocks of 20 bytes: f16 d, f16 m, 16 quant bytes (nibbles as
 *            MQ_Q4_0);  w = d*q + m.
 *   MQ_Q5_0: 32-element blocks of 22 bytes: f16 d, a 32-bit little-endian word whose
 *            bit e is the fifth bit of element e, 16 quant bytes (low four bits as
 *            MQ_Q4_0);  w = d*(q - 16), q in [0, 31].
 *   MQ_Q5_1: 32-element blocks of 24 bytes: f16 d, f16 m, the fifth-bit word, 16 quant
 *            bytes;  w = d*q + m.
 *   MQ_Q8_0: 32-element blocks of 34 bytes: f16 d, 32 x int8 q;  w = d*q.
 *   MQ_Q4_K: 256-element super-blocks of 144 bytes: f16 d, f16 dmin, 12 bytes
 *            of packed 6-bit sub-block scales/mins, 128 bytes of 4-bit quants;
 *            w = d*sc_j*q - dmin*m_j.
 *   MQ_Q5_K: 256-element super-blocks of 176 bytes: as MQ_Q4_K (f16 d, f16 dmin,
 *            12 bytes of scales/mins) then 32 bytes of fifth bits (bit 2c + h of
 *            byte l for element 64c + 32h + l) and 128 bytes of low 4 bits;
 *            w = d*sc_j*q - dmin*m_j with q in [0, 31].
 *   MQ_Q6_K: 256-element super-blocks of 210 bytes: 128 bytes low 4 bits,
 *            64 bytes high 2 bits, 16 int8 sub-scales, f16 d;
 *            w = d*sc*(q - 32).
 *   MQ_F16, MQ_BF16: unquantised weights, one little-endian IEEE binary16 (or bfloat16,
 *            the upper half of a binary32) per element, rows of K elements; K must be a
 *            multiple of 32.  Decode matvec only ("CUDA Backend Design" §4.4: the f16 and
 *            bf16 kernels); they have no integer form, so mq_mmq, mq_mmq_blockdots and
 *            mq_ffn_gu_mmq return MQ_ERR_TYPE, and registration builds no prefill planes.
 * Byte ratios as in "CUDA Backend Design" §2.3 (34/32, 144/256, 210/256); Q4_0, Q4_1,
 * Q5_0, Q5_1 and Q5_K are among the types its matmul whitelist and weight gate admit
 * (§4.3, §4.6). */
typedef enum {
    MQ_F16 = 1, MQ_Q4_0 = 2, MQ_Q4_1 = 3, MQ_Q5_0 = 6, MQ_Q5_1 = 7, MQ_Q8_0 = 8,
    MQ_Q4_K = 12, MQ_Q5_K = 13, MQ_Q6_K = 14, MQ_BF16 = 30
} mq_type;

typedef enum {
    MQ_OK = 0,
    MQ_ERR_ARG = 1,      /* null / host / misaligned pointer, bad flag, B or M out of range */
    MQ_ERR_TYPE = 2,     /* unsupported type, or type differs from the weight's */
    MQ_ERR_SHAPE = 3,    /* N, K invalid, K not a multiple of the block, or N/K differ from W */
    MQ_ERR_PAYLOAD = 4,  /* nbytes != N*(K/blk)*blkbytes (equality, "CUDA Backend Design" §2.3) */
    MQ_ERR_ALIGN = 5,    /* a buffer is not 16-byte aligned */
    MQ_ERR_CUDA = 6,     /* a CUDA runtime call failed (message names it) */
    MQ_ERR_OOM = 7,      /* device allocation failed at registration */
    MQ_ERR_LAUNCH = 8,   /* a kernel launch or smem opt-in was refused (message names the kernel) */
    MQ_ERR_TIMEOUT = 9,  /* a bounded device-side wait expired (reported by mq_stream_status) */
    MQ_ERR_STATE = 10    /* mq_init was not called for the current device */
} mq_status;

/* Opaque weight handle: library-owned device planes built at registration. */
typedef struct mq_weight mq_weight;

/* Stream handle: a cudaStream_t (NULL = the legacy default stream). */
typedef void *mq_stream;

/* Registration flags. */
#define MQ_REG_DEFAULT 0u
/* Skip the prefill operand planes; mq_mmq then returns MQ_ERR_ARG for this weight. */
#define MQ_REG_NO_MMQ_PLANE 1u
/* Q4_K only (MQ_ERR_ARG for other types): build no f16 integer weight plane (2 bytes per
 * element, 3.56x the GGUF payload); the MMQ calls copy the decode plane's 144-byte-per-row
 * tiles and expand them to the same f16 integers sc_j * nib in shared memory.  Results are
 * bit-identical to the default; the prefill MMQ takes longer (measured on 512 x 18944 x 3584:
 * 151 against 110 us).  Device bytes fall from 5.3x to 1.8x the payload. */
#define MQ_REG_MMQ_FROM_DECODE_PLANE 2u

/* mq_init -- prepare the library for CUDA device `device` (makes it current on
 * the calling thread).  Queries the SM count and the shared-memory opt-in
 * limit, opts every kernel that needs more than 48 KiB of dynamic shared
 * memory in (once per device, outside any stream capture: "CUDA Backend
 * Design" §2.4, the eager pre-warm), allocates the per-device status word
 * used by bounded waits and looks up the address of mq_mmq_fused_static's
 * scratch.  Idempotent.  Must precede every other call for that device.  Each
 * call also reads the tests' switches MQ_TEST_FAIL_LAUNCH, MQ_TEST_EXPIRE_WAIT and
 * MQ_TEST_NO_XPLANE from the environment (no hot-path call reads it).
 * Errors: MQ_ERR_CUDA, MQ_ERR_LAUNCH (an opt-in refused). */
mq_status mq_init(int device);

/* mq_register_weight -- copy an N x K GGUF tensor (rows contiguous, blocks
 * along K, exactly as stored in a GGUF file) to the current device and build
 * the device planes ("CUDA Backend Design" §2.3 weight residency and
 * registry: uploaded once at load, quant-specific repacks):
 *   - the decode plane: the same bytes, regrouped so that each thread of a
 *     tensor-core fragment reads 16-byte words (lossless: mq_weight_unpack
 *     restores the original bytes);
 *   - unless MQ_REG_NO_MMQ_PLANE: the prefill operand planes (integer-valued
 *     f16 weights [N][K], none with MQ_REG_MMQ_FROM_DECODE_PLANE, plus f32
 *     block-scale planes).
 * host_bytes: host pointer to nbytes bytes (read only during the call).
 * Validation before any device work: type supported (MQ_ERR_TYPE); N >= 1,
 * K >= 1, K a multiple of the block size (MQ_ERR_SHAPE); nbytes ==
 * N*(K/blk)*blkbytes (MQ_ERR_PAYLOAD).  Synchronous: uses the library's own
 * stream and synchronises it before returning, so it never enters a caller's
 * stream-capture window ("CUDA Backend Design" §2.4).  *out receives the
 * handle (owned by the caller, released with mq_weight_free).
 * Errors also: MQ_ERR_OOM, MQ_ERR_CUDA, MQ_ERR_STATE. */
mq_status mq_register_weight(mq_type type, const void *host_bytes, size_t nbytes, int64_t N,
                             int64_t K, uint32_t flags, mq_weight **out);

/* mq_weight_free -- release the weight's device planes (synchronises the
 * device first so no queued kernel still reads them).  NULL is a no-op. */
mq_status mq_weight_free(mq_weight *w);

/* mq_weight_info -- type, N, K and total device bytes of a weight. */
mq_status mq_weight_info(const mq_weight *w, int *type, int64_t *N, int64_t *K,
                         size_t *device_bytes);

/* mq_weight_unpack -- write the original GGUF bytes of W back to host memory
 * (nbytes must equal the registered payload size).  Test/diagnostic call:
 * rebuilds the bytes from the decode plane on the device.  Synchronous. */
mq_status mq_weight_unpack(const mq_weight *w, void *host_bytes, size_t nbytes);

/* mq_matvec -- decode matvec.  x: device f32 [B][K] row-major; y: device f32
 * [B][N] row-major (written, never read); 1 <= B <= 8.  type, N, K must match
 * W.  x and y 16-byte aligned.  Every column b of a batched call is computed
 * exactly as the B = 1 call on x[b] (bitwise; "Architecture Execution Plan"
 * ADR-0010, the bitwise-by-default identity rule).  Float result within
 * 1e-4 * sum_k |w[n][k]| |x[b][k]| of the exact product.  The calls with
 * B = 5..8 on wide Q4_K / Q5_K weights use a per-call buffer from the
 * library's stream-ordered pool (see Pointers above). */
mq_status mq_matvec(mq_type type, const mq_weight *W, const float *x, float *y, int64_t N,
                    int64_t K, int B, mq_stream stream);

/* mq_act_bytes -- size of the quantised-activation buffer xq for M x K.
 * Layout (each section starts on a 256-byte boundary, in this order;
 * Mt = M rounded up to a multiple of 128):
 *   qs      int8  [M][K]       the quantised values q
 *   scale   f32   [M][K/32]    the block scales s = max|x| / 127
 *   bsum    int32 [M][K/32]    the block sums S = sum q
 *   operand f16   [M][K]       q as f16 (exact), the tensor-core operand
 *   scaleT  f32   [K/32][Mt]   s transposed (rows >= M unspecified)
 *   minT    f32   [K/32][Mt]   s * S transposed, the min-term factor (rows >= M unspecified)
 *   amin    f16   [M][L]       min-term operand, L = 3*K/32 rounded up to a multiple of 8:
 *                              row m holds hi | hi | lo over the blocks b of t = s*S / u_m,
 *                              hi = f16(t), lo = f16(t - hi) (columns 3*K/32..L-1 unspecified)
 *   urow    f32   [Mt]         u_m = 2^k, k = E - 140 clamped to [-100, 100], E the biased
 *                              binary32 exponent of max_b |s*S| (so max_b |s*S| / u_m is in
 *                              [2^13, 2^14) for a normal maximum); k = 0 when the row's s*S
 *                              are all 0 (rows >= M unspecified)
 *   sync    u32   [2]          the grid barrier of mq_mmq_fused: an arrival count, which
 *                              must be zero before the buffer's first mq_mmq_fused call
 *                              and which every call leaves zero, and a generation word
 *                              (any value; each call advances it).  mq_quantize_act and
 *                              mq_mmq neither read nor write them.
 * Returns 0 if K is not a positive multiple of 32 or M < 1. */
size_t mq_act_bytes(int64_t M, int64_t K);

/* mq_quantize_act -- quantise f32 activations per 32-element block ("CUDA
 * Backend Design" §4.4: prefill quantises A into per-32 int8 blocks;
 * "Architecture Execution Plan" C4 S2b design decision 4: amax/127,
 * round half to even).  In IEEE binary32: amax = max|x|, s = amax/127
 * (correctly rounded), q = round_half_even(x/s) clamped to [-127, 127],
 * S = sum q; a block whose s is 0 gets q = 0.  x: device f32 [M][K];
 * xq: device buffer of mq_act_bytes(M, K) bytes (256-byte aligned).
 * K % 32 == 0, M >= 1. */
mq_status mq_quantize_act(const float *x, void *xq, int64_t M, int64_t K, mq_stream stream);

/* mq_mmq -- prefill matmul y[m][n] = sum_b s[m][b] * (d[n][b]*D[m][n][b] -
 * dmin_term[n][b]*S[m][b]) where D is the exact integer block dot of the
 * weight's integer values with q (see mq_mmq_blockdots).  xq from
 * mq_quantize_act(M, K); y: device f32 [M][N] row-major.  W must have its
 * MMQ planes.  Float result within 1e-4 * sum_k |w| |s*q| of the exact
 * product of W with the dequantised activations. */
mq_status mq_mmq(mq_type type, const mq_weight *W, const void *xq, float *y, int64_t M,
                 int64_t N, int64_t K, mq_stream stream);

/* mq_matvec_host, mq_mmq_host -- the decode matvec and the prefill (mq_quantize_act +
 * mq_mmq) from host buffers x_host (f32 [B][K] / [M][K]) and y_host (f32 [B][N] / [M][N]);
 * x_dev, y_dev are the caller's device buffers of the same shapes and xq_dev its
 * quantised-activation buffer (mq_act_bytes(M, K)).  Nothing is allocated.  Like every call
 * here they return once the work is enqueued on `stream`: y_host is complete when `stream`
 * is.  Transfers:
 *   - a host buffer that is page-locked (cudaHostAlloc, cudaHostRegister, a pinned tensor)
 *     and 16-byte aligned is accessed by the kernels through its device view, over the
 *     host link: the matvec's x is pulled into x_dev by a small copy kernel that the
 *     matvec overlaps (its weight stream starts at once; x is read after the grid
 *     dependency wait), the matvec stores y into y_host (y_dev is not written), and the
 *     prefill's quantiser reads x_host itself (x_dev is not written);
 *   - any other host buffer, and the prefill's y always, goes through x_dev / y_dev with
 *     cudaMemcpyAsync copies (synchronous with the host for pageable memory, as CUDA
 *     defines them).  The prefill's MMQ runs in up to four chunks of 128-row tiles, and
 *     each chunk's rows of y are copied back on a stream the library owns (created by
 *     mq_init) while the next chunk runs; that stream waits on events recorded on `stream`
 *     and `stream` waits on it before the call returns, so the work stays ordered on
 *     `stream` (also when `stream` is being captured into a CUDA graph).
 * The results are identical on both routes.  Host pointers that CUDA reports as device
 * memory are refused (MQ_ERR_ARG); the rest is validated as mq_matvec / mq_mmq, all before
 * anything is enqueued.  The device reads the activations as f32, as in the decisions
 * listed on "CUDA Backend Design" (ADR-0013). */
mq_status mq_matvec_host(mq_type type, const mq_weight *W, const float *x_host, float *y_host,
                         float *x_dev, float *y_dev, int64_t N, int64_t K, int B,
                         mq_stream stream);
mq_status mq_mmq_host(mq_type type, const mq_weight *W, const float *x_host, float *y_host,
                      float *x_dev, void *xq_dev, float *y_dev, int64_t M, int64_t N, int64_t K,
                      mq_stream stream);

/* mq_mmq_fused -- mq_quantize_act followed by mq_mmq in one kernel: every CTA of the
 * persistent MMQ first quantises a slice of the rows of x into xq, a grid-wide barrier
 * follows, then the contraction runs as in mq_mmq ("CUDA Backend Design" §3 and §8: the
 * quantisation fused into the GEMM's prologue, named there as the open step change; §4:
 * the quantised activations stay valid for the next matmul on the same rows).
 * x: device f32 [M][K]; xq: device buffer of mq_act_bytes(M, K) bytes (256-byte aligned)
 * whose sync count is zero before its first fused call (each call leaves it zero; one
 * call in flight per buffer); on return xq holds exactly what mq_quantize_act writes and y
 * equals the result of mq_quantize_act + mq_mmq bit for bit.  The launch is cooperative
 * (all CTAs co-resident, or MQ_ERR_LAUNCH); the barrier wait is bounded (an expiry is
 * reported by mq_stream_status).  Quantised weights with MMQ planes only (MQ_ERR_TYPE for
 * F16 / BF16, MQ_ERR_ARG for a fused gate/up weight or one registered without planes). */
mq_status mq_mmq_fused(mq_type type, const mq_weight *W, const float *x, void *xq, float *y,
                       int64_t M, int64_t N, int64_t K, mq_stream stream);

/* mq_mmq_fused_static -- mq_mmq_fused with its scratch in the library instead of a caller
 * buffer, so that the call allocates nothing (no counterpart in the pages, which always
 * hand the quantised activations over in a buffer).  The scratch is one file-scope static
 * device array of MQ_STATIC_XQ_BYTES per device, created by the driver with the library's
 * device code; mq_init looks its address up (cudaGetSymbolAddress, checked), which loads
 * that code, so the array exists once mq_init has returned and a call allocates nothing.  Its first 256 bytes hold the
 * grid barrier's words, the rest an xq buffer: mq_act_bytes(M, K) must not exceed
 * MQ_STATIC_XQ_BYTES - 256 (else MQ_ERR_SHAPE, before any device work).  After a call the
 * scratch holds that call's quantised activations in the mq_act_bytes layout (there is no
 * accessor; the next call overwrites them).  Calls that overlap in time (on different
 * streams, or from different host threads) share the scratch and race: their results, and
 * the barrier, are then undefined (an expired barrier wait is reported by
 * mq_stream_status).  y and x as for mq_mmq_fused; y equals mq_mmq_fused's bit for bit. */
#define MQ_STATIC_XQ_BYTES (16u << 20)
mq_status mq_mmq_fused_static(mq_type type, const mq_weight *W, const float *x, float *y,
                              int64_t M, int64_t N, int64_t K, mq_stream stream);

/* mq_mmq_blockdots -- test export of the contraction's integer part:
 * D[(m*N + n)*(K/32) + b] = sum_{k in block b} W_int[n][k] * q[m][k], int32,
 * where W_int is the weight's integer value: Q8_0 the int8 quant; Q4_K the
 * 6-bit sub-block scale times the 4-bit quant; Q6_K the int8 16-element
 * sub-scale times (6-bit quant - 32).  Same tensor-core code path as mq_mmq.
 * D: device int32 buffer of M*N*(K/32) elements. */
mq_status mq_mmq_blockdots(mq_type type, const mq_weight *W, const void *xq, int32_t *D,
                           int64_t M, int64_t N, int64_t K, mq_stream stream);

/* ---- fused FFN gate/up with SwiGLU ("minfer CUDA Backend Design" §4.3: the FusedFFN
 * and SwiGLU ops; §4.6: the loader's ffn_gu concat of the gate and up weights).  The
 * pages name the operation without writing it out; it is read as the usual
 * h = silu(W_gate x) * (W_up x), silu(v) = v / (1 + e^-v), elementwise. */

/* mq_register_ffn_gu -- register the gate and up weights of one FFN as a single fused
 * weight of 2N rows.  gate_bytes, up_bytes: raw GGUF bytes of an N x K tensor each
 * (host memory, read only during the call), nbytes_each = the exact size of one of
 * them; N % 8 == 0.  The rows are stored in units of 16 (8 gate rows, then the same 8
 * rows of the up weight), so one kernel thread holds a gate result and its up result.
 * flags as for mq_register_weight.  mq_weight_unpack returns the gate bytes followed by
 * the up bytes.  A fused weight is used only through mq_ffn_gu_matvec / mq_ffn_gu_mmq
 * (the plain calls return MQ_ERR_ARG, and vice versa).  mq_weight_info reports 2N rows.
 * Errors as for mq_register_weight; MQ_ERR_SHAPE if N % 8 != 0. */
mq_status mq_register_ffn_gu(mq_type type, const void *gate_bytes, const void *up_bytes,
                             size_t nbytes_each, int64_t N, int64_t K, uint32_t flags,
                             mq_weight **out);

/* mq_ffn_gu_matvec -- decode form: h[b][n] = silu(g[b][n]) * u[b][n] with
 * g = W_gate x, u = W_up x computed as by mq_matvec (same kernels, one launch).
 * x: device f32 [B][K]; h: device f32 [B][N] (N = gate rows); 1 <= B <= 8.
 * Within silu's slope (<= 1.1) times the matvec bound of g, times |u|, plus
 * |silu(g)| times the bound of u. */
mq_status mq_ffn_gu_matvec(mq_type type, const mq_weight *W, const float *x, float *h,
                           int64_t N, int64_t K, int B, mq_stream stream);

/* mq_ffn_gu_mmq -- prefill form: h[m][n] = silu(g[m][n]) * u[m][n] with g, u computed
 * as by mq_mmq from xq (mq_quantize_act(M, K)).  h: device f32 [M][N]; the weight must
 * have its MMQ planes.  Bound as for mq_ffn_gu_matvec with the MMQ bounds of g and u. */
mq_status mq_ffn_gu_mmq(mq_type type, const mq_weight *W, const void *xq, float *h, int64_t M,
                        int64_t N, int64_t K, mq_stream stream);

/* mq_stream_status -- synchronise `stream`, then read and clear the current
 * device's status word written by bounded device-side waits.  Returns MQ_OK,
 * or MQ_ERR_TIMEOUT if a wait expired since the last call (the message names
 * the kernel), or MQ_ERR_CUDA if the synchronisation failed. */
mq_status mq_stream_status(mq_stream stream);

/* mq_last_error -- message of the last failing call on this thread: the call,
 * the violated invariant and the values involved.  Never NULL. */
const char *mq_last_error(void);

/* mq_status_name -- "MQ_OK", "MQ_ERR_ARG", ... */
const char *mq_status_name(mq_status s);

#ifdef __cplusplus
}
#endif

#endif /* MQ_H */
