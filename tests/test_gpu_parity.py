"""GPU parity of libmq's CUDA path against the CPU oracle, through the C ABI.

Integer work (decode-plane round trip, quantised activations, per-block integer
dots) must match bit for bit; float outputs must satisfy
|y - y_ref| <= 1e-4 * sum_k |w||x| per element (the decode matvec and the MMQ,
the latter against the dequantised activations s*q).  Sizes: small shapes that
span several tiles with ragged tails, and the five hot-path workloads at full
size in the launch configuration the bench uses (outputs compared in full where
the oracle is fast enough, else on sampled rows)."""
import functools

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quantized_q4_gb300 as mq  # noqa: E402
from gguf_block_quantized_q4_gb300 import build as mqbuild  # noqa: E402

REL = 1e-4  # the per-element bound: |y - y_ref| <= REL * sum |w||x|


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mqbuild.build()
    mq.init(0)
    yield


@functools.lru_cache(maxsize=None)
def weights(qtype, N, K, seed):
    return synth.weights(qtype, N, K, seed)


@functools.lru_cache(maxsize=8)
def registered(qtype, N, K, seed, flags=0):
    return mq.register_weight(qtype, weights(qtype, N, K, seed), N, K, flags)


def assert_bound(y, yref, bnd, what):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - yref)
    lim = REL * bnd
    bad = err > lim + 1e-37
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside the bound; worst "
                           f"err/bound {np.max(err / np.maximum(bnd, 1e-300)):.3e}")


def gpu_matvec(W, x):
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    y = mq.matvec(W, xt)
    torch.cuda.synchronize()
    return y.cpu().numpy()


# ---- decode planes -----------------------------------------------------------

@pytest.mark.parametrize("qtype,N,K", [(8, 37, 96), (8, 896, 896), (12, 19, 512),
                                       (12, 18944, 3584), (14, 21, 768), (14, 3584, 18944),
                                       (2, 37, 96), (2, 4864, 896), (13, 19, 512),
                                       (13, 18944, 3584), (3, 37, 96), (3, 4864, 896),
                                       (6, 37, 96), (6, 18944, 3584), (7, 37, 96),
                                       (7, 3584, 18944), (1, 37, 96), (1, 130, 800),
                                       (30, 37, 96), (30, 4864, 896)])
def test_decode_plane_roundtrip_is_byte_exact(qtype, N, K):
    W = registered(qtype, N, K, 7)
    assert np.array_equal(W.unpack(), weights(qtype, N, K, 7))
    t, n, k, nbytes = W.info()
    assert (t, n, k) == (qtype, N, K) and nbytes > 0


# ---- decode matvec -----------------------------------------------------------

SMALL = [(8, 1, 32), (8, 37, 96), (8, 130, 288), (8, 64, 896),
         (12, 1, 256), (12, 19, 512), (12, 100, 768), (12, 257, 2560),
         (14, 1, 256), (14, 21, 768), (14, 130, 512), (14, 64, 4608),
         (2, 1, 32), (2, 37, 96), (2, 130, 288), (2, 64, 896), (2, 300, 4864),
         (13, 1, 256), (13, 19, 512), (13, 100, 768), (13, 257, 2560),
         (3, 1, 32), (3, 37, 96), (3, 130, 288), (3, 300, 4864),
         (6, 1, 32), (6, 37, 96), (6, 130, 288), (6, 300, 4864),
         (7, 1, 32), (7, 37, 96), (7, 130, 288), (7, 300, 4864),
         (1, 1, 32), (1, 37, 96), (1, 130, 288), (1, 300, 4864),
         (30, 1, 32), (30, 37, 96), (30, 130, 288), (30, 300, 4864)]


@pytest.mark.parametrize("qtype,N,K", SMALL)
@pytest.mark.parametrize("B", [1, 3, 8])
def test_matvec_small_shapes(qtype, N, K, B):
    W = registered(qtype, N, K, 11)
    x = synth.activations(B, K, seed=100 + B)
    y = gpu_matvec(W, x)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, 11), N, K, x)
    assert_bound(y, yref, bnd, f"type {qtype} {N}x{K} B={B}")


@pytest.mark.parametrize("name,B", [("q8_0_matvec_896x896", 1), ("q4_k_matvec_18944x3584", 1),
                                    ("q6_k_matvec_3584x18944", 1), ("q6_k_matvec_3584x18944", 2),
                                    ("q6_k_matvec_3584x18944", 4), ("q6_k_matvec_3584x18944", 8),
                                    ("q6_k_lm_head_151936x3584", 1)])
def test_matvec_workloads_full(name, B):
    c = synth.WORKLOADS[name]
    qtype, N, K = c["qtype"], c["N"], c["K"]
    W = registered(qtype, N, K, c["w_seed"])
    x = synth.activations(B, K, c["x_seed"], c["x_scale"])
    y = gpu_matvec(W, x)
    # every output element; the LM head's 151936 rows on all host cores (the oracle's
    # OpenMP build, the same bits as the plain one)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, c["w_seed"]), N, K, x,
                              parallel=N > 20000)
    assert_bound(y, yref, bnd, name)


@pytest.mark.parametrize("qtype", [12, 13, 14])
@pytest.mark.parametrize("B", [1, 2, 4, 5, 8])
def test_matvec_persistent_kernel_several_groups_per_cta(qtype, B):
    """Weights of at least SMs / 2 row groups run the persistent kernel; at 39000 rows each CTA
    takes two or three 128-row groups in turn (the last one ragged), and every column of the
    batch equals the B = 1 call bit for bit."""
    N, K = 39000, 768
    W = registered(qtype, N, K, 19)
    x = synth.activations(B, K, seed=200 + B)
    y = gpu_matvec(W, x)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, 19), N, K, x, parallel=True)
    assert_bound(y, yref, bnd, f"type {qtype} {N}x{K} B={B}")
    y1 = gpu_matvec(W, x[B - 1:B])
    assert np.array_equal(y1[0].view(np.uint32), y[B - 1].view(np.uint32))


def test_matvec_batch_columns_equal_single_calls_bitwise():
    c = synth.WORKLOADS["q6_k_matvec_3584x18944"]
    W = registered(c["qtype"], c["N"], c["K"], c["w_seed"])
    x = synth.activations(8, c["K"], c["x_seed"], 1.0)
    y8 = gpu_matvec(W, x)
    for b in range(8):
        y1 = gpu_matvec(W, x[b:b + 1])
        assert np.array_equal(y1[0].view(np.uint32), y8[b].view(np.uint32)), b
    y3 = gpu_matvec(W, x[2:5])
    assert np.array_equal(y3.view(np.uint32), y8[2:5].view(np.uint32))


@pytest.mark.parametrize("qtype,N,K", [(8, 70, 288), (12, 70, 768), (14, 70, 768),
                                       (2, 70, 288), (13, 70, 768), (3, 70, 288), (6, 70, 288),
                                       (7, 70, 288), (1, 70, 288), (30, 70, 288)])
def test_matvec_extreme_magnitudes(qtype, N, K):
    W = registered(qtype, N, K, 13)
    rng = np.random.default_rng(5)
    x = synth.activations(4, K, seed=6)
    x[0] *= np.float32(1e30)       # f16 would overflow without the per-chunk exponent
    x[1] *= np.float32(1e-30)      # and underflow
    x[2, : K // 2] *= np.float32(1e20)
    x[2, K // 2:] *= np.float32(1e-10)  # chunks of very different range
    x[3] = 0.0
    x[3, rng.integers(0, K, 5)] = np.float32(3.0)
    y = gpu_matvec(W, x)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, 13), N, K, x)
    assert_bound(y, yref, bnd, f"extreme type {qtype}")
    y0 = gpu_matvec(W, np.zeros((2, K), np.float32))
    assert np.all(y0 == 0.0)


# ---- activation quantiser ----------------------------------------------------

def gpu_quantize(x):
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    M, K = x.shape
    xq = mq.quantize_act(xt)
    torch.cuda.synchronize()
    qs, sc, bs, op = (v.cpu().numpy() for v in mq.act_views(xq, M, K))
    return xq, qs, sc, bs, op


def assert_quant_exact(x):
    xq, qs, sc, bs, op = gpu_quantize(x)
    rq, rs, rb = oracle.quantize_act(x)
    assert np.array_equal(qs, rq)
    assert np.array_equal(sc.view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(bs, rb)
    assert np.array_equal(op.astype(np.float32), rq.astype(np.float32))
    st, tt = (v.cpu().numpy() for v in mq.act_views_transposed(xq, *x.shape))
    assert np.array_equal(st.T.view(np.uint32), rs.view(np.uint32))
    with np.errstate(over="ignore"):
        assert np.array_equal(tt.T, rs * rb.astype(np.float32))
    assert_min_operand(xq, rs, rb)


def assert_min_operand(xq, rs, rb):
    """The min-term operand sections against their definition (mq.h, mq_act_bytes):
    u_m = 2^k, k = E - 140 clamped to [-100, 100] with E the biased binary32 exponent of
    max_b |s*S| (so max/u_m is in [2^13, 2^14) for a normal maximum; k = 0 for an all-zero
    row and 100 for an infinite one); t = s*S / u_m; hi = f16(t); lo = f16(t - hi);
    row = hi | hi | lo.  Operand bytes are compared on rows whose s*S are all finite."""
    M, nb = rs.shape
    am, ur = (v.cpu().numpy() for v in mq.act_views_min(xq, M, nb * 32))
    with np.errstate(over="ignore", invalid="ignore"):
        t = (rs * rb.astype(np.float32)).astype(np.float32)
        mx = np.abs(t).max(axis=1).astype(np.float32)
        E = ((mx.view(np.uint32) >> 23) & 255).astype(np.int64)
        k = np.where(mx == 0, 0, np.clip(E - 140, -100, 100))
        u = np.ldexp(np.float32(1), k).astype(np.float32)
        assert np.array_equal(ur.view(np.uint32), u.view(np.uint32))
        fin = np.isfinite(mx)
        ts = (t / u[:, None]).astype(np.float32)[fin]
        hi = ts.astype(np.float16)
        lo = (ts - hi.astype(np.float32)).astype(np.float16)
    am = am.view(np.uint16)[fin]
    assert np.array_equal(am[:, :nb], hi.view(np.uint16))
    assert np.array_equal(am[:, nb:2 * nb], hi.view(np.uint16))
    assert np.array_equal(am[:, 2 * nb:], lo.view(np.uint16))


@pytest.mark.parametrize("name,M", [("q4_k_mmq_512x18944x3584", 512),
                                    ("q6_k_lm_head_151936x3584", 2048)])
def test_quantize_workloads_bit_exact(name, M):
    c = synth.WORKLOADS[name]
    assert_quant_exact(synth.activations(M, c["K"], c["x_seed"], c["x_scale"]))


@pytest.mark.parametrize("M,K", [(1, 32), (7, 96), (65, 288), (3, 4096)])
def test_quantize_small_and_edge_blocks(M, K):
    quantize_edge_blocks(M, K)


def quantize_edge_blocks(M, K):
    x = synth.activations(M, K, seed=M * 7 + K)
    x[0, :32] = 0.0                                   # s = 0 block
    if K >= 64:
        x[0, 32:64] = np.float32(1e-41)               # subnormal block
    if M > 1:
        s = np.float32(0.125)
        x[1, :32] = s * np.array([127, 2.5, -2.5, 3.5, 0.5, -0.5, 1.5, -1.5] * 4, np.float32)
    if M > 2:
        x[2, :32] = np.float32(3e38) * np.sign(x[2, :32])  # near the f32 maximum
    assert_quant_exact(x)


# ---- MMQ -------------------------------------------------------------------

SMALL_MMQ = [(8, 37, 96, 5), (8, 130, 288, 70), (12, 19, 512, 9), (12, 200, 768, 65),
             (14, 21, 768, 3), (14, 130, 512, 129),
             (2, 37, 96, 5), (2, 130, 288, 70), (13, 19, 512, 9), (13, 200, 768, 65),
             (3, 37, 96, 5), (3, 130, 288, 70), (6, 37, 96, 5), (6, 130, 288, 70),
             (7, 37, 96, 5), (7, 130, 288, 70), (7, 200, 800, 131)]


@pytest.mark.parametrize("qtype,N,K,M", SMALL_MMQ)
def test_blockdots_bit_exact_small(qtype, N, K, M):
    W = registered(qtype, N, K, 17)
    x = synth.activations(M, K, seed=M + K)
    xq, qs, _, _, _ = gpu_quantize(x)
    D = mq.mmq_blockdots(W, xq, M)
    torch.cuda.synchronize()
    ref = oracle.blockdots(qtype, weights(qtype, N, K, 17), N, K, qs)
    assert np.array_equal(D.cpu().numpy(), ref.astype(np.int32))


# A Q4_K weight registered with MQ_REG_MMQ_FROM_DECODE_PLANE has no f16 integer plane: the
# MMQ copies the decode-plane tiles (one 256-element chunk per bulk copy, three chunk slots)
# and expands them in shared memory.  Shapes with one chunk per tile, one tile per CTA with
# the in-loop chunk prefetch, and two or three tiles per CTA whose chunk sequence continues
# across tiles; ragged N and M.  Block dots bit-exact against the oracle, y within its bound
# and bit-identical to the default registration's (the same integers reach the MMA), also
# through the fused quantise + MMQ.
@pytest.mark.parametrize("N,K,M", [(25637, 256, 130), (2437, 768, 300), (12805, 768, 257)])
def test_q4k_mmq_from_decode_plane_tiles(N, K, M):
    qtype = 12
    W = registered(qtype, N, K, 23, mq.REG_MMQ_FROM_DECODE_PLANE)
    Wd = registered(qtype, N, K, 23)
    assert W.info()[3] == Wd.info()[3] - N * K * 2  # the f16 plane alone is missing
    x = synth.activations(M, K, seed=M + 3 * K)
    xq, qs, sc, _, _ = gpu_quantize(x)
    D = mq.mmq_blockdots(W, xq, M)
    y = mq.mmq(W, xq, M)
    yd = mq.mmq(Wd, xq, M)
    yf, _ = mq.mmq_fused(W, torch.from_numpy(x).cuda(), mq.act_buffer(M, K))
    torch.cuda.synchronize()
    mq.stream_status()
    assert np.array_equal(y.cpu().numpy(), yd.cpu().numpy())
    assert np.array_equal(yf.cpu().numpy(), yd.cpu().numpy())
    wb = weights(qtype, N, K, 23)
    ref = oracle.blockdots(qtype, wb, N, K, qs)
    assert np.array_equal(D.cpu().numpy(), ref.astype(np.int32))
    if N * K * M <= 2437 * 768 * 300:
        yref, bnd = oracle.mmq(qtype, wb, N, K, qs, sc)
        assert_bound(y.cpu().numpy(), yref, bnd, f"Q4_K {M}x{N}x{K}")


@pytest.mark.parametrize("name", ["q4_k_mmq_512x18944x3584", "q6_k_lm_head_151936x3584"])
def test_blockdots_bit_exact_workload_tiles(name):
    """A 128 x 256 x (all blocks) tile of each prefill workload: the first 256 weight rows
    and 128 activation rows, with the workload's distributions and seeds."""
    c = synth.WORKLOADS[name]
    qtype, K = c["qtype"], c["K"]
    rowbytes = K // 256 * synth.BLOCK[qtype][1]
    Wfull = weights(qtype, c["N"], K, c["w_seed"])
    Wt = np.ascontiguousarray(Wfull[:256 * rowbytes])
    W = mq.register_weight(qtype, Wt, 256, K)
    x = synth.activations(128, K, c["x_seed"], c["x_scale"])
    xq, qs, _, _, _ = gpu_quantize(x)
    D = mq.mmq_blockdots(W, xq, 128)
    torch.cuda.synchronize()
    ref = oracle.blockdots(qtype, Wt, 256, K, qs)
    assert np.array_equal(D.cpu().numpy(), ref.astype(np.int32))
    W.free()


@pytest.mark.parametrize("qtype", [12, 3])
@pytest.mark.parametrize("N,K,M", [(19, 256, 9), (70, 8192, 5), (130, 3584, 130)])
def test_mmq_min_term_stages(qtype, N, K, M):
    """Min-term GEMM (Q4_K sub-block mins, Q4_1 block mins) over 1, 12 (two rounds of the
    operand ring) and 6 stages."""
    W = registered(qtype, N, K, 23)
    x = synth.activations(M, K, seed=K + M)
    xq, qs, sc, _, _ = gpu_quantize(x)
    y = mq.mmq(W, xq, M)
    torch.cuda.synchronize()
    mq.stream_status()
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, 23), N, K, qs, sc)
    assert_bound(y.cpu().numpy(), yref, bnd, f"mmq type {qtype} {M}x{N}x{K}")


@pytest.mark.parametrize("qtype,N,K,M", SMALL_MMQ)
def test_mmq_small_shapes(qtype, N, K, M):
    W = registered(qtype, N, K, 17)
    x = synth.activations(M, K, seed=M + K)
    xq, qs, sc, _, _ = gpu_quantize(x)
    y = mq.mmq(W, xq, M)
    torch.cuda.synchronize()
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, 17), N, K, qs, sc)
    assert_bound(y.cpu().numpy(), yref, bnd, f"mmq type {qtype} {M}x{N}x{K}")


def test_mmq_prefill_workload_full():
    """The Q4_K prefill workload (M = 512, N = 18944, K = 3584) compared on every output
    element, the oracle's rows on all host cores."""
    c = synth.WORKLOADS["q4_k_mmq_512x18944x3584"]
    qtype, N, K, M = c["qtype"], c["N"], c["K"], c["M"][0]
    W = registered(qtype, N, K, c["w_seed"])
    x = synth.activations(M, K, c["x_seed"], c["x_scale"])
    xq, qs, sc, _, _ = gpu_quantize(x)
    y = mq.mmq(W, xq, M)
    torch.cuda.synchronize()
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, c["w_seed"]), N, K, qs, sc,
                           parallel=True)
    assert_bound(y.cpu().numpy(), yref, bnd, "q4_k_mmq_512x18944x3584 (all outputs)")


@pytest.mark.parametrize("name", ["q4_k_mmq_512x18944x3584", "q6_k_lm_head_151936x3584"])
def test_mmq_workloads_sampled(name):
    c = synth.WORKLOADS[name]
    qtype, N, K, M = c["qtype"], c["N"], c["K"], c["M"][0]
    W = registered(qtype, N, K, c["w_seed"])
    x = synth.activations(M, K, c["x_seed"], c["x_scale"])
    xq, qs, sc, _, _ = gpu_quantize(x)
    y = mq.mmq(W, xq, M)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    rng = np.random.default_rng(1)
    rows = sorted(set([0, 1, M // 4 - 1, M // 2, M - 1] + list(rng.integers(0, M, 11))))
    # all N columns of the sampled rows (the LM head's 2048 x 151936 outputs in full would
    # be about 10^12 double multiply-adds)
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, c["w_seed"]), N, K, qs, sc, mrows=rows,
                           parallel=True)
    assert_bound(y[rows], yref, bnd, f"{name} sampled rows")
    assert np.isfinite(y).all()


def test_bounded_wait_expiry_is_reported_and_the_result_stays_correct(monkeypatch):
    """With the failure-injection seam, the MMQ epilogue waits on a barrier nothing
    arrives on; the bounded wait expires, the status word reports MQ_ERR_TIMEOUT,
    and the kernel finishes with the correct result (the context stays usable)."""
    qtype, N, K, M = 12, 200, 768, 65
    W = registered(qtype, N, K, 17)
    x = synth.activations(M, K, seed=M + K)
    xq, qs, sc, _, _ = gpu_quantize(x)
    mq.stream_status()
    monkeypatch.setenv("MQ_TEST_EXPIRE_WAIT", "1")
    mq.init(0)  # the seams are read by mq_init
    y = mq.mmq(W, xq, M)
    with pytest.raises(mq.MQError) as e:
        mq.stream_status()
    assert e.value.name == "MQ_ERR_TIMEOUT"
    monkeypatch.delenv("MQ_TEST_EXPIRE_WAIT")
    mq.init(0)
    mq.stream_status()  # cleared
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, 17), N, K, qs, sc)
    assert_bound(y.cpu().numpy(), yref, bnd, "after an expired wait")
    y2 = mq.mmq(W, xq, M)
    mq.stream_status()
    assert np.array_equal(y.cpu().numpy(), y2.cpu().numpy())


# ---- errors on the device path -----------------------------------------------

def test_errors_are_reported_not_fallen_back():
    W = registered(12, 19, 512, 17)
    x = torch.zeros((1, 512), device="cuda")
    y = torch.zeros((1, 19), device="cuda")
    L = mq.lib()
    P = lambda t: t.data_ptr()
    st = L.mq_matvec(14, W.handle, P(x), P(y), 19, 512, 1, None)
    assert mq.STATUS[st] == "MQ_ERR_TYPE"
    st = L.mq_matvec(12, W.handle, P(x), P(y), 20, 512, 1, None)
    assert mq.STATUS[st] == "MQ_ERR_SHAPE"
    for B in (0, 9):
        assert mq.STATUS[L.mq_matvec(12, W.handle, P(x), P(y), 19, 512, B, None)] == "MQ_ERR_ARG"
    xh = np.zeros(512, np.float32)
    st = L.mq_matvec(12, W.handle, xh.ctypes.data, P(y), 19, 512, 1, None)
    assert mq.STATUS[st] == "MQ_ERR_ARG" and "host memory" in L.mq_last_error().decode() or \
        "not a CUDA pointer" in L.mq_last_error().decode()
    yb = torch.zeros(64, device="cuda")
    st = L.mq_matvec(12, W.handle, P(x), P(yb) + 4, 19, 512, 1, None)
    assert mq.STATUS[st] == "MQ_ERR_ALIGN"
    Wn = mq.register_weight(12, weights(12, 19, 512, 17), 19, 512, mq.REG_NO_MMQ_PLANE)
    xq = mq.quantize_act(torch.zeros((4, 512), device="cuda"))
    with pytest.raises(mq.MQError) as e:
        mq.mmq(Wn, xq, 4)
    assert e.value.name == "MQ_ERR_ARG"
    Wn.free()
    mq.stream_status()


# ---- the Q4_0, Q4_1, Q5_0, Q5_1 and Q5_K types at model-sized shapes -----------

@pytest.mark.parametrize("qtype,N,K,B", [(2, 4864, 896, 1), (2, 18944, 3584, 4),
                                         (13, 18944, 3584, 1), (13, 3584, 18944, 8),
                                         (3, 18944, 3584, 1), (3, 4864, 896, 8),
                                         (6, 18944, 3584, 2), (6, 3584, 18944, 1),
                                         (7, 18944, 3584, 1), (7, 3584, 18944, 5),
                                         (1, 4864, 896, 1), (1, 3584, 18944, 8),
                                         (30, 18944, 3584, 1), (30, 896, 4864, 3)])
def test_matvec_new_types_ffn_shapes(qtype, N, K, B):
    W = registered(qtype, N, K, 41, mq.REG_NO_MMQ_PLANE)
    x = synth.activations(B, K, seed=42)
    y = gpu_matvec(W, x)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, 41), N, K, x)
    assert_bound(y, yref, bnd, f"type {qtype} {N}x{K} B={B}")


@pytest.mark.parametrize("qtype", [2, 13, 3, 6, 7])
def test_mmq_new_types_prefill_shape_sampled(qtype):
    N, K, M = 18944, 3584, 512
    W = registered(qtype, N, K, 43)
    x = synth.activations(M, K, seed=44)
    xq, qs, sc, _, _ = gpu_quantize(x)
    y = mq.mmq(W, xq, M)
    torch.cuda.synchronize()
    mq.stream_status()
    rows = np.array([0, 127, 128, 300, 511])
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, 43), N, K, qs, sc, mrows=rows)
    assert_bound(y.cpu().numpy()[rows], yref, bnd, f"mmq type {qtype} 512x18944x3584")


@pytest.mark.parametrize("qtype", [1, 30])
def test_float_weights_have_no_mmq_form(qtype):
    N, K = 40, 96
    W = mq.register_weight(qtype, weights(qtype, N, K, 3), N, K)
    xq = mq.quantize_act(torch.zeros((4, K), device="cuda"))
    with pytest.raises(mq.MQError) as e:
        mq.mmq(W, xq, 4)
    assert e.value.name == "MQ_ERR_TYPE"
    with pytest.raises(mq.MQError) as e:
        mq.mmq_blockdots(W, xq, 4)
    assert e.value.name == "MQ_ERR_TYPE"
    W.free()
    mq.stream_status()


def test_refused_launches_are_reported_and_leave_no_error(monkeypatch):
    """With the failure-injection seam the matvec and MMQ launches get an empty grid, which
    the runtime refuses before any kernel runs: the call returns MQ_ERR_LAUNCH naming the
    kernel, and the next calls run normally and stay within the oracle's bound."""
    qtype, N, K, M = 12, 200, 768, 9
    W = registered(qtype, N, K, 17)
    x = synth.activations(2, K, seed=3)
    xa = synth.activations(M, K, seed=4)
    xq, qs, sc, _, _ = gpu_quantize(xa)
    monkeypatch.setenv("MQ_TEST_FAIL_LAUNCH", "1")
    mq.init(0)  # the seams are read by mq_init
    with pytest.raises(mq.MQError) as e:
        mq.matvec(W, torch.from_numpy(x).cuda())
    assert e.value.name == "MQ_ERR_LAUNCH" and "matvec_kernel<Q4_K" in str(e.value)
    with pytest.raises(mq.MQError) as e:
        mq.mmq(W, xq, M)
    assert e.value.name == "MQ_ERR_LAUNCH" and "mmq_tc_kernel<Q4_K" in str(e.value)
    monkeypatch.delenv("MQ_TEST_FAIL_LAUNCH")
    mq.init(0)
    y = gpu_matvec(W, x)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, 17), N, K, x)
    assert_bound(y, yref, bnd, "matvec after a refused launch")
    ym = mq.mmq(W, xq, M)
    torch.cuda.synchronize()
    mq.stream_status()
    yref, bnd = oracle.mmq(qtype, weights(qtype, N, K, 17), N, K, qs, sc)
    assert_bound(ym.cpu().numpy(), yref, bnd, "mmq after a refused launch")


@pytest.mark.parametrize("qtype,N,K", [(1, 700, 2080), (30, 700, 2080), (2, 700, 2080),
                                       (3, 700, 2080), (6, 700, 2080), (7, 700, 2080),
                                       (8, 700, 2080), (12, 700, 2048), (13, 700, 2048),
                                       (14, 700, 2048)])
def test_batch_columns_equal_single_calls_bitwise_every_type(qtype, N, K):
    """Every column of a B = 8 (two-tile kernel) and a B = 3 call equals the B = 1 call bit for
    bit: the K split and the accumulation order depend on (N, K) only."""
    W = registered(qtype, N, K, 51, mq.REG_NO_MMQ_PLANE)
    x = synth.activations(8, K, seed=52)
    y8 = gpu_matvec(W, x)
    y3 = gpu_matvec(W, x[3:6])
    for b in range(8):
        y1 = gpu_matvec(W, x[b:b + 1])
        assert np.array_equal(y1[0].view(np.uint32), y8[b].view(np.uint32)), (qtype, b)
    assert np.array_equal(y3.view(np.uint32), y8[3:6].view(np.uint32))


@pytest.mark.parametrize("qtype,N,K", [(8, 300, 4864), (12, 300, 4864), (14, 300, 4864),
                                       (3, 1000, 8192)])
def test_wide_k_split_over_large_clusters(qtype, N, K):
    """Few row groups and many chunks: the K split goes past the portable cluster size (up to
    16 CTAs per cluster, where every cluster fits at once); the result stays within the bound
    and every column of a B = 8 call equals its B = 1 call bit for bit."""
    W = registered(qtype, N, K, 53, mq.REG_NO_MMQ_PLANE)
    x = synth.activations(8, K, seed=54)
    y8 = gpu_matvec(W, x)
    yref, bnd = oracle.matvec(qtype, weights(qtype, N, K, 53), N, K, x)
    assert_bound(y8, yref, bnd, f"type {qtype} {N}x{K} B=8")
    for b in (0, 5, 7):
        y1 = gpu_matvec(W, x[b:b + 1])
        assert np.array_equal(y1[0].view(np.uint32), y8[b].view(np.uint32)), (qtype, b)


def test_host_buffer_calls_equal_the_device_calls():
    """mq_matvec_host / mq_mmq_host give the device-pointer calls' results bit for bit on both
    transfer routes: page-locked aligned buffers (the kernels read and write them through
    their device views, so the matvec's y_dev and the prefill's x_dev stay untouched) and
    pageable or misaligned ones (copies through x_dev / y_dev).  A device pointer is refused as a host
    buffer."""
    qtype, N, K, B, M = 12, 700, 2048, 3, 70
    W = registered(qtype, N, K, 17)
    x, a = synth.activations(B, K, seed=81), synth.activations(M, K, seed=82)
    yref = mq.matvec(W, torch.from_numpy(x).cuda()).cpu()
    mref = mq.mmq(W, mq.quantize_act(torch.from_numpy(a).cuda()), M).cpu()
    xq = torch.empty(mq.act_bytes(M, K), dtype=torch.uint8, device="cuda")
    nan = float("nan")

    def bits_equal(u, v):
        return torch.equal(u.contiguous().view(torch.int32), v.contiguous().view(torch.int32))

    # page-locked, aligned: direct access
    xh, ah = torch.from_numpy(x).pin_memory(), torch.from_numpy(a).pin_memory()
    yh, mh = torch.full((B, N), nan).pin_memory(), torch.full((M, N), nan).pin_memory()
    xd, yd = torch.empty((B, K), device="cuda"), torch.full((B, N), nan, device="cuda")
    ad, md = torch.full((M, K), nan, device="cuda"), torch.full((M, N), nan, device="cuda")
    mq.matvec_host(W, xh, yh, xd, yd)
    mq.mmq_host(W, ah, mh, ad, xq, md)
    torch.cuda.synchronize()
    mq.stream_status()
    assert bits_equal(yh, yref) and bits_equal(mh, mref)
    assert torch.equal(xd.cpu(), xh)  # the matvec's x is pulled into x_dev
    assert torch.isnan(yd).all() and torch.isnan(ad).all()  # y and the prefill's x go direct
    assert bits_equal(md.cpu(), mref)  # the prefill's y goes out through y_dev

    # pageable: copies through the device buffers
    yp, mp = torch.full((B, N), nan), torch.full((M, N), nan)
    mq.matvec_host(W, torch.from_numpy(x.copy()), yp, xd, yd)
    mq.mmq_host(W, torch.from_numpy(a.copy()), mp, ad, xq, md)
    torch.cuda.synchronize()
    mq.stream_status()
    assert bits_equal(yp, yref) and bits_equal(mp, mref)
    assert bits_equal(yd.cpu(), yref) and bits_equal(md.cpu(), mref)

    # page-locked but 4 bytes off a 16-byte boundary: copies as well
    xbig, ybig = torch.empty(B * K + 1).pin_memory(), torch.full((B * N + 1,), nan).pin_memory()
    abig, mbig = torch.empty(M * K + 1).pin_memory(), torch.full((M * N + 1,), nan).pin_memory()
    xm, ym = xbig[1:].view(B, K), ybig[1:].view(B, N)
    am, mm = abig[1:].view(M, K), mbig[1:].view(M, N)
    xm.copy_(torch.from_numpy(x))
    am.copy_(torch.from_numpy(a))
    yd.fill_(nan)
    md.fill_(nan)
    mq.matvec_host(W, xm, ym, xd, yd)
    mq.mmq_host(W, am, mm, ad, xq, md)
    torch.cuda.synchronize()
    mq.stream_status()
    assert bits_equal(ym, yref) and bits_equal(mm, mref)
    assert bits_equal(yd.cpu(), yref) and bits_equal(md.cpu(), mref)

    with pytest.raises(mq.MQError) as e:
        mq.matvec_host(W, xd, yh, xd, yd)  # x_host is device memory
    assert e.value.name == "MQ_ERR_ARG" and "host buffer" in str(e.value)
