"""Seeded random shapes for every weight type, against the oracle through the C ABI: the
decode matvec (B = 1..8) and, for the quantised types, the block dots (bit-exact), the MMQ
and the fused quantise + MMQ (within the bound).  Shapes are drawn so that K spans partial
chunks and super-blocks, N spans partial row groups and tiles, M partial tiles; the same
seed always draws the same cases.  Plus concurrent calls on two streams."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quantized_q4_gb300 as mq  # noqa: E402
from gguf_block_quantized_q4_gb300 import build as mqbuild  # noqa: E402

TYPES = [synth.F16, synth.BF16, synth.Q4_0, synth.Q4_1, synth.Q5_0, synth.Q5_1, synth.Q8_0,
         synth.Q4_K, synth.Q5_K, synth.Q6_K]
REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mqbuild.build()
    mq.init(0)
    yield


def draw(seed):
    rng = np.random.default_rng(seed)
    qtype = TYPES[seed % len(TYPES)]
    be = 256 if qtype in (synth.Q4_K, synth.Q5_K, synth.Q6_K) else 32
    K = be * int(rng.integers(1, 2048 // be + 3))
    N = int(rng.integers(1, 700))
    B = int(rng.integers(1, 9))
    M = int(rng.integers(1, 300))
    return qtype, N, K, B, M


def within(y, yref, bnd, what):
    err = np.abs(np.asarray(y, np.float64) - yref)
    assert (err <= REL * bnd + 1e-37).all(), (
        f"{what}: worst err/bound {np.max(err / np.maximum(bnd, 1e-300)):.3e}")


@pytest.mark.parametrize("seed", range(40))
def test_random_shape(seed):
    qtype, N, K, B, M = draw(1000 + seed)
    raw = synth.weights(qtype, N, K, 2000 + seed)
    quantised = qtype not in (synth.F16, synth.BF16)
    W = mq.register_weight(qtype, raw, N, K)
    what = f"seed {seed}: type {qtype} N={N} K={K}"
    x = synth.activations(B, K, 3000 + seed)
    y = mq.matvec(W, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    yref, bnd = oracle.matvec(qtype, raw, N, K, x)
    within(y.cpu().numpy(), yref, bnd, what + f" matvec B={B}")
    if quantised:
        xa = synth.activations(M, K, 4000 + seed)
        xq = mq.quantize_act(torch.from_numpy(xa).cuda())
        D = mq.mmq_blockdots(W, xq, M)
        ym = mq.mmq(W, xq, M)
        yf, _ = mq.mmq_fused(W, torch.from_numpy(xa).cuda())
        torch.cuda.synchronize()
        mq.stream_status()
        qs, sc, _ = oracle.quantize_act(xa)
        rows = np.unique(np.linspace(0, M - 1, min(M, 9)).astype(np.int64))
        Dref = oracle.blockdots(qtype, raw, N, K, qs, mrows=rows)
        assert np.array_equal(D.cpu().numpy()[rows], Dref.astype(np.int32)), what + " blockdots"
        yref, bnd = oracle.mmq(qtype, raw, N, K, qs, sc, mrows=rows)
        within(ym.cpu().numpy()[rows], yref, bnd, what + f" mmq M={M}")
        assert torch.equal(yf.view(torch.int32), ym.view(torch.int32)), what + " fused"
    W.free()


def test_concurrent_streams():
    """Matvecs and MMQs of two weights issued on two streams at once give the results of
    the same calls issued one after the other (the calls share only read-only state)."""
    cases = [(synth.Q4_K, 3000, 3584), (synth.Q6_K, 2000, 4096)]
    Ws = [mq.register_weight(q, synth.weights(q, N, K, 5 + i), N, K)
          for i, (q, N, K) in enumerate(cases)]
    xs = [torch.from_numpy(synth.activations(4, K, 6 + i)).cuda() for i, (_, _, K) in enumerate(cases)]
    xa = [torch.from_numpy(synth.activations(200, K, 8 + i)).cuda() for i, (_, _, K) in enumerate(cases)]
    ref = []
    for W, x, a in zip(Ws, xs, xa):
        xq = mq.quantize_act(a)
        ref.append((mq.matvec(W, x), mq.mmq(W, xq, a.shape[0])))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    out = []
    for W, x, a, s in zip(Ws, xs, xa, streams):
        with torch.cuda.stream(s):
            res = []
            for _ in range(5):
                xq = mq.quantize_act(a, stream=s)
                res.append((mq.matvec(W, x, stream=s), mq.mmq(W, xq, a.shape[0], stream=s)))
            out.append(res)
    torch.cuda.synchronize()
    mq.stream_status()
    for (yv, ym), res in zip(ref, out):
        for rv, rm in res:
            assert torch.equal(rv.view(torch.int32), yv.view(torch.int32))
            assert torch.equal(rm.view(torch.int32), ym.view(torch.int32))
    for W in Ws:
        W.free()
