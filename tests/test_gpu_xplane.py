"""Two-tile calls (B = 5..8) of the persistent decode matvec on Q4_K / Q5_K weights (of at
least SMs / 2 row groups) convert x once per call into an activation fragment plane, a
per-call buffer from the library's stream-ordered pool, that every CTA copies from.  These
check the forms that plane takes part in beyond the single eager call (which the parity tests
cover): calls captured in a CUDA graph (allocation and free nodes), and calls on two streams at
once on the same weight (each with its own plane).  B = 3 (no plane), a Q6_K weight (no plane)
and a split-K weight are controls."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quantized_q4_gb300 as mq  # noqa: E402
from gguf_block_quantized_q4_gb300 import build as mqbuild  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mqbuild.build()
    mq.init(0)
    yield


def bits(t):
    return t.contiguous().view(torch.int32).cpu().numpy()


# persistent-kernel weights (148 or more row groups; Q6_K with a ragged last group) and a
# split-K weight (Q6_K, 6 row groups)
CASES = [(12, 18944, 1024, 61), (13, 18944, 768, 65), (14, 20000, 512, 66), (14, 700, 2048, 62)]


@pytest.mark.parametrize("qtype,N,K,seed", CASES)
@pytest.mark.parametrize("B", [3, 5, 8])
def test_graph_captured_batched_calls_equal_eager_calls(qtype, N, K, seed, B):
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, seed), N, K, mq.REG_NO_MMQ_PLANE)
    xs = [torch.from_numpy(synth.activations(B, K, seed=seed + 10 * r)).cuda() for r in range(3)]
    ys = [torch.empty((B, N), device="cuda") for _ in range(3)]
    eager = [mq.matvec(W, x) for x in xs]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for x, y in zip(xs, ys):
                mq.matvec(W, x, y)
    for _ in range(3):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for y, e in zip(ys, eager):
            assert np.array_equal(bits(y), bits(e))
    mq.stream_status()
    W.free()


def test_two_streams_at_once_on_one_weight():
    qtype, N, K = 12, 18944, 2048
    wb = synth.weights(qtype, N, K, 64)
    W = mq.register_weight(qtype, wb, N, K, mq.REG_NO_MMQ_PLANE)
    B, reps = 8, 20
    xa = [torch.from_numpy(synth.activations(B, K, seed=70 + r)).cuda() for r in range(2)]
    ref = [mq.matvec(W, x) for x in xa]
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = [[torch.empty((B, N), device="cuda") for _ in range(reps)] for _ in range(2)]
    for s in (sa, sb):
        s.wait_stream(torch.cuda.current_stream())
    for i in range(reps):
        for j, s in enumerate((sa, sb)):
            with torch.cuda.stream(s):
                mq.matvec(W, xa[j], outs[j][i], stream=s)
    torch.cuda.synchronize()
    for j in range(2):
        for y in outs[j]:
            assert np.array_equal(bits(y), bits(ref[j])), j
    yref, bnd = oracle.matvec(qtype, wb, N, K, xa[1].cpu().numpy(), parallel=True)
    err = np.abs(ref[1].cpu().numpy().astype(np.float64) - yref)
    assert (err <= 1e-4 * bnd + 1e-37).all()
    mq.stream_status()
    W.free()


@pytest.mark.parametrize("qtype", [12, 13])
def test_without_the_plane_the_same_bits(monkeypatch, qtype):
    """With MQ_TEST_NO_XPLANE=1 at mq_init (the path taken when the pool cannot give a plane)
    the x warps convert x themselves at two tiles: the result equals the plane's bit for bit
    and stays within the oracle's bound."""
    N, K, B = 18944, 1024, 8
    wb = synth.weights(qtype, N, K, 67)
    W = mq.register_weight(qtype, wb, N, K, mq.REG_NO_MMQ_PLANE)
    x = torch.from_numpy(synth.activations(B, K, seed=68)).cuda()
    with_plane = mq.matvec(W, x)
    torch.cuda.synchronize()
    monkeypatch.setenv("MQ_TEST_NO_XPLANE", "1")
    mq.init(0)
    try:
        without = mq.matvec(W, x)
        torch.cuda.synchronize()
    finally:
        monkeypatch.delenv("MQ_TEST_NO_XPLANE")
        mq.init(0)
    assert np.array_equal(bits(without), bits(with_plane))
    yref, bnd = oracle.matvec(qtype, wb, N, K, x.cpu().numpy(), parallel=True)
    err = np.abs(without.cpu().numpy().astype(np.float64) - yref)
    assert (err <= 1e-4 * bnd + 1e-37).all()
    mq.stream_status()
    W.free()
