"""The quantiser and the MMQ (and the matvec) are launched with programmatic stream
serialisation: a launch may start while the previous kernel in the stream is finishing, and
waits for it before it reads what that kernel writes, or writes what it reads.  This chains
quantise -> MMQ -> matvec -> quantise -> MMQ ... on one stream with every call reusing the
same xq buffer (so a quantiser that wrote xq before the previous MMQ had finished reading it
would change that MMQ's result), eagerly and captured into a graph, and checks every result
bit for bit against calls separated by device synchronisation."""
import numpy as np
import pytest

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


@pytest.mark.parametrize("qtype", [12, 14])
def test_prefill_chain_reusing_one_xq_buffer(qtype):
    N, K, M, L = 18944 if qtype == 12 else 4096, 1024, 256, 4
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 71), N, K)
    xs = [torch.from_numpy(synth.activations(M, K, seed=72 + i)).cuda() for i in range(L)]
    xd = [torch.from_numpy(synth.activations(2, N, seed=80 + i)).cuda() for i in range(L)]
    Wd = mq.register_weight(12, synth.weights(12, 512, N, 73), 512, N, mq.REG_NO_MMQ_PLANE) \
        if N % 256 == 0 else None
    xq = torch.empty(mq.act_bytes(M, K), dtype=torch.uint8, device="cuda")
    # reference: every call followed by a device synchronisation
    ref_y, ref_d = [], []
    for i in range(L):
        mq.quantize_act(xs[i], xq)
        torch.cuda.synchronize()
        ref_y.append(mq.mmq(W, xq, M))
        torch.cuda.synchronize()
        if Wd is not None:
            ref_d.append(mq.matvec(Wd, xd[i]))
            torch.cuda.synchronize()
    ys = [torch.empty((M, N), device="cuda") for _ in range(L)]
    ds = [torch.empty((2, 512), device="cuda") for _ in range(L)]

    def chain():
        for i in range(L):
            mq.quantize_act(xs[i], xq)
            mq.mmq(W, xq, M, ys[i])
            if Wd is not None:
                mq.matvec(Wd, xd[i], ds[i])

    chain()  # eager, back to back
    torch.cuda.synchronize()
    for i in range(L):
        assert np.array_equal(bits(ys[i]), bits(ref_y[i])), i
        if Wd is not None:
            assert np.array_equal(bits(ds[i]), bits(ref_d[i])), i
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            chain()
    for _ in range(3):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i in range(L):
            assert np.array_equal(bits(ys[i]), bits(ref_y[i])), i
    mq.stream_status()
    W.free()
    if Wd is not None:
        Wd.free()
