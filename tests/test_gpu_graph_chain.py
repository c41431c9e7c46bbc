"""Decode chains captured as one CUDA graph ("Architecture Execution Plan": decode
graphs captured after a warm-up and replayed).  The C-ABI calls enqueue work only
(no host synchronisation, no allocation), so a chain of matvecs records into a
graph; its replay must reproduce the eager chain bit for bit, and every link must
stay within the oracle's bound given the previous link's GPU output as its input."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import gguf_block_quantized_q4_gb300 as mq  # noqa: E402
from gguf_block_quantized_q4_gb300 import build as mqbuild  # noqa: E402

REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mqbuild.build()
    mq.init(0)
    yield


def run_chain(Ws, x0, ys):
    h = x0
    for W, y in zip(Ws, ys):
        mq.matvec(W, h, y)
        h = y
    return h


def check_chain(shapes, B, x_seed):
    """shapes: (qtype, N, K, w_seed) per link; K of link l+1 equals N of link l."""
    raws = [synth.weights(qt, N, K, s) for qt, N, K, s in shapes]
    Ws = [mq.register_weight(qt, r, N, K, mq.REG_NO_MMQ_PLANE)
          for (qt, N, K, _), r in zip(shapes, raws)]
    K0 = shapes[0][2]
    x0 = torch.from_numpy(synth.activations(B, K0, x_seed)).cuda()
    eager = [torch.empty((B, N), device="cuda") for _, N, _, _ in shapes]
    graphed = [torch.empty((B, N), device="cuda") for _, N, _, _ in shapes]
    xin = x0.clone()
    run_chain(Ws, x0, eager)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(3):  # warm-up before capture
            run_chain(Ws, xin, graphed)
    torch.cuda.current_stream().wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_chain(Ws, xin, graphed)
    for o in graphed:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    mq.stream_status()
    for l, (e, o) in enumerate(zip(eager, graphed)):
        assert torch.equal(e, o), f"link {l}: graph replay differs from the eager call"
    # each link against the oracle, fed with the GPU's previous output
    h = x0.cpu().numpy()
    for l, ((qt, N, K, _), raw) in enumerate(zip(shapes, raws)):
        yref, bnd = oracle.matvec(qt, raw, N, K, h)
        y = eager[l].cpu().numpy().astype(np.float64)
        err = np.abs(y - yref)
        assert (err <= REL * bnd + 1e-37).all(), (
            f"link {l}: worst err/bound {np.max(err / np.maximum(bnd, 1e-300)):.3e}")
        h = eager[l].cpu().numpy()
    for W in Ws:
        W.free()


def test_q8_0_decode_chain_of_eight_links_replays_bitwise():
    """Eight 896 x 896 Q8_0 links (the launch-bound decode size), B = 1."""
    shapes = [(synth.Q8_0, 896, 896, 300 + l) for l in range(8)]
    check_chain(shapes, 1, 7)


@pytest.mark.parametrize("B", [1, 3])
def test_ffn_shaped_chain_replays_bitwise(B):
    """Q4_K 18944 x 3584 up-projection then Q6_K 3584 x 18944 down-projection, twice."""
    shapes = [(synth.Q4_K, 18944, 3584, 102), (synth.Q6_K, 3584, 18944, 103),
              (synth.Q4_K, 18944, 3584, 104), (synth.Q6_K, 3584, 18944, 105)]
    check_chain(shapes, B, 11)
