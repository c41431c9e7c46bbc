"""Activation quantisation fused into the MMQ ("minfer CUDA Backend Design" §3 and §8: the
q8_1 GEMM-prologue fusion, the open step change): mq_mmq_fused quantises x in the
persistent MMQ's prologue, crosses a grid-wide barrier and runs the contraction.  Its xq
bytes must equal mq_quantize_act's and its y must equal mq_quantize_act + mq_mmq bit for
bit (the arithmetic is the same, only the kernel boundary moves); the barrier count must be
back to zero after every call (the generation word advances), so the buffer serves
repeated calls and graph replays."""
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


def fused_vs_separate(W, x):
    M, K = x.shape
    xd = torch.from_numpy(x).cuda()
    # both buffers zero-filled, so that the bytes the layout leaves unspecified (padding,
    # rows past M of the transposed planes) compare equal too
    y_f, xq_f = mq.mmq_fused(W, xd, mq.act_buffer(M, K))
    xq_s = mq.quantize_act(xd, mq.act_buffer(M, K))
    y_s = mq.mmq(W, xq_s, M)
    torch.cuda.synchronize()
    mq.stream_status()
    sync = mq.act_layout(M, K)["sync"]
    assert torch.equal(xq_f[:sync], xq_s[:sync]), "xq differs from mq_quantize_act"
    assert int(xq_f[sync:sync + 4].count_nonzero()) == 0, "barrier count not back to zero"
    assert torch.equal(y_f.view(torch.int32), y_s.view(torch.int32)), "y differs from the two calls"
    return y_f, xq_f


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q8_0, 37, 96, 5), (synth.Q4_K, 200, 768, 65), (synth.Q6_K, 130, 512, 129),
    (synth.Q4_1, 136, 288, 70), (synth.Q5_K, 19, 512, 9), (synth.Q4_0, 300, 4864, 300)])
def test_fused_equals_quantise_then_mmq(qtype, N, K, M):
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 61), N, K)
    x = synth.activations(M, K, seed=62)
    y, _ = fused_vs_separate(W, x)
    qs, sc, _ = oracle.quantize_act(x)
    yref, bnd = oracle.mmq(qtype, synth.weights(qtype, N, K, 61), N, K, qs, sc)
    err = np.abs(y.cpu().numpy().astype(np.float64) - yref)
    assert (err <= 1e-4 * bnd + 1e-37).all()
    W.free()


def test_fused_prefill_workload_bitwise():
    """Q4_K 18944 x 3584, M = 512 (the prefill workload): 152 CTAs quantise 3-4 rows each."""
    qtype, N, K, M = synth.Q4_K, 18944, 3584, 512
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 63), N, K)
    fused_vs_separate(W, synth.activations(M, K, seed=64))
    W.free()


def test_barrier_words_serve_repeated_calls_and_graph_replays():
    qtype, N, K, M = synth.Q4_K, 512, 1024, 200
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 65), N, K)
    xd = torch.from_numpy(synth.activations(M, K, seed=66)).cuda()
    xq = mq.act_buffer(M, K)
    y0 = torch.empty((M, N), device="cuda")
    mq.mmq_fused(W, xd, xq, y0)
    ys = [torch.empty((M, N), device="cuda") for _ in range(3)]
    for y in ys:  # the same buffer, back to back
        mq.mmq_fused(W, xd, xq, y)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    yg = torch.empty((M, N), device="cuda")
    with torch.cuda.stream(stream):
        mq.mmq_fused(W, xd, xq, yg, stream=stream)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mq.mmq_fused(W, xd, xq, yg)
    for _ in range(3):
        yg.zero_()
        g.replay()
    torch.cuda.synchronize()
    mq.stream_status()
    for y in ys + [yg]:
        assert torch.equal(y.view(torch.int32), y0.view(torch.int32))
    sync = mq.act_layout(M, K)["sync"]
    assert int(xq[sync:sync + 4].count_nonzero()) == 0
    # the generation word advanced once per executed call: 1 + 3 eager, 1 warm-up on the
    # capture stream, 3 graph replays (capturing runs nothing)
    assert int(xq[sync + 4:sync + 8].view(torch.int32)[0]) == 8
    W.free()


def test_fused_rejects_what_the_mmq_rejects():
    K, M = 256, 4
    x = torch.zeros((M, K), device="cuda")
    Wf = mq.register_weight(synth.F16, synth.weights(synth.F16, 8, K, 67), 8, K)
    with pytest.raises(mq.MQError) as e:
        mq.mmq_fused(Wf, x)
    assert e.value.name == "MQ_ERR_TYPE"
    Wn = mq.register_weight(synth.Q4_K, synth.weights(synth.Q4_K, 8, K, 68), 8, K,
                            mq.REG_NO_MMQ_PLANE)
    with pytest.raises(mq.MQError) as e:
        mq.mmq_fused(Wn, x)
    assert e.value.name == "MQ_ERR_ARG"
    Wf.free()
    Wn.free()
    mq.stream_status()


@pytest.mark.parametrize("qtype,N,K,M", [(synth.Q8_0, 1, 32, 1), (synth.Q4_0, 3, 32, 2),
                                         (synth.Q5_1, 1, 64, 1), (synth.Q4_K, 1, 256, 1),
                                         (synth.Q6_K, 2, 256, 1)])
def test_fused_minimal_shapes(qtype, N, K, M):
    """One output tile that is almost all padding, a single activation row, K one block."""
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 69), N, K)
    x = synth.activations(M, K, seed=70)
    fused_vs_separate(W, x)
    xd = torch.from_numpy(x).cuda()
    ys = mq.mmq_fused_static(W, xd)
    yf, _ = mq.mmq_fused(W, xd)
    torch.cuda.synchronize()
    mq.stream_status()
    assert torch.equal(ys.view(torch.int32), yf.view(torch.int32))
    W.free()
