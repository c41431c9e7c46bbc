"""mq_mmq_fused_static: the fused quantise + MMQ with the library's static device scratch in
place of a caller buffer.  Two consecutive calls of different shapes and weight types must
each equal the buffer-based mq_mmq_fused bit for bit (the second call finds the barrier in
its entry state although the first left quantised data of another shape in the scratch),
the device's free memory must not change across them, the first call on the device
included (mq_init looked the scratch up; nothing is allocated), and a shape
whose scratch would not fit is refused before any device work.  A call whose bounded wait
expired leaves the scratch in its entry state for the next call."""
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


def test_two_consecutive_calls_equal_the_buffered_entry_point():
    cases = [(synth.Q4_K, 2000, 3584, 300), (synth.Q6_K, 1000, 2048, 77)]
    Ws, xs, ys, refs = [], [], [], []
    for qtype, N, K, M in cases:
        W = mq.register_weight(qtype, synth.weights(qtype, N, K, 71 + N), N, K)
        x = torch.from_numpy(synth.activations(M, K, seed=72 + M)).cuda()
        ref, _ = mq.mmq_fused(W, x)
        Ws.append(W)
        xs.append(x)
        ys.append(torch.empty((M, N), device="cuda"))
        refs.append(ref)
    # mq_init has looked the scratch up (which loads the module holding it), so even the
    # first call on the device allocates nothing
    torch.cuda.synchronize()
    mq.stream_status()
    free_before = torch.cuda.mem_get_info()[0]
    for W, x, y in zip(Ws, xs, ys):
        mq.mmq_fused_static(W, x, y)
    torch.cuda.synchronize()
    mq.stream_status()
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed"
    for y, ref in zip(ys, refs):
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    for W in Ws:
        W.free()


def test_a_shape_beyond_the_scratch_is_refused():
    qtype, N, K = synth.Q4_K, 256, 3584
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 73), N, K)
    M = 2048  # about 26 MB of xq, more than the 16 MB scratch
    assert mq.act_bytes(M, K) > mq.STATIC_XQ_BYTES - 256
    x = torch.zeros((M, K), device="cuda")
    y = torch.empty((M, N), device="cuda")
    with pytest.raises(mq.MQError) as e:
        mq.mmq_fused_static(W, x, y)
    assert e.value.name == "MQ_ERR_SHAPE" and "static scratch" in str(e.value)
    mq.stream_status()
    W.free()


def test_a_call_after_an_expired_wait_finds_the_scratch_in_its_entry_state(monkeypatch):
    """With the failure-injection seam the fused kernel's epilogue waits, after the grid
    barrier, on a barrier nothing arrives on: the wait expires, the status word reports
    MQ_ERR_TIMEOUT and the result is still correct.  The next static call (the seam off,
    another shape and weight type) finds the scratch's barrier words in their entry state
    and equals mq_mmq_fused bit for bit."""
    qtype, N, K, M = synth.Q4_K, 600, 1024, 130
    W = mq.register_weight(qtype, synth.weights(qtype, N, K, 74), N, K)
    x = torch.from_numpy(synth.activations(M, K, seed=75)).cuda()
    ref, _ = mq.mmq_fused(W, x)
    torch.cuda.synchronize()
    mq.stream_status()
    monkeypatch.setenv("MQ_TEST_EXPIRE_WAIT", "1")
    mq.init(0)  # the seams are read by mq_init
    y = mq.mmq_fused_static(W, x)
    torch.cuda.synchronize()
    with pytest.raises(mq.MQError) as e:
        mq.stream_status()
    assert e.value.name == "MQ_ERR_TIMEOUT"
    monkeypatch.delenv("MQ_TEST_EXPIRE_WAIT")
    mq.init(0)
    mq.stream_status()  # cleared
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    q2, N2, K2, M2 = synth.Q6_K, 300, 512, 40
    W2 = mq.register_weight(q2, synth.weights(q2, N2, K2, 76), N2, K2)
    x2 = torch.from_numpy(synth.activations(M2, K2, seed=77)).cuda()
    ref2, _ = mq.mmq_fused(W2, x2)
    y2 = mq.mmq_fused_static(W2, x2)
    torch.cuda.synchronize()
    mq.stream_status()
    assert torch.equal(y2.view(torch.int32), ref2.view(torch.int32))
    W.free()
    W2.free()
