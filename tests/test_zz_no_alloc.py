"""mq_mmq_fused_static: the fused quantise + MMQ with the library's static device scratch in
place of a caller buffer.  Two consecutive calls of different shapes and weight types must
each equal the buffer-based mq_mmq_fused bit for bit (the second call finds the barrier in
its entry state although the first left quantised data of another shape in the scratch),
the device's free memory must not change across them, the first call on the device
included (mq_init looked the scratch up; nothing is allocated), and a shape
whose scratch would not fit is refused before any device work."""
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
