"""Fused FFN gate/up with SwiGLU ("minfer CUDA Backend Design" §4.3 FusedFFN/SwiGLU,
§4.6 the ffn_gu concat): h = silu(W_gate x) * (W_up x), through the C ABI, against
the oracle's composition of two matvecs / MMQs with silu, and its propagated bound."""
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


def assert_within(h, href, bnd, what):
    h = np.asarray(h, dtype=np.float64)
    # the bound of the composition, plus a few f32 roundings in the kernel's silu and product
    lim = bnd + 2.0 ** -20 * np.abs(href)
    err = np.abs(h - href)
    bad = err > lim + 1e-37
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside the bound; worst "
                           f"err/bound {np.max(err / np.maximum(lim, 1e-300)):.3e}")


def pair(qtype, N, K, s):
    return synth.weights(qtype, N, K, s), synth.weights(qtype, N, K, s + 1)


@pytest.mark.parametrize("qtype,N,K", [
    (synth.Q8_0, 8, 96), (synth.Q8_0, 136, 288), (synth.Q4_K, 8, 256), (synth.Q4_K, 72, 512),
    (synth.Q4_K, 200, 768), (synth.Q6_K, 24, 256), (synth.Q6_K, 136, 512),
    (synth.Q4_1, 72, 288), (synth.Q5_0, 136, 96), (synth.Q5_1, 8, 512),
    (synth.F16, 72, 288), (synth.BF16, 136, 512)])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_ffn_gu_matvec_small_shapes(qtype, N, K, B):
    g, u = pair(qtype, N, K, 500 + N)
    W = mq.register_ffn_gu(qtype, g, u, N, K, mq.REG_NO_MMQ_PLANE)
    x = synth.activations(B, K, 77)
    h = mq.ffn_gu_matvec(W, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    href, bnd = oracle.ffn_gu_matvec(qtype, g, u, N, K, x)
    assert_within(h.cpu().numpy(), href, bnd, f"type {qtype} {N}x{K} B={B}")
    W.free()


@pytest.mark.parametrize("qtype,N,K", [(synth.Q4_K, 18944, 3584), (synth.Q6_K, 3584, 18944)])
@pytest.mark.parametrize("B", [1, 4])
def test_ffn_gu_matvec_ffn_shapes(qtype, N, K, B):
    """FFN-sized gate/up pairs (Qwen2.5-7B: 18944 x 3584), in the bench's launch setup."""
    g, u = pair(qtype, N, K, 610)
    W = mq.register_ffn_gu(qtype, g, u, N, K, mq.REG_NO_MMQ_PLANE)
    x = synth.activations(B, K, 78)
    h = mq.ffn_gu_matvec(W, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    mq.stream_status()
    href, bnd = oracle.ffn_gu_matvec(qtype, g, u, N, K, x)
    assert_within(h.cpu().numpy(), href, bnd, f"type {qtype} {N}x{K} B={B}")
    W.free()


@pytest.mark.parametrize("qtype,N,K,M", [
    (synth.Q8_0, 8, 96, 5), (synth.Q8_0, 136, 320, 130), (synth.Q4_K, 8, 256, 19),
    (synth.Q4_K, 200, 768, 140), (synth.Q6_K, 72, 512, 64), (synth.Q4_1, 136, 288, 70),
    (synth.Q5_0, 8, 96, 5), (synth.Q5_1, 72, 512, 129)])
def test_ffn_gu_mmq_small_shapes(qtype, N, K, M):
    g, u = pair(qtype, N, K, 700 + N)
    W = mq.register_ffn_gu(qtype, g, u, N, K)
    x = synth.activations(M, K, 79)
    xq = mq.quantize_act(torch.from_numpy(x).cuda())
    h = mq.ffn_gu_mmq(W, xq, M)
    torch.cuda.synchronize()
    qs, sc, _ = oracle.quantize_act(x)
    href, bnd = oracle.ffn_gu_mmq(qtype, g, u, N, K, qs, sc)
    assert_within(h.cpu().numpy(), href, bnd, f"type {qtype} {N}x{K} M={M}")
    W.free()


def test_ffn_gu_mmq_ffn_shape_sampled_rows():
    """Q4_K 18944 x 3584 gate/up, M = 512 (the prefill workload), on sampled rows."""
    qtype, N, K, M = synth.Q4_K, 18944, 3584, 512
    g, u = pair(qtype, N, K, 620)
    W = mq.register_ffn_gu(qtype, g, u, N, K)
    x = synth.activations(M, K, 80)
    xq = mq.quantize_act(torch.from_numpy(x).cuda())
    h = mq.ffn_gu_mmq(W, xq, M)
    torch.cuda.synchronize()
    mq.stream_status()
    rows = np.array([0, 1, 127, 128, 255, 300, 511])
    qs, sc, _ = oracle.quantize_act(x)
    href, bnd = oracle.ffn_gu_mmq(qtype, g, u, N, K, qs, sc, mrows=rows)
    assert_within(h.cpu().numpy()[rows], href, bnd, "ffn_gu mmq 512x18944x3584")
    W.free()


@pytest.mark.parametrize("qtype,N,K", [(synth.Q8_0, 24, 96), (synth.Q4_K, 136, 512),
                                       (synth.Q6_K, 8, 256)])
def test_ffn_gu_unpack_returns_gate_then_up(qtype, N, K):
    g, u = pair(qtype, N, K, 800)
    W = mq.register_ffn_gu(qtype, g, u, N, K)
    assert np.array_equal(W.unpack(), np.concatenate([g, u]))
    assert W.info()[1] == 2 * N
    W.free()


def test_plain_and_fused_calls_do_not_mix():
    qtype, N, K = synth.Q4_K, 16, 256
    g, u = pair(qtype, N, K, 900)
    Wf = mq.register_ffn_gu(qtype, g, u, N, K)
    Wp = mq.register_weight(qtype, g, N, K)
    x = torch.from_numpy(synth.activations(1, K, 81)).cuda()
    y = torch.empty((1, 2 * N), device="cuda")
    with pytest.raises(mq.MQError, match="fused gate/up weight; use"):
        mq._check(mq.lib().mq_matvec(qtype, Wf.handle, mq._ptr(x), mq._ptr(y), 2 * N, K, 1,
                                     mq._stream(None)))
    with pytest.raises(mq.MQError, match="not a fused gate/up weight"):
        mq._check(mq.lib().mq_ffn_gu_matvec(qtype, Wp.handle, mq._ptr(x), mq._ptr(y), N, K, 1,
                                            mq._stream(None)))
    xq = mq.quantize_act(x)
    with pytest.raises(mq.MQError, match="fused gate/up weight; use"):
        mq._check(mq.lib().mq_mmq_blockdots(qtype, Wf.handle, mq._ptr(xq), mq._ptr(y), 1, 2 * N,
                                            K, mq._stream(None)))
    Wf.free()
    Wp.free()
