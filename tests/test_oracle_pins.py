"""Pins for the CPU oracle, against facts that do not come from the oracle itself:
hand-worked golden blocks (tests/golden/), IEEE binary16 as numpy decodes it,
invariants of the block formats and of the activation quantiser, special cases
that reduce to a plain float64 matrix product, Python big-integer brute force, and
a second, vectorised decoder.  CPU only."""
import math
import os

import numpy as np
import pytest

import oracle
import synth
from tests import gguf_pack as gp

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    kv, flips = {}, []
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split(":", 1)
        if k == "flip":
            flips.append(v.split())
        else:
            kv[k] = v.strip()
    return kv, flips


def _ints(s):
    return [int(t) for t in s.split()]


# ---- IEEE binary16 ---------------------------------------------------------

def test_f16_all_bit_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_f16_golden_values():
    for line in open(os.path.join(GOLD, "f16_values.txt")):
        if line.startswith("#") or not line.strip():
            continue
        b, v = line.split()
        got = oracle.f16_to_double(int(b, 16))
        assert got == float(v) and np.signbit(got) == np.signbit(float(v)), (b, v, got)


def test_bf16_all_bit_patterns_match_binary32():
    """bfloat16 is the upper half of a binary32: numpy's f32 decoding of bits << 16."""
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_golden_values():
    for line in open(os.path.join(GOLD, "bf16_values.txt")):
        if line.startswith("#") or not line.strip():
            continue
        b, v = line.split()
        got = oracle.bf16_to_double(int(b, 16))
        assert got == float(v) and np.signbit(got) == np.signbit(float(v)), (b, v, got)


def test_float_weight_rows_worked_by_hand():
    """f16 row (1, 2, -0.5, 65504) and bf16 row (1, -123.5, 0.25, 10) against x = (1, 1, 2, 1/4):
    1 + 2 - 1 + 16376 = 16378 and 1 - 123.5 + 0.5 + 2.5 = -119.5."""
    x = np.array([[1.0, 1.0, 2.0, 0.25]], np.float32)
    wf = np.array([0x3C00, 0x4000, 0xB800, 0x7BFF], "<u2").view(np.uint8)
    y, bnd = oracle.matvec(1, wf, 1, 4, x)
    assert y[0, 0] == 16378.0 and bnd[0, 0] == 1 + 2 + 1 + 16376.0
    wb = np.array([0x3F80, 0xC2F7, 0x3E80, 0x4120], "<u2").view(np.uint8)
    y, bnd = oracle.matvec(30, wb, 1, 4, x)
    assert y[0, 0] == -119.5 and bnd[0, 0] == 1 + 123.5 + 0.5 + 2.5
    # no integer form: the block-dot reference refuses float weights
    with pytest.raises(ValueError):
        oracle.blockdots(1, np.zeros(64, np.uint8), 1, 32, np.zeros((1, 32), np.int8))


# ---- hand-worked blocks ----------------------------------------------------

def test_q8_0_ramp_block():
    kv, _ = _read("q8_0_ramp.txt")
    blk = np.frombuffer(bytes.fromhex(kv["hex"]), dtype=np.uint8)
    w = oracle.dequant_row(8, blk, 32)
    assert w.tolist() == [float(v) for v in _ints(kv["w"])]
    y, _ = oracle.matvec(8, blk, 1, 32, np.ones(32, np.float32))
    assert y[0, 0] == int(kv["dot_ones"])


def test_q8_0_negative_subnormal_scale():
    kv, _ = _read("q8_0_neg_subnormal.txt")
    blk = np.frombuffer(bytes.fromhex(kv["hex"]), dtype=np.uint8)
    w = oracle.dequant_row(8, blk, 32)
    assert (w * 2.0 ** 24).tolist() == [float(v) for v in _ints(kv["w_times_2p24"])]
    y, _ = oracle.matvec(8, blk, 1, 32, np.ones(32, np.float32))
    assert y[0, 0] * 2.0 ** 24 == int(kv["dot_ones_times_2p24"])


def test_q4_0_ramp_block():
    kv, _ = _read("q4_0_ramp.txt")
    blk = np.frombuffer(bytes.fromhex(kv["hex"]), dtype=np.uint8)
    assert oracle.dequant_row(2, blk, 32).tolist() == [float(v) for v in _ints(kv["w"])]
    y, _ = oracle.matvec(2, blk, 1, 32, np.ones(32, np.float32))
    assert y[0, 0] == int(kv["dot_ones"])


@pytest.mark.parametrize("fname", ["q4_1_as_q4_0.txt", "q5_0_ramp.txt", "q5_1_halves.txt"])
def test_q32_min_and_fifth_bit_blocks(fname):
    kv, _ = _read(fname)
    qtype = int(kv["type"])
    blk = np.frombuffer(bytes.fromhex(kv["hex"]), dtype=np.uint8)
    assert oracle.dequant_row(qtype, blk, 32).tolist() == [float(v) for v in kv["w"].split()]
    y, _ = oracle.matvec(qtype, blk, 1, 32, np.ones(32, np.float32))
    assert y[0, 0] == float(kv["dot_ones"])


def test_q5_k_high_bits_block():
    kv, _ = _read("q5_k_high_bits.txt")
    blk = np.frombuffer(bytes.fromhex(kv["hex"]), dtype=np.uint8)
    expect = []
    for run in kv["w_runs"].split():
        v, n = run.split("x")
        expect += [float(v)] * int(n)
    assert oracle.dequant_row(13, blk, 256).tolist() == expect
    y, _ = oracle.matvec(13, blk, 1, 256, np.ones(256, np.float32))
    assert y[0, 0] == int(kv["dot_ones"])


def test_q4_k_ones_twos_block():
    kv, _ = _read("q4_k_ones_twos.txt")
    blk = np.frombuffer(bytes.fromhex(kv["hex"]), dtype=np.uint8)
    expect = []
    for run in kv["w_runs"].split():
        v, n = run.split("x")
        expect += [float(v)] * int(n)
    assert oracle.dequant_row(12, blk, 256).tolist() == expect
    y, _ = oracle.matvec(12, blk, 1, 256, np.ones(256, np.float32))
    assert y[0, 0] == int(kv["dot_ones"])


def test_q4_k_scale_packing_all_fields():
    kv, _ = _read("q4_k_scales_distinct.txt")
    raw = bytes.fromhex(kv["hex"])
    sc, mn = _ints(kv["sc"]), _ints(kv["mn"])
    for j in range(8):
        assert oracle.q4_k_scale_min(raw[4:16], j) == (sc[j], mn[j])
    blk = np.frombuffer(raw, dtype=np.uint8)
    w = oracle.dequant_row(12, blk, 256)
    per = [float(v) for v in kv["w_per_subblock"].split()]
    for j in range(8):
        assert w[32 * j:32 * j + 32].tolist() == [per[j]] * 32
    y, _ = oracle.matvec(12, blk, 1, 256, np.ones(256, np.float32))
    assert y[0, 0] == int(kv["dot_ones"])


def test_q4_k_nibble_order():
    kv, _ = _read("q4_k_nibble_order.txt")
    raw = (bytes([0x00, 0x3C, 0x00, 0x00]) + bytes.fromhex(kv["scale_bytes"]) +
           bytes(range(128)))
    w = oracle.dequant_row(12, np.frombuffer(raw, dtype=np.uint8), 256)
    for c in range(4):
        for l in range(32):
            assert w[64 * c + l] == (l & 15)
            assert w[64 * c + 32 + l] == 2 * c + (l >> 4)
    assert w.sum() == int(kv["dot_ones"])


def test_q6_k_constant_blocks():
    kv, _ = _read("q6_k_constant.txt")
    d = bytes([0x00, 0x3C])
    ones = bytes([1] * 16)
    a = bytes(128) + bytes(64) + ones + d
    b = bytes(128) + bytes([0xAA] * 64) + ones + d
    c = bytes([0x11] * 128) + bytes([0xAA] * 64) + bytes(range(1, 17)) + d
    x1 = np.ones(256, np.float32)
    for raw, key in ((a, "caseA_dot_ones"), (b, "caseB_dot_ones"), (c, "caseC_dot_ones")):
        y, _ = oracle.matvec(14, np.frombuffer(raw, dtype=np.uint8), 1, 256, x1)
        assert y[0, 0] == int(kv[key])
    wc = oracle.dequant_row(14, np.frombuffer(c, dtype=np.uint8), 256)
    assert wc.tolist() == [float(e // 16 + 1) for e in range(256)]
    assert np.all(oracle.dequant_row(14, np.frombuffer(a, dtype=np.uint8), 256) == -32.0)


def test_q6_k_single_bit_flips():
    _, flips = _read("q6_k_bitflips.txt")
    assert flips
    base = bytearray(bytes(128) + bytes([0xAA] * 64) + bytes([1] * 16) + bytes([0x00, 0x3C]))
    for plane, byte, bit, _arrow, elem, delta in flips:
        raw = bytearray(base)
        off = (0 if plane == "ql" else 128) + int(byte)
        raw[off] ^= 1 << int(bit)
        w = oracle.dequant_row(14, np.frombuffer(bytes(raw), dtype=np.uint8), 256)
        expect = np.zeros(256)
        expect[int(elem)] = float(delta)
        assert np.array_equal(w, expect), (plane, byte, bit)


# ---- format invariants -----------------------------------------------------

def test_q4_k_scale_pack_unpack_roundtrip():
    rng = np.random.default_rng(7)
    cases = [([0] * 8, [0] * 8), ([63] * 8, [63] * 8), (list(range(8)), list(range(56, 64)))]
    cases += [(list(rng.integers(0, 64, 8)), list(rng.integers(0, 64, 8))) for _ in range(200)]
    for sc, mn in cases:
        s12 = gp.pack_q4_k_scales(sc, mn)
        assert [oracle.q4_k_scale_min(s12, j) for j in range(8)] == list(zip(sc, mn))
    # every byte with its top bits set decodes to fields in range
    for j in range(8):
        s, m = oracle.q4_k_scale_min(bytes([0xFF] * 12), j)
        assert s == 63 and m == 63


def test_q4_k_zero_quants_give_minus_min():
    rng = np.random.default_rng(1)
    sc = rng.integers(0, 64, 8)
    mn = rng.integers(0, 64, 8)
    raw = gp.pack_q4_k(gp.f16_bits(0.75), gp.f16_bits(0.125), sc, mn, np.zeros(256, int))
    w = oracle.dequant_row(12, np.frombuffer(raw, dtype=np.uint8), 256)
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == -0.125 * mn[j])


def test_zero_scales_give_zero_weights():
    rng = np.random.default_rng(2)
    r4 = gp.pack_q4_k(gp.f16_bits(1.0), gp.f16_bits(1.0), [0] * 8, [0] * 8,
                      rng.integers(0, 16, 256))
    r6 = gp.pack_q6_k(gp.f16_bits(1.0), [0] * 16, rng.integers(0, 64, 256))
    r8 = gp.pack_q8_0(0, rng.integers(-128, 128, 32))
    for t, raw, K in ((12, r4, 256), (14, r6, 256), (8, r8, 32)):
        assert np.all(oracle.dequant_row(t, np.frombuffer(raw, dtype=np.uint8), K) == 0.0)


def test_linearity_in_d_and_dmin():
    rng = np.random.default_rng(3)
    nib, sc, mn = rng.integers(0, 16, 256), rng.integers(0, 64, 8), rng.integers(0, 64, 8)
    w1 = oracle.dequant_row(12, np.frombuffer(
        gp.pack_q4_k(gp.f16_bits(0.5), gp.f16_bits(0.25), sc, mn, nib), np.uint8), 256)
    w2 = oracle.dequant_row(12, np.frombuffer(
        gp.pack_q4_k(gp.f16_bits(1.0), gp.f16_bits(0.5), sc, mn, nib), np.uint8), 256)
    assert np.array_equal(2 * w1, w2)
    q6, s6 = rng.integers(0, 64, 256), rng.integers(-128, 128, 16)
    a = oracle.dequant_row(14, np.frombuffer(gp.pack_q6_k(gp.f16_bits(0.25), s6, q6), np.uint8),
                           256)
    b = oracle.dequant_row(14, np.frombuffer(gp.pack_q6_k(gp.f16_bits(-1.0), s6, q6), np.uint8),
                           256)
    assert np.array_equal(-4 * a, b)


# ---- special cases that reduce to a plain float64 product --------------------

@pytest.mark.parametrize("qtype", [2, 3, 6, 7, 8, 12, 13, 14])
def test_unit_scales_reduce_to_integer_matrix_product(qtype):
    rng = np.random.default_rng(4 + qtype)
    N, K, B = 5, 512, 3
    rows, ints = [], np.zeros((N, K), dtype=np.int64)
    one = gp.f16_bits(1.0)
    for n in range(N):
        row = b""
        for blk in range(K // (32 if qtype in (2, 3, 6, 7, 8) else 256)):
            if qtype == 8:
                q = rng.integers(-128, 128, 32)
                row += gp.pack_q8_0(one, q)
                ints[n, 32 * blk:32 * blk + 32] = q
            elif qtype == 2:
                q = rng.integers(-8, 8, 32)
                row += gp.pack_q4_0(one, q)
                ints[n, 32 * blk:32 * blk + 32] = q
            elif qtype in (3, 6, 7):
                q = rng.integers(0, 16 if qtype == 3 else 32, 32)
                row += gp.pack_q32(qtype, one, 0, q)
                ints[n, 32 * blk:32 * blk + 32] = q - (16 if qtype == 6 else 0)
            elif qtype == 13:
                q = rng.integers(0, 32, 256)
                row += gp.pack_q5_k(one, 0, [1] * 8, [0] * 8, q)
                ints[n, 256 * blk:256 * blk + 256] = q
            elif qtype == 12:
                q = rng.integers(0, 16, 256)
                row += gp.pack_q4_k(one, 0, [1] * 8, [0] * 8, q)
                ints[n, 256 * blk:256 * blk + 256] = q
            else:
                q = rng.integers(0, 64, 256)
                row += gp.pack_q6_k(one, [1] * 16, q)
                ints[n, 256 * blk:256 * blk + 256] = q - 32
        rows.append(row)
    W = np.frombuffer(b"".join(rows), dtype=np.uint8)
    x = rng.standard_normal((B, K)).astype(np.float32)
    y, bnd = oracle.matvec(qtype, W, N, K, x)
    ref = x.astype(np.float64) @ ints.T.astype(np.float64)
    assert np.allclose(y, ref.reshape(B, N), rtol=1e-13, atol=1e-12)
    assert np.allclose(bnd, np.abs(x.astype(np.float64)) @ np.abs(ints.T), rtol=1e-13)


# ---- second formulation (vectorised numpy) and brute force ----------------

@pytest.mark.parametrize("qtype", [1, 30, 2, 3, 6, 7, 8, 12, 13, 14])
def test_dequant_matches_vectorised_numpy_decoder(qtype):
    N, K = 7, 512
    W = synth.weights(qtype, N, K, seed=11)
    assert np.array_equal(oracle.dequant(qtype, W, N, K), gp.np_dequant(qtype, W, N, K))


@pytest.mark.parametrize("qtype", [1, 30, 2, 3, 6, 7, 8, 12, 13, 14])
def test_matvec_bound_is_sum_of_absolute_products(qtype):
    """The per-row bound is sum_k |w||x| with w from the independent numpy decoder."""
    N, K, B = 3, 512, 2
    W = synth.weights(qtype, N, K, seed=31)
    x = synth.activations(B, K, seed=32)
    _, bnd = oracle.matvec(qtype, W, N, K, x)
    w = gp.np_dequant(qtype, W, N, K)
    ref = np.abs(x.astype(np.float64)) @ np.abs(w).T
    assert np.allclose(bnd, ref, rtol=1e-12, atol=0.0)


@pytest.mark.parametrize("qtype", [1, 30, 2, 3, 6, 7, 8, 12, 13, 14])
@pytest.mark.parametrize("N,K,B", [(1, 256, 1), (2, 256, 8), (3, 512, 4), (3, 512, 2)])
def test_brute_force_tiny_matvec(qtype, N, K, B):
    W = synth.weights(qtype, N, K, seed=N * 100 + K + B)
    x = synth.activations(B, K, seed=B)
    y, bnd = oracle.matvec(qtype, W, N, K, x)
    w = gp.np_dequant(qtype, W, N, K)
    for b in range(B):
        for n in range(N):
            exact = sum(float(w[n, k]) * float(x[b, k]) for k in range(K))
            assert abs(y[b, n] - exact) <= 1e-12 * bnd[b, n] + 1e-300


@pytest.mark.parametrize("qtype", [2, 3, 6, 7, 8, 12, 13, 14])
def test_blockdots_python_big_integers(qtype):
    N, K, M = 3, 512, 4
    W = synth.weights(qtype, N, K, seed=21)
    x = synth.activations(M, K, seed=22)
    qs, sc, bs = oracle.quantize_act(x)
    D = oracle.blockdots(qtype, W, N, K, qs)
    wf = gp.np_dequant(qtype, W, N, K)
    rowbytes = len(W) // N
    for n in range(N):
        wi = oracle.int_weights_row(qtype, W[n * rowbytes:(n + 1) * rowbytes], K)
        # the integer weight times the block scale (minus the q4_K min term) is the weight
        be = 32 if qtype in (2, 3, 6, 7, 8) else 256
        blk = W[n * rowbytes:(n + 1) * rowbytes].reshape(-1, rowbytes // (K // be))
        for k in range(K):
            b = blk[k // be]
            if qtype == 14:
                d = np.frombuffer(bytes(b[208:210]), np.float16)[0].astype(np.float64)
                assert wf[n, k] == d * wi[k]
            elif qtype in (2, 6, 8):
                d = np.frombuffer(bytes(b[0:2]), np.float16)[0].astype(np.float64)
                assert wf[n, k] == d * wi[k]
            elif qtype in (3, 7):
                d, m = np.frombuffer(bytes(b[0:4]), np.float16).astype(np.float64)
                assert wf[n, k] == d * wi[k] + m
        for m in range(M):
            for blk_i in range(K // 32):
                ref = sum(int(wi[k]) * int(qs[m, k]) for k in range(32 * blk_i, 32 * blk_i + 32))
                assert D[m, n, blk_i] == ref
    assert np.abs(D).max() < 2 ** 24  # exact in f32 partial sums


@pytest.mark.parametrize("qtype", [2, 3, 6, 7, 8, 12, 13, 14])
def test_mmq_reference_equals_block_structured_sum(qtype):
    """The plain definition sum_k w * (s q) equals the block-structured form
    sum_b s_b * (d * D_b - dmin * m_j * S_b) built from the block dots."""
    N, K, M = 3, 512, 3
    W = synth.weights(qtype, N, K, seed=31)
    x = synth.activations(M, K, seed=32)
    qs, sc, bs = oracle.quantize_act(x)
    y, bnd = oracle.mmq(qtype, W, N, K, qs, sc)
    D = oracle.blockdots(qtype, W, N, K, qs)
    be = 32 if qtype in (2, 3, 6, 7, 8) else 256
    rowbytes = len(W) // N
    for n in range(N):
        blocks = W[n * rowbytes:(n + 1) * rowbytes].reshape(K // be, -1)
        for m in range(M):
            acc = 0.0
            for b in range(K // 32):
                blk = blocks[b * 32 // be]
                if qtype in (2, 6, 8):
                    d = float(np.frombuffer(bytes(blk[0:2]), np.float16)[0])
                    acc += float(sc[m, b]) * d * float(D[m, n, b])
                elif qtype in (3, 7):
                    d, mm = (float(v) for v in np.frombuffer(bytes(blk[0:4]), np.float16))
                    acc += float(sc[m, b]) * (d * float(D[m, n, b]) + mm * float(bs[m, b]))
                elif qtype in (12, 13):
                    d = float(np.frombuffer(bytes(blk[0:2]), np.float16)[0])
                    dmin = float(np.frombuffer(bytes(blk[2:4]), np.float16)[0])
                    _, mj = oracle.q4_k_scale_min(bytes(blk[4:16]), b % 8)
                    acc += float(sc[m, b]) * (d * float(D[m, n, b]) - dmin * mj * float(bs[m, b]))
                else:
                    d = float(np.frombuffer(bytes(blk[208:210]), np.float16)[0])
                    acc += float(sc[m, b]) * d * float(D[m, n, b])
            assert abs(acc - y[m, n]) <= 1e-12 * bnd[m, n]


# ---- activation quantiser --------------------------------------------------

def test_activation_quantiser_ties_golden():
    kv, _ = _read("act_quant_ties.txt")
    s = float(kv["scale"])
    x = (np.array([float(v) for v in kv["x_over_scale"].split()]) * s).astype(np.float32)
    qs, sc, bs = oracle.quantize_act(x.reshape(1, 32))
    assert sc[0, 0] == np.float32(s)
    assert qs[0].tolist() == _ints(kv["q"])
    assert bs[0, 0] == int(kv["bsum"])


def test_activation_quantiser_zero_block_and_invariants():
    x = synth.activations(6, 256, seed=5) * np.float32(3.0)
    x[2, 32:64] = 0.0
    x[3, :32] = np.float32(1e-30)
    qs, sc, bs = oracle.quantize_act(x)
    assert sc[2, 1] == 0 and np.all(qs[2, 32:64] == 0) and bs[2, 1] == 0
    assert np.array_equal(bs, qs.reshape(6, 8, 32).astype(np.int64).sum(-1))
    nz = sc > 0
    assert np.all(np.abs(qs.reshape(6, 8, 32)).max(-1)[nz] == 127)
    assert np.abs(qs).max() <= 127
    # |x - s q| <= s/2 (plus f32 rounding of s)
    err = np.abs(x.reshape(6, 8, 32) - sc[..., None].astype(np.float64) * qs.reshape(6, 8, 32))
    assert np.all(err <= sc[..., None] * (0.5 + 1e-6))


def test_requantising_a_dequantised_q8_0_block_is_the_identity():
    """A q8_0 block with max |q| = 127 dequantises to x = d*q exactly in f32, and the
    activation quantiser maps it back to scale d and the same q."""
    rng = np.random.default_rng(9)
    for trial in range(200):
        q = rng.integers(-127, 128, 32)
        q[rng.integers(0, 32)] = 127 if trial % 2 else -127
        d = np.float16(abs(rng.standard_normal()) * 0.05 + 1e-3)
        raw = gp.pack_q8_0(int(np.array([d]).view(np.uint16)[0]), q)
        x = oracle.dequant_row(8, np.frombuffer(raw, np.uint8), 32).astype(np.float32)
        qs, sc, bs = oracle.quantize_act(x.reshape(1, 32))
        assert sc[0, 0] == np.float32(d)
        assert qs[0].tolist() == q.tolist()
        assert bs[0, 0] == q.sum()


def test_power_of_two_scaled_blocks_roundtrip():
    rng = np.random.default_rng(10)
    for e in range(-20, 21, 5):
        q = rng.integers(-127, 128, (4, 32))
        q[:, 0] = 127
        x = (q * 2.0 ** e).astype(np.float32)
        qs, sc, bs = oracle.quantize_act(x.reshape(1, 128))
        assert np.all(sc == np.float32(2.0 ** e))
        assert np.array_equal(qs.reshape(4, 32), q)


# ---- fused FFN gate/up (SwiGLU) ----------------------------------------------------

def test_silu_closed_forms():
    """silu(v) = v * sigma(v): silu(0) = 0, silu(1) = e/(1+e), silu(-1) = -1/(1+e), and
    silu(v) - silu(-v) = v (sigma(v) + sigma(-v) = 1); far tails -> v and -0."""
    e = math.e
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - e / (1 + e)) < 1e-15
    assert abs(oracle.silu(-1.0) + 1 / (1 + e)) < 1e-15
    v = np.linspace(-30, 30, 601)
    assert np.allclose(oracle.silu(v) - oracle.silu(-v), v, rtol=0, atol=1e-12)
    assert oracle.silu(800.0) == 800.0
    big_neg = oracle.silu(-800.0)
    assert big_neg == 0.0 and math.copysign(1, big_neg) < 0


def test_silu_matches_tanh_form_and_slope_bound():
    """Independent formulas for sigma, and the slope bound used by
    swiglu_bound: max |silu'| on a fine grid stays below SILU_SLOPE."""
    v = np.linspace(-40, 40, 160001)
    # tanh form for v >= 0; e^v / (1 + e^v) below 0, where 1 + tanh(v/2) cancels
    ref = np.where(v >= 0, v * (1 + np.tanh(v / 2)) / 2, v * np.exp(v) / (1 + np.exp(v)))
    assert np.allclose(oracle.silu(v), ref, rtol=1e-13, atol=1e-300)
    slope = np.abs(np.diff(oracle.silu(v)) / np.diff(v))
    assert slope.max() < oracle.SILU_SLOPE
    assert slope.max() > 1.09  # the bound is tight, not arbitrary


def test_swiglu_bound_covers_perturbations():
    """Random g, u and perturbations inside their bounds never leave swiglu_bound."""
    rng = np.random.Generator(np.random.PCG64(5))
    g = rng.standard_normal(20000) * 4
    u = rng.standard_normal(20000) * 4
    bg = np.abs(rng.standard_normal(20000)) * 50
    bu = np.abs(rng.standard_normal(20000)) * 50
    rel = 1e-4
    dg = (rng.random(20000) * 2 - 1) * rel * bg
    du = (rng.random(20000) * 2 - 1) * rel * bu
    err = np.abs(oracle.silu(g + dg) * (u + du) - oracle.silu(g) * u)
    assert (err <= oracle.swiglu_bound(g, u, bg, bu, rel) * (1 + 1e-12)).all()


@pytest.mark.parametrize("qtype", [synth.Q8_0, synth.Q4_K, synth.Q6_K])
def test_ffn_gu_matvec_is_silu_gate_times_up(qtype):
    """The fused oracle against an explicit float64 dequantise + matmul + tanh-form silu."""
    N, K, B = 5, 512, 3
    Wg = synth.weights(qtype, N, K, 41)
    Wu = synth.weights(qtype, N, K, 42)
    x = synth.activations(B, K, 43)
    h, bnd = oracle.ffn_gu_matvec(qtype, Wg, Wu, N, K, x)
    g = x.astype(np.float64) @ oracle.dequant(qtype, Wg, N, K).T
    u = x.astype(np.float64) @ oracle.dequant(qtype, Wu, N, K).T
    ref = g * (1 + np.tanh(g / 2)) / 2 * u
    assert np.allclose(h, ref, rtol=1e-12, atol=1e-12)
    assert (bnd > 0).all()


@pytest.mark.parametrize("qtype", [synth.Q8_0, synth.Q4_K, synth.Q6_K, synth.Q5_1])
def test_all_cores_build_returns_the_plain_builds_bits(qtype):
    """The OpenMP build of oracle.c (rows on all cores; the full-output GPU parity checks
    and the all-cores CPU baseline use it) returns exactly the plain build's bits: each
    row's arithmetic and summation order are the same in both."""
    if oracle.lib_omp() is None:
        pytest.skip("no OpenMP in this host's compiler")
    N, K = 301, 1024
    W = synth.weights(qtype, N, K, 61)
    x = synth.activations(3, K, 62)
    for a, b in zip(oracle.matvec(qtype, W, N, K, x), oracle.matvec(qtype, W, N, K, x,
                                                                    parallel=True)):
        assert np.array_equal(a.view(np.uint64), b.view(np.uint64))
    qs, sc, _ = oracle.quantize_act(synth.activations(5, K, 63))
    rows = [4, 0, 2]
    for a, b in zip(oracle.mmq(qtype, W, N, K, qs, sc, mrows=rows, n0=7, n1=290),
                    oracle.mmq(qtype, W, N, K, qs, sc, mrows=rows, n0=7, n1=290, parallel=True)):
        assert np.array_equal(a.view(np.uint64), b.view(np.uint64))
    assert np.array_equal(oracle.blockdots(qtype, W, N, K, qs, mrows=rows),
                          oracle.blockdots(qtype, W, N, K, qs, mrows=rows, parallel=True))
