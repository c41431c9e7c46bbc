"""Test-side block encoders: build GGUF block bytes from chosen integer fields.

These are the inverse of the block layouts (GGUF q4_0 / q8_0 / q4_K / q5_K / q6_K), written
independently of the oracle so that the oracle's decoders can be checked
against blocks whose field values the tests choose.  Also a vectorised numpy
decoder: a second, loop-free formulation used to cross-check the oracle.
"""
import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def pack_q8_0(d_bits: int, q) -> bytes:
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= -128 and q.max() <= 127
    return bytes([d_bits & 255, d_bits >> 8]) + q.astype(np.int8).tobytes()


def pack_q4_k_scales(sc, mn) -> bytes:
    """12 bytes holding eight 6-bit scales and eight 6-bit mins.
    bytes 0-3 : low 6 bits = scale j,   top 2 bits = bits 4-5 of scale j+4
    bytes 4-7 : low 6 bits = min j,     top 2 bits = bits 4-5 of min j+4
    bytes 8-11: low nibble = low 4 bits of scale j+4, high nibble = low 4 bits of min j+4"""
    sc = [int(v) for v in sc]
    mn = [int(v) for v in mn]
    assert len(sc) == 8 and len(mn) == 8 and all(0 <= v < 64 for v in sc + mn)
    out = [0] * 12
    for j in range(4):
        out[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        out[j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)
        out[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    return bytes(out)


def pack_q4_k(d_bits: int, dmin_bits: int, sc, mn, nib) -> bytes:
    """nib[e] for e in 0..255; element 64c + l lives in the low nibble and 64c + 32 + l in
    the high nibble of qs byte 32c + l."""
    nib = np.asarray(nib, dtype=np.int64)
    assert nib.shape == (256,) and nib.min() >= 0 and nib.max() <= 15
    qs = bytearray(128)
    for c in range(4):
        for l in range(32):
            qs[32 * c + l] = int(nib[64 * c + l]) | (int(nib[64 * c + 32 + l]) << 4)
    return (bytes([d_bits & 255, d_bits >> 8, dmin_bits & 255, dmin_bits >> 8]) +
            pack_q4_k_scales(sc, mn) + bytes(qs))


def pack_q6_k(d_bits: int, scales, q) -> bytes:
    """q[e] in 0..63 for e in 0..255 (value q - 32); scales: 16 int8 sub-scales.
    Element e = 128h + 32r + l: low 4 bits in ql[64h + 32(r%2) + l] (low nibble for r<2,
    high nibble for r>=2), top 2 bits at bit 2r of qh[32h + l]."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() <= 63
    ql = bytearray(128)
    qh = bytearray(64)
    for h in range(2):
        for r in range(4):
            for l in range(32):
                v = int(q[128 * h + 32 * r + l])
                p = 64 * h + 32 * (r % 2) + l
                ql[p] |= (v & 15) << (4 if r >= 2 else 0)
                qh[32 * h + l] |= (v >> 4) << (2 * r)
    sc = np.asarray(scales, dtype=np.int64)
    assert sc.shape == (16,) and sc.min() >= -128 and sc.max() <= 127
    return bytes(ql) + bytes(qh) + sc.astype(np.int8).tobytes() + bytes([d_bits & 255,
                                                                        d_bits >> 8])


def pack_q4_0(d_bits: int, q) -> bytes:
    """q[e] in -8..7 for e in 0..31; element j < 16 is the low nibble of quant byte j,
    element 16 + j its high nibble (stored value q + 8)."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= -8 and q.max() <= 7
    qs = bytes(int(q[j] + 8) | (int(q[16 + j] + 8) << 4) for j in range(16))
    return bytes([d_bits & 255, d_bits >> 8]) + qs


def pack_q32(qtype: int, d_bits: int, m_bits: int, q) -> bytes:
    """Q4_1 (q in 0..15), Q5_0 / Q5_1 (q in 0..31; the stored quant, before Q5_0's -16):
    f16 d, [f16 m], [fifth-bit word: bit e = bit 4 of q[e]], then the nibbles as Q4_0."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= 0 and q.max() <= (15 if qtype == 3 else 31)
    out = bytes([d_bits & 255, d_bits >> 8])
    if qtype in (3, 7):
        out += bytes([m_bits & 255, m_bits >> 8])
    if qtype in (6, 7):
        qh = sum(int((q[e] >> 4) & 1) << e for e in range(32))
        out += qh.to_bytes(4, "little")
    return out + bytes(int(q[j] & 15) | (int(q[16 + j] & 15) << 4) for j in range(16))


def pack_q5_k(d_bits: int, dmin_bits: int, sc, mn, q5) -> bytes:
    """q5[e] in 0..31 for e in 0..255; element 64c + 32h + l: low 4 bits in quant byte
    32c + l (low nibble for h = 0, high for h = 1), fifth bit at bit 2c + h of high-bit
    byte l."""
    q5 = np.asarray(q5, dtype=np.int64)
    assert q5.shape == (256,) and q5.min() >= 0 and q5.max() <= 31
    qh = bytearray(32)
    qs = bytearray(128)
    for c in range(4):
        for h in range(2):
            for l in range(32):
                v = int(q5[64 * c + 32 * h + l])
                qs[32 * c + l] |= (v & 15) << (4 * h)
                qh[l] |= (v >> 4) << (2 * c + h)
    return (bytes([d_bits & 255, d_bits >> 8, dmin_bits & 255, dmin_bits >> 8]) +
            pack_q4_k_scales(sc, mn) + bytes(qh) + bytes(qs))


# ---- second formulation: vectorised numpy decoders ------------------------

def _f16(u8pair: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(u8pair).view(np.float16).astype(np.float64)[..., 0]


def np_dequant(qtype: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = np.asarray(W, dtype=np.uint8)
    if qtype == 1:  # f16, little-endian
        return W.view("<f2").astype(np.float64).reshape(N, K)
    if qtype == 30:  # bf16: the upper half of a binary32
        bits = W.view("<u2").astype(np.uint32) << 16
        return bits.view(np.float32).astype(np.float64).reshape(N, K)
    if qtype == 8:
        blk = W.reshape(N, K // 32, 34)
        d = _f16(blk[:, :, 0:2])
        q = blk[:, :, 2:].view(np.int8).astype(np.float64)
        return (d[:, :, None] * q).reshape(N, K)
    if qtype == 12:
        blk = W.reshape(N, K // 256, 144)
        d = _f16(blk[:, :, 0:2])
        dmin = _f16(blk[:, :, 2:4])
        s = blk[:, :, 4:16].astype(np.int64)
        sc = np.concatenate([s[..., 0:4] & 63,
                             (s[..., 8:12] & 15) | ((s[..., 0:4] >> 6) << 4)], axis=-1)
        mn = np.concatenate([s[..., 4:8] & 63,
                             (s[..., 8:12] >> 4) | ((s[..., 4:8] >> 6) << 4)], axis=-1)
        qs = blk[:, :, 16:].astype(np.int64).reshape(N, K // 256, 4, 32)
        nib = np.stack([qs & 15, qs >> 4], axis=3)  # [N, nb, c, h, l]
        nib = nib.reshape(N, K // 256, 8, 32)  # sub-block j = 2c + h
        w = d[..., None, None] * sc[..., None] * nib - dmin[..., None, None] * mn[..., None]
        return w.reshape(N, K)
    if qtype == 2:
        blk = W.reshape(N, K // 32, 18)
        d = _f16(blk[:, :, 0:2])
        qs = blk[:, :, 2:18].astype(np.int64)
        q = np.concatenate([qs & 15, qs >> 4], axis=-1) - 8  # elements 0..15, 16..31
        return (d[:, :, None] * q).reshape(N, K)
    if qtype in (3, 6, 7):
        bb = {3: 20, 6: 22, 7: 24}[qtype]
        blk = W.reshape(N, K // 32, bb)
        d = _f16(blk[:, :, 0:2])
        m = _f16(blk[:, :, 2:4]) if qtype in (3, 7) else np.zeros_like(d)
        qo = {3: 4, 6: 6, 7: 8}[qtype]
        qs = blk[:, :, qo:qo + 16].astype(np.int64)
        q = np.concatenate([qs & 15, qs >> 4], axis=-1)  # elements 0..15, 16..31
        if qtype in (6, 7):
            ho = qo - 4
            qh = blk[:, :, ho:ho + 4].astype(np.int64)
            word = qh[..., 0] | (qh[..., 1] << 8) | (qh[..., 2] << 16) | (qh[..., 3] << 24)
            q = q | (((word[..., None] >> np.arange(32)) & 1) << 4)
        if qtype == 6:
            q = q - 16
        return (d[:, :, None] * q + m[:, :, None]).reshape(N, K)
    if qtype == 13:
        blk = W.reshape(N, K // 256, 176)
        d = _f16(blk[:, :, 0:2])
        dmin = _f16(blk[:, :, 2:4])
        s = blk[:, :, 4:16].astype(np.int64)
        sc = np.concatenate([s[..., 0:4] & 63,
                             (s[..., 8:12] & 15) | ((s[..., 0:4] >> 6) << 4)], axis=-1)
        mn = np.concatenate([s[..., 4:8] & 63,
                             (s[..., 8:12] >> 4) | ((s[..., 4:8] >> 6) << 4)], axis=-1)
        qh = blk[:, :, 16:48].astype(np.int64)[:, :, None, :]  # [N, nb, 1, l]
        qs = blk[:, :, 48:176].astype(np.int64).reshape(N, K // 256, 4, 32)
        nib = np.stack([qs & 15, qs >> 4], axis=3).reshape(N, K // 256, 8, 32)  # j = 2c + h
        hib = (qh >> np.arange(8)[None, None, :, None]) & 1  # bit j of byte l
        q = nib | (hib << 4)
        w = d[..., None, None] * sc[..., None] * q - dmin[..., None, None] * mn[..., None]
        return w.reshape(N, K)
    if qtype == 14:
        blk = W.reshape(N, K // 256, 210)
        ql = blk[:, :, 0:128].astype(np.int64).reshape(N, K // 256, 2, 2, 32)  # h, r%2, l
        qh = blk[:, :, 128:192].astype(np.int64).reshape(N, K // 256, 2, 1, 32)
        sc = blk[:, :, 192:208].view(np.int8).astype(np.float64).reshape(N, K // 256, 2, 4, 2)
        d = _f16(blk[:, :, 208:210])
        lo = np.concatenate([ql & 15, ql >> 4], axis=3)  # r = 0..3
        hi = (qh >> (2 * np.arange(4)[None, None, None, :, None])) & 3
        q = (lo | (hi << 4)) - 32  # [N, nb, h, r, l]
        scl = np.repeat(sc, 16, axis=-1)  # [N, nb, h, r, 32]
        return (d[..., None, None, None] * scl * q).reshape(N, K)
    raise ValueError(qtype)
