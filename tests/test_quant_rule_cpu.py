"""The activation quantiser's kernels compute q = clamp(rint(fl(x / s)), -127, 127)
(binary32 division, round half to even) as w = fl(x * fl(1 / s)) rounded to an integer by
adding 1.5 * 2^23, falling back to the division when w is within 2^-14 of a half-integer
(its exact residual w - rint(w) is at least 1/2 - 2^-14 in magnitude), not below 127.25 in
magnitude, or not finite.  This checks that rule in binary32 numpy arithmetic (each
operation correctly rounded, as on the GPU) against the definition, on random blocks over a
wide range of scales, subnormal ones included, and on values placed at and next to every
rounding boundary.  The kernels' bytes are compared with the oracle's bit for bit by the GPU
tests."""
import numpy as np

F = np.float32
MAGIC = F(12582912.0)  # 1.5 * 2^23


def rule(x, s):
    with np.errstate(over="ignore", invalid="ignore"):
        r = F(1) / s
        w = x * r
        t = w + MAGIC  # ties to even: MAGIC + rint(w) for |w| < 2^22
        rw = t - MAGIC
        d = w - rw
        fast = (np.abs(d) < F(0.5) - F(2.0 ** -14)) & (np.abs(w) < F(127.25))
        slow = np.clip(np.rint(x / s), -127, 127)
    assert t.dtype == np.float32 and d.dtype == np.float32
    return np.where(fast, rw, slow)


def definition(x, s):
    return np.clip(np.rint(x / s), -127, 127)


def blocks(rng, n, exp_lo, exp_hi):
    amax = (rng.random(n, dtype=np.float32) + F(0.5)) * np.exp2(
        rng.integers(exp_lo, exp_hi, n)).astype(np.float32)
    s = (amax / F(127)).astype(np.float32)
    x = ((rng.random((n, 32), dtype=np.float32) * 2 - 1) * amax[:, None]).astype(np.float32)
    x[:, 0] = amax  # the block's maximum itself
    return x, s[:, None]


def test_random_blocks_every_scale():
    rng = np.random.Generator(np.random.PCG64(11))
    for lo, hi in ((-140, -120), (-30, 30), (60, 100)):
        x, s = blocks(rng, 200000, lo, hi)
        ok = s[:, 0] > 0
        x, s = x[ok], s[ok]
        assert np.array_equal(rule(x, s), definition(x, s))


def test_values_at_and_next_to_every_boundary():
    rng = np.random.Generator(np.random.PCG64(12))
    s = (rng.random(4000, dtype=np.float32) + F(0.5)) * np.exp2(
        rng.integers(-20, 20, 4000)).astype(np.float32)
    k = np.arange(-128, 128, dtype=np.float32) + F(0.5)  # every half-integer, +-127.5 too
    base = (k[None, :] * s[:, None]).astype(np.float32)
    for steps in range(-3, 4):
        x = base
        for _ in range(abs(steps)):
            x = np.nextafter(x, np.float32(np.inf) if steps > 0 else np.float32(-np.inf))
        x = x.astype(np.float32)
        ss = np.broadcast_to(s[:, None], x.shape)
        assert np.array_equal(rule(x, ss), definition(x, ss)), steps


def test_fallback_is_needed_and_codes_read_from_the_bits():
    # without the division fallback the boundary values do round differently (the test
    # above is sensitive to it)
    rng = np.random.Generator(np.random.PCG64(13))
    s = (rng.random(4000, dtype=np.float32) + F(0.5)) * np.exp2(
        rng.integers(-20, 20, 4000)).astype(np.float32)
    k = np.arange(-127, 127, dtype=np.float32) + F(0.5)
    x = (k[None, :] * s[:, None]).astype(np.float32)
    ss = np.broadcast_to(s[:, None], x.shape)
    with np.errstate(over="ignore", invalid="ignore"):
        naive = (x * (F(1) / ss) + MAGIC) - MAGIC
    assert not np.array_equal(naive, definition(x, ss))
    # MAGIC + q: its bits less MAGIC's are q, its low byte is q as int8
    q = np.arange(-127, 128)
    bits = (q.astype(np.float32) + MAGIC).view(np.int32)
    assert np.array_equal(bits - np.int32(0x4B400000), q)
    assert np.array_equal((bits & 255).astype(np.uint8).view(np.int8), q.astype(np.int8))


def div127_rule(bits):
    """The kernels' s = amax / 127: q0 = fl(a c), r = fl(fma(-q0, 127, a)), fl(fma(r, c, q0)),
    c = fl(1/127), emulated exactly in float64 (the products are exact there; the final sum is
    rounded once to binary32, ties resolved by the exact error of the float64 sum)."""
    a = bits.view(np.float32)
    c = F(1) / F(127)
    q0 = a * c
    r = (a.astype(np.float64) - 127.0 * q0.astype(np.float64)).astype(np.float32)
    q064 = q0.astype(np.float64)
    rc = r.astype(np.float64) * np.float64(c)
    s = q064 + rc
    bb = s - q064
    e = (q064 - (s - bb)) + (rc - bb)
    t = s.astype(np.float32)
    t64 = t.astype(np.float64)
    up = np.nextafter(t, np.float32(np.inf))
    dn = np.nextafter(t, np.float32(-np.inf))
    res = t.copy()
    m1 = (s == (t64 + up.astype(np.float64)) / 2) & (e > 0)
    res[m1] = up[m1]
    m2 = (s == (t64 + dn.astype(np.float64)) / 2) & (e < 0)
    res[m2] = dn[m2]
    return res


def test_division_by_127_is_correctly_rounded():
    """Every 61st non-negative finite binary32 bit pattern (35 M values from 0 to FLT_MAX,
    subnormals included) and every pattern near powers of two and of 127: the kernels'
    fma-corrected quotient equals the correctly rounded a / 127.  With MQ_EXHAUSTIVE=1 every
    one of the 2^31 - 2^23 patterns is checked (a few minutes; it passes)."""
    import os
    top = int(np.float32(3.4028235e38).view(np.uint32))
    stride = 1 if os.environ.get("MQ_EXHAUSTIVE") == "1" else 61
    step = 1 << 24
    for start in range(0, top + 1, step * stride):
        bits = np.arange(start, min(start + step * stride, top + 1), stride,
                         dtype=np.uint64).astype(np.uint32)
        a = bits.view(np.float32)
        assert np.array_equal(div127_rule(bits).view(np.uint32), (a / F(127)).view(np.uint32))
    near = []
    for e in range(-149, 128):
        for base in (np.float32(2.0) ** e, np.float32(127.0) * np.float32(2.0) ** (e - 7)):
            b = np.float32(base).view(np.uint32).astype(np.int64)
            near.append(np.arange(b - 64, b + 64))
    nb = np.unique(np.clip(np.concatenate(near), 0, top)).astype(np.uint32)
    assert np.array_equal(div127_rule(nb).view(np.uint32), (nb.view(np.float32) / F(127)).view(np.uint32))
