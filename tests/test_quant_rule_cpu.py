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
