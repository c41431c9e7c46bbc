"""The activation quantiser's kernels compute q = rint(fl(x / s)) (binary32 division, round
half to even) as w = fl(x * fl(1 / s)), falling back to the division when w is within 2^-14
of a half-integer, not below 128 in magnitude, or not finite.  This checks that rule in
binary32 numpy arithmetic (each operation correctly rounded, as on the GPU) against the
definition, on random blocks over a wide range of scales, subnormal ones included, and on
values placed at and next to every rounding boundary.  The kernels' bytes are compared with
the oracle's bit for bit by the GPU tests."""
import numpy as np

F = np.float32


def rule(x, s):
    r = F(1) / s
    with np.errstate(over="ignore", invalid="ignore"):
        w = x * r
        a = np.abs(w)
        f = a - np.floor(a)
        fallback = (np.abs(f - F(0.5)) < F(2.0 ** -14)) | ~(a < F(128))
    return np.where(fallback, np.rint(x / s), np.rint(w))


def definition(x, s):
    return np.rint(x / s)


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
    k = np.arange(-127, 127, dtype=np.float32) + F(0.5)  # every half-integer in range
    base = (k[None, :] * s[:, None]).astype(np.float32)
    for steps in range(-3, 4):
        x = base
        for _ in range(abs(steps)):
            x = np.nextafter(x, np.float32(np.inf) if steps > 0 else np.float32(-np.inf))
        x = x.astype(np.float32)
        ss = np.broadcast_to(s[:, None], x.shape)
        assert np.array_equal(rule(x, ss), definition(x, ss)), steps
