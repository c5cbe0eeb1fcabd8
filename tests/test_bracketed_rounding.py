"""The bracketed rounding that the depthwise QLinearConv's requantization and
the staged row quantization of A use for their 8-bit codes, checked with
exact rational arithmetic on the host (no GPU, no oracle: the kernels' own
parity tests compare their codes with the oracle's).

Claim: with q the IEEE fp32 quotient fl(v / s), r = fl(1 / s),
rh = fl(r * (1 + 2^-20)), rl = fl(r * (1 - 2^-20)) and mz = 1.5 * 2^23 + z,
let H = round(v * rh + mz) and L = round(v * rl + mz) (one rounding each,
to the nearest integer, ties to even: the fma's result in [2^23, 2^24)).
If H == L then H - 1.5 * 2^23 == z + rint(q) (rint: nearest, ties to even),
for |v / s| below 2^20.
"""
from fractions import Fraction as F

import numpy as np
import pytest

M15 = 3 << 22  # 1.5 * 2^23


def rint_even(x):
    """Nearest integer to the rational x, ties to even."""
    fl = x.numerator // x.denominator
    d = x - fl
    if d > F(1, 2):
        return fl + 1
    if d < F(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def ends(v, s, z):
    r = np.float32(1) / s
    rh = np.float32(r * np.float32(1 + 2.0 ** -20))
    rl = np.float32(r * np.float32(1 - 2.0 ** -20))
    mz = F(M15 + z)
    return rint_even(F(float(v)) * F(float(rh)) + mz), rint_even(F(float(v)) * F(float(rl)) + mz)


def check(v, s, z):
    """(bracket agreed, agreed value is right); a disagreement is allowed."""
    H, L = ends(v, s, z)
    q = np.float32(v) / np.float32(s)   # IEEE division, correctly rounded
    want = z + rint_even(F(float(q)))
    return H == L, (H != L) or (H - M15 == want)


@pytest.mark.parametrize("seed", range(4))
def test_random_quotients(seed):
    rng = np.random.default_rng(seed)
    small = small_agreed = 0
    for _ in range(3000):
        s = np.float32(rng.choice([1.0, 0.5, 2.0, 0.05, 0.0037 * 0.01, 3.0, 7.3e-3]) * rng.uniform(0.5, 2.0))
        z = int(rng.integers(-128, 256))
        mag = rng.choice([1.0, 300.0, 2.0 ** 19])
        v = np.float32(rng.uniform(-1, 1) * float(s) * mag)
        agree, right = check(v, s, z)
        assert right, (v, s, z)
        if mag <= 300.0:
            small += 1
            small_agreed += agree
    # the window is 2^-20 |q| wide: below 300 the ends almost always agree
    assert small_agreed > 0.99 * small


@pytest.mark.parametrize("s", [1.0, 0.5, 2.0, 3.0, 0.1, 1.0 / 3.0])
def test_ties_and_their_neighbours(s):
    """Quotients on a tie and one or two ulps beside it: where the ends
    agree they give the right code, and an exact tie never agrees."""
    s = np.float32(s)
    for j in range(-300, 300, 7):
        t = np.float32(j + 0.5) * s
        for v in (t, np.nextafter(t, np.float32(np.inf)), np.nextafter(t, np.float32(-np.inf)),
                  np.nextafter(np.nextafter(t, np.float32(np.inf)), np.float32(np.inf))):
            v = np.float32(v)
            agree, right = check(v, s, 7)
            assert right, (v, s)
            q = np.float32(v) / s
            if F(float(q)) - F(float(q)).numerator // F(float(q)).denominator == F(1, 2):
                assert not agree, (v, s)


def test_zero_and_extremes():
    for s in (np.float32(1.0), np.float32(0.0037)):
        for v in (np.float32(0.0), np.float32(-0.0)):
            H, L = ends(v, s, 9)
            assert H == L == M15 + 9
        big = np.float32(float(s) * (2.0 ** 20 - 1))
        assert check(big, s, 0)[1] and check(np.float32(-big), s, 255)[1]
