"""The quantizer kernels divide by the tile scale without a division
instruction: with r = RN(1/s), q0 = RN(v r), then two corrections
q <- RN(q + (v - q s) r) with the residual taken exactly by an FMA (the
second correction is Markstein's, IBM J. Res. Dev. 34(1), 1990). This test
checks, in exact rational arithmetic on the CPU, that the result is the
correctly rounded fp32 quotient RN(v/s) that the quantization recipe
specifies, on BF16 inputs and absmax-derived scales (including exact E4M3
midpoints and -0), in the negated form the kernels use. It pins the method,
not the kernels: the GPU parity tests compare the kernels with the oracle."""
import random
from fractions import Fraction as F

import numpy as np


def rn32(x: F) -> F:
    """Round a rational to the nearest fp32 value, ties to even (subnormals
    kept, no overflow in this test's range)."""
    if x == 0:
        return F(0)
    sgn = -1 if x < 0 else 1
    a = -x if x < 0 else x
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    elif F(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = F(2) ** (e - 23)
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return sgn * n * ulp


def quotient(v: F, s: F) -> F:
    """The kernels' steps on negated inputs (nv = -v, nr = -r), each FMA or
    product rounded once."""
    nr = -rn32(1 / s)
    nv = -v
    q = rn32(nv * nr)
    for _ in range(2):
        q = rn32(rn32(q * s + nv) * nr + q)
    return q


def bf16(bits: int) -> F:
    return F(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


def test_fp32_rounding_helper_is_nearest_even():
    """rn32 returns an fp32 value, no farther from x than either fp32
    neighbour of it, and the even one on exact ties."""
    rng = random.Random(5)
    for _ in range(3000):
        x = F(rng.getrandbits(50) + 1, rng.getrandbits(30) + 1) * F(2) ** rng.randint(-60, 20)
        r = rn32(x)
        f = np.float32(float(r))
        assert F(float(f)) == r
        for nb in (np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0))):
            assert abs(r - x) <= abs(F(float(nb)) - x)
    tie = F(1) + F(2) ** -24            # halfway between 1 and 1 + 2^-23
    assert rn32(tie) == 1


def test_two_step_quotient_is_correctly_rounded():
    rng = random.Random(7)
    cases = mismatches = 0
    for tile in range(48):
        lo = rng.randint(-30, 20)
        vals = []
        while len(vals) < 400:
            b = rng.getrandbits(16)
            e = (b >> 7) & 0xFF
            if lo + 127 <= e <= lo + 127 + rng.randint(0, 10):
                vals.append(bf16(b))
        amax = max(abs(v) for v in vals)
        s = rn32(amax / 448)
        # E4M3 midpoints times s and their neighbours, plus signed zeros
        vals += [rn32(F(m, 2) * s) for m in (169 * 2 + 1, 335, 23, 3)] + [F(0)]
        for v in vals:
            cases += 1
            if quotient(v, s) != rn32(v / s):
                mismatches += 1
    assert cases > 19000 and mismatches == 0


def test_negated_form_keeps_the_sign_of_zero():
    """On the negated inputs the chain maps -0 to -0 and +0 to +0 (with the
    textbook order v - q s, a -0 input would come out as +0). With zero
    operands every product and sum below is exact, so float32 numpy
    arithmetic follows the FMA results exactly."""
    s = np.float32(3.0 / 448.0)
    nr = -np.float32(1.0) / s
    for v in (np.float32(-0.0), np.float32(0.0)):
        nv = -v
        q = nv * nr
        for _ in range(2):
            q = (q * s + nv) * nr + q
        assert q == 0 and np.signbit(q) == np.signbit(v)
    # textbook order for comparison: q0 = v r, q1 = q0 + (v - q0 s) r loses -0
    v = np.float32(-0.0)
    r = np.float32(1.0) / s
    q0 = v * r
    q1 = (v - q0 * s) * r + q0
    assert not np.signbit(q1)
