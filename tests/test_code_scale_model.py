"""Host model of the quantisers' code arithmetic (CPU, exact rationals).

The kernels turn y into its e4m3 code as e4m3(fma(s, hi, s * lo)). Here
s = y * pre, hi = RN(448 / A), lo = RN((448 - hi A) / A), and A = max|y| * pre.
Every fp32 rounding RN is modelled exactly with fractions. The tests check the
three facts the parity tests rely on:
- the fma residual 448 - hi A is exact in fp32;
- with bf16 inputs, the code equals the e4m3 rounding of RN(448 y / max|y|),
  exact midpoints included;
- with fp32 inputs, it differs from that only where 448 y / max|y| lies within
  2^-44 relative of an fp32 rounding boundary.
A single-word reciprocal would miss the bf16 midpoints; this is shown on the
worked case max|y| = 25.5, y = 1.1953125, whose quotient is exactly 21."""
from fractions import Fraction

import numpy as np
import pytest
import torch


def rn32(r: Fraction) -> Fraction:
    """Round a rational to the nearest fp32 value, ties to even (normal range)."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = a / Fraction(2) ** (e - 23)  # in [2^23, 2^24)
    m = round(q)  # Fraction.__round__ rounds half to even
    return sign * m * Fraction(2) ** (e - 23)


def e4m3(v: Fraction) -> int:
    f = np.float32(float(v))  # v is an fp32 value, so the conversion is exact
    t = torch.tensor([min(max(float(f), -448.0), 448.0)], dtype=torch.float32)
    return int(t.to(torch.float8_e4m3fn).view(torch.uint8)[0])


def kernel_code(y: Fraction, amax: Fraction) -> int:
    pre = Fraction(2) ** 100 if amax < Fraction(2) ** -100 else Fraction(1)
    a = amax * pre
    hi = rn32(Fraction(448) / a)
    resid = 448 - hi * a
    assert rn32(resid) == resid, "the fma residual must be exact"
    lo = rn32(resid / a)
    s = y * pre
    return e4m3(rn32(s * hi + rn32(s * lo)))


def single_word_code(y: Fraction, amax: Fraction) -> int:
    return e4m3(rn32(y * rn32(Fraction(448) / amax)))


def exact_code(y: Fraction, amax: Fraction) -> int:
    return e4m3(rn32(Fraction(448) * y / amax))


def _draw(n, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, generator=g) * torch.exp2(torch.randint(-6, 7, (n,), generator=g).float())
    return [Fraction(float(v)) for v in x.to(dtype).float()]


def test_worked_midpoint():
    # 448 / 25.5 * 1.1953125 = 21 exactly, midway between e4m3 20 and 22:
    # ties to even gives 20.
    y, amax = Fraction(1.1953125), Fraction(25.5)
    assert Fraction(448) * y / amax == 21
    assert exact_code(y, amax) == kernel_code(y, amax)
    assert single_word_code(y, amax) != exact_code(y, amax)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_bf16_codes_equal_the_exact_rounding(seed):
    # max|y| = 25.5 = 51/2, as in the outlier draws; bf16 values whose
    # significand is 153 = 3 x 51 give quotients 21 x 2^k, e4m3 midpoints.
    amax = Fraction(25.5)
    xs = [v for v in _draw(600, torch.bfloat16, seed) if abs(v) < amax]
    xs += [amax, -amax] + [sgn * Fraction(153) * Fraction(2) ** k for k in range(-12, -2) for sgn in (1, -1)]
    midpoints = 0
    for y in xs:
        assert kernel_code(y, amax) == exact_code(y, amax), (y, amax)
        q = Fraction(448) * y / amax
        midpoints += rn32(q) == q and e4m3(q) != e4m3(rn32(q * (1 + Fraction(1, 1 << 20))))
    assert midpoints > 0  # the draw does reach exact e4m3 midpoints


@pytest.mark.parametrize("seed", [4, 5])
def test_fp32_codes_differ_only_next_to_a_boundary(seed):
    xs = _draw(600, torch.float32, seed)
    amax = max(abs(v) for v in xs)
    for y in xs:
        if kernel_code(y, amax) != exact_code(y, amax):
            q = Fraction(448) * y / amax
            lo, hi = q * (1 - Fraction(1, 1 << 44)), q * (1 + Fraction(1, 1 << 44))
            assert exact_code(lo, Fraction(448)) != exact_code(hi, Fraction(448)), y


def test_tiny_maximum_is_prescaled():
    # max|y| below 2^-100: 448 / max|y| would overflow fp32 without the 2^100
    # pre-scale; with it the codes are the exact rounding's.
    # |y| in [2^-138, 2^-122): exact fp32 subnormals for 8-bit significands
    xs = [v * Fraction(2) ** -124 for v in _draw(400, torch.bfloat16, 6) if Fraction(2) ** -14 <= abs(v) < 4]
    amax = max(abs(v) for v in xs)
    assert Fraction(448) / amax > Fraction(2) ** 128
    for y in xs:
        assert kernel_code(y, amax) == exact_code(y, amax)
