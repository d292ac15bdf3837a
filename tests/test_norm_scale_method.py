"""Error bound of the RMSNorm row scale's double-float method, on the CPU.

The GPU kernels form sqrt(d) / (sqrt(h + l) + eps) as an unevaluated fp32 pair
from approximate reciprocal and reciprocal-square-root values of the special
function unit, each refined by a Newton step and corrected by exact FMA
residues.  This test replays those steps in exactly rounded fp32 arithmetic
(every fma rounded once from its exact value) with the approximate values
pushed to the edges of their documented error bands, and checks the pair
against the quotient evaluated to 50 significant digits.  The bound the kernel
relies on is 2^-44 relative (the bf16 outputs it scales are 2^-8 wide).
"""
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

getcontext().prec = 50

F32 = np.float32
SFU_RSQRT_REL = 2.0 ** -22.9  # rsqrt.approx.f32 maximum relative error
SFU_RCP_REL = 2.0 ** -23  # rcp.approx.f32: about one ulp


def to_f32(x: Fraction) -> np.float32:
    """Correctly rounded (nearest-even) fp32 value of an exact rational."""
    if x == 0:
        return F32(0.0)
    f64 = float(x)  # nearest double; fix the rare double rounding at an fp32 midpoint
    f = F32(f64)
    lo, hi = (np.nextafter(f, F32(-np.inf)), f) if Fraction(float(f)) > x else (f, np.nextafter(f, F32(np.inf)))
    mid = (Fraction(float(lo)) + Fraction(float(hi))) / 2
    if x < mid:
        return lo
    if x > mid:
        return hi
    return lo if (lo.view(np.uint32) & 1) == 0 else hi


def fma(a, b, c) -> np.float32:
    return to_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def add(a, b):
    return to_f32(Fraction(float(a)) + Fraction(float(b)))


def sub(a, b):
    return to_f32(Fraction(float(a)) - Fraction(float(b)))


def mul(a, b):
    return to_f32(Fraction(float(a)) * Fraction(float(b)))


def two_sum(a, b):
    s = add(a, b)
    z = sub(s, a)
    e = add(sub(a, sub(s, z)), sub(b, z))
    return s, e


class Sfu:
    """Approximate values at a chosen point of their error bands."""

    def __init__(self, rng):
        self.rng = rng

    def _err(self, bound):
        return self.rng.choice([-bound, -bound / 2, 0.0, bound / 2, bound])

    def rsqrt(self, x):
        if float(x) == 0.0:
            return F32(np.inf)
        exact = Decimal(1) / Decimal(float(x)).sqrt()
        return to_f32(Fraction(exact) * Fraction(1 + self._err(SFU_RSQRT_REL)))

    def rcp(self, x):
        return to_f32(Fraction(1) / Fraction(float(x)) * Fraction(1 + self._err(SFU_RCP_REL)))


def sqrt_pair(v, v_lo, sfu):
    g = sfu.rsqrt(v)
    pos = float(v) > 0.0
    s0 = mul(v, g) if pos else F32(0.0)
    s = fma(fma(-s0, s0, v), mul(F32(0.5), g) if pos else F32(0.0), s0)
    half_inv_s = mul(F32(0.5), sfu.rcp(s)) if pos else F32(0.0)
    p = mul(s, s)
    pe = fma(s, s, -p)
    s_lo = mul(add(sub(sub(v, p), pe), v_lo), half_inv_s)
    return s, s_lo


def row_scale(h, l, d, eps, sfu):
    r, r_lo = sqrt_pair(h, l, sfu)
    dh, de = two_sum(r, eps)
    de = add(de, r_lo)
    den_hi = add(dh, de)
    den_lo = sub(de, sub(den_hi, dh))
    sd, sd_lo = sqrt_pair(F32(d), F32(0.0), sfu)
    c = sfu.rcp(den_hi)
    q0 = mul(sd, c)
    q = fma(fma(-q0, den_hi, sd), c, q0)
    rem = add(fma(-q, den_hi, sd), fma(-q, den_lo, sd_lo))
    q_lo = mul(rem, c)
    inv_hi = add(q, q_lo)
    inv_lo = sub(q_lo, sub(inv_hi, q))
    return inv_hi, inv_lo


def exact_scale(h, l, d, eps) -> Decimal:
    norm = (Decimal(float(h)) + Decimal(float(l))).sqrt()
    return Decimal(d).sqrt() / (norm + Decimal(float(eps)))


@pytest.mark.parametrize("d", [128, 1000, 1024, 2816, 4096])
@pytest.mark.parametrize("eps", [1e-6, 0.25, 0.0])
def test_row_scale_pair_within_bound(d, eps):
    rng = np.random.default_rng(d * 7 + int(eps * 1e6))
    sfu = Sfu(rng)
    eps32 = F32(eps)
    worst = 0.0
    for _ in range(60):
        h = F32(10.0 ** rng.uniform(-20, 20))
        # the low part of a TwoSum-accumulated sum of squares: at most half an ulp of h
        ulp = float(np.spacing(h))
        l = F32(rng.uniform(-0.5, 0.5) * ulp)
        hi, lo = row_scale(h, l, d, eps32, sfu)
        got = Decimal(float(hi)) + Decimal(float(lo))
        want = exact_scale(h, l, d, eps32)
        worst = max(worst, float(abs(got - want) / want))
        # the pair is normalised: |lo| <= half an ulp of hi
        assert abs(float(lo)) <= float(np.spacing(hi)) / 2
    assert worst < 2.0 ** -44, worst


def test_row_scale_zero_row():
    """An all-zero row has norm 0: the scale is sqrt(d) / eps, not a NaN."""
    sfu = Sfu(np.random.default_rng(1))
    hi, lo = row_scale(F32(0.0), F32(0.0), 1024, F32(0.25), sfu)
    got = Decimal(float(hi)) + Decimal(float(lo))
    assert abs(got - Decimal(128)) / Decimal(128) < Decimal(2) ** -44
