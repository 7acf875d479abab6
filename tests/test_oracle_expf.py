"""Pins for the oracle's table-driven expf ("Kestrel_VLLM - 18", §3.3)."""

import math
from fractions import Fraction

import mpmath
import numpy as np
import pytest

from conftest import read_golden
from oracle import expf_tang as E


def f32_ulps(a, b):
    """Distance in float32 ULPs between two non-negative float32 values."""
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


def test_constants_reproduce_page_decimals():
    g = read_golden("expf_constants.txt")
    assert E.K == float(g["K"])
    assert E.C2 == float(g["C2"])
    assert E.C0 == float(g["C0"])
    assert E.C1 == float(g["C1"])
    assert E.OVERFLOW_X == float(np.float32(float(g["overflow_x"])))
    assert E.UNDERFLOW_X == float(g["underflow_x"])


def test_constants_correctly_rounded_against_mpmath():
    # mpmath is a different arbitrary-precision library than the decimal
    # module the oracle uses; each constant must be within half an ULP.
    mpmath.mp.dps = 60
    ln2 = mpmath.log(2)
    for got, exact in ((E.K, 64 / ln2), (E.C2, ln2 / 64), (E.C0, mpmath.mpf(1) / 6)):
        assert abs(mpmath.mpf(got) - exact) <= mpmath.mpf(math.ulp(got)) / 2


def test_table_is_round_to_nearest_of_2_pow_j_over_64():
    # t = RN(2^(j/64)) iff the exact value lies within half an ULP of t, i.e.
    # (t - h)^64 < 2^j < (t + h)^64 -- checked in exact rational arithmetic.
    assert len(E.TABLE) == 64
    assert E.TABLE[0] == 1.0
    assert E.TABLE[32] == math.sqrt(2.0)   # sqrt is correctly rounded
    for j in range(1, 64):
        t = Fraction(E.TABLE[j])
        h = Fraction(math.ulp(E.TABLE[j])) / 2
        assert (t - h) ** 64 < 2 ** j < (t + h) ** 64, j


def test_fma_is_exact_single_rounding():
    # a*b + c where the exact result needs more than 53 bits
    a = 1.0 + 2.0 ** -30
    b = 1.0 + 2.0 ** -30
    c = -1.0
    exact = Fraction(a) * Fraction(b) + Fraction(c)       # 2^-29 + 2^-60
    assert E.fma(a, b, c) == float(exact)
    assert E.fma(a, b, c) != a * b + c                     # two roundings differ
    assert E.fma(2.0, 3.0, 4.0) == 10.0


def test_special_values():
    assert E.expf_tang(0.0) == np.float32(1.0)
    assert E.expf_tang(-0.0) == np.float32(1.0)
    assert E.expf_tang(-np.inf) == 0.0
    assert E.expf_tang(np.float32(-104.5)) == 0.0
    assert E.expf_tang(np.float32(-103.0)) > 0.0           # subnormal result
    assert E.expf_tang(np.float32(100.0)) == np.inf
    assert f32_ulps(E.expf_tang(np.float32(1.0)), np.float32(math.exp(1.0))) <= 1


def test_polynomial_relative_error_bound():
    # The page's accuracy statement: relative error ~ r^4/24 ~ 3.6e-11 before
    # the final float rounding.  A wrong coefficient or table entry breaks it.
    bound = float(read_golden("expf_constants.txt")["rel_error_bound"])
    mpmath.mp.dps = 40
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.uniform(-100, 0, 3000), rng.uniform(-0.05, 0, 1000)])
    worst = 0.0
    for x in xs.astype(np.float32):
        got = E.expf_tang_double(float(x))
        ref = mpmath.exp(mpmath.mpf(float(x)))
        worst = max(worst, float(abs(got - ref) / ref))
    assert worst <= 1.1 * bound, worst


def test_within_one_ulp_of_correctly_rounded_on_400002_samples():
    # Same probe design as the page: 400002 float32 samples in [-100, 0],
    # random plus dense near 0, compared with (float)exp(double).
    g = read_golden("expf_constants.txt")
    n = int(g["samples"])
    rng = np.random.default_rng(20260101)
    xs = np.concatenate([
        rng.uniform(-100.0, 0.0, n // 2),
        -np.abs(rng.standard_normal(n - n // 2 - 2)) * 1e-3,
        [0.0, -100.0],
    ]).astype(np.float32)
    got = E.expf_tang_array(xs)
    ref = np.array([np.float32(math.exp(float(x))) for x in xs], dtype=np.float32)
    d = f32_ulps(got, ref)
    assert d.max() <= 1
    rate = float((d > 0).mean())
    # The page measured 0.007%; allow an order of magnitude of sampling slack.
    assert rate <= 10 * float(g["mismatch_rate"]), rate
