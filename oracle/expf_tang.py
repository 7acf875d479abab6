"""Table-driven float32 exp in double arithmetic (oracle).

Source: "Kestrel_VLLM - 18 · 投机解码位级对拍收口", §3.3 ("消除 t=27").  The page
describes an expf built from a 64-entry table of 2^(j/64) and a three-term
polynomial, evaluated in double with explicit fused multiply-adds, and rounded
once to float at the end.  This is the classic table-driven method of
P. T. P. Tang, "Table-driven implementation of the exponential function in
IEEE floating-point arithmetic", ACM TOMS 15(2), 1989.  For x in float32:

    n = rint_half_even(x * K)                 K  = RN(64 / ln 2)
    r = fma(-n, C2, x)                        C2 = RN(ln 2 / 64)
    j = n mod 64,  m = floor(n / 64)
    p = fma(fma(r, C0, C1), r*r, r)           C0 = RN(1/6), C1 = 1/2
    q = fma(T[j], p, T[j])                    T[j] = RN(2^(j/64))
    expf(x) = RN_f32(2^m * q)

so exp(x) = 2^m * 2^(j/64) * e^r with |r| <= ln2/128 and
e^r - 1 ~= r + r^2/2 + r^3/6 (relative error ~ r^4/24 ~ 3.6e-11).
x > RN_f32(88.7228394) returns RN_f32(exp(x)) (overflow side); x < -104
returns 0.

Constants are computed here from first principles with the decimal module at
60 significant digits and rounded once to double (CPython's float(Decimal)
is correctly rounded).  The decimals the page prints for K, C2, C0, C1 are used
only as a cross-check in the tests.  The fused multiply-add is done exactly in
rational arithmetic (CPython's int / int true division is correctly rounded),
because Python 3.12 has no math.fma.
"""

from __future__ import annotations

import math
from decimal import Decimal, localcontext

import numpy as np

with localcontext() as _ctx:
    _ctx.prec = 60
    _LN2 = Decimal(2).ln()
    K = float(Decimal(64) / _LN2)
    C2 = float(_LN2 / Decimal(64))
    C0 = float(Decimal(1) / Decimal(6))
    C1 = 0.5
    TABLE = tuple(float((_LN2 * Decimal(j) / Decimal(64)).exp()) for j in range(64))

OVERFLOW_X = float(np.float32(88.7228394))
UNDERFLOW_X = -104.0


def fma(a: float, b: float, c: float) -> float:
    """Correctly rounded a*b + c for finite doubles (exact rational sum)."""
    na, da = float(a).as_integer_ratio()
    nb, db = float(b).as_integer_ratio()
    nc, dc = float(c).as_integer_ratio()
    dab = da * db                     # both denominators are powers of two
    d = max(dab, dc)
    n = na * nb * (d // dab) + nc * (d // dc)
    return n / d                      # correctly rounded


def expf_tang_double(x) -> float:
    """The double 2^m * q before the final float rounding (x in range)."""
    x = float(np.float32(x))
    t = x * K
    n = round(t)                      # Python round(): ties to even
    r = fma(-float(n), C2, x)
    j = n & 63                        # two's-complement semantics on ints
    m = n >> 6                        # arithmetic shift = floor(n / 64)
    z = r * r
    p = fma(fma(r, C0, C1), z, r)
    q = fma(TABLE[j], p, TABLE[j])
    return math.ldexp(q, m)           # exact: 2^m * q stays a normal double


def expf_tang(x) -> np.float32:
    """float32 exp by the table-driven method (scalar)."""
    x = float(np.float32(x))
    if x > OVERFLOW_X:
        if x >= 710.0:                      # math.exp would raise
            return np.float32(np.inf)
        with np.errstate(over="ignore"):
            return np.float32(math.exp(x))  # beyond float32 max -> inf
    if x < UNDERFLOW_X:
        return np.float32(0.0)
    return np.float32(expf_tang_double(x))


def expf_tang_array(x) -> np.ndarray:
    """Elementwise expf_tang over a float32 array (plain loop)."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.float32)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = expf_tang(flat_in[i])
    return out
