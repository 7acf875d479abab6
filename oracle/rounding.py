"""Rounding of the attention weights P (oracle).

Source: "在 agent 时代如何快速验证 kernel 对精度的影响", section
"注意力权重：直接转 fp8 随上下文变差，先放大就和 bf16 差不多".  The naive
kernel there rounds only the P that multiplies V, in one of four ways:
keep f32, round to bf16, round to fp8 e4m3, or multiply by 448 (the e4m3
maximum), round to e4m3 and divide the 448 back out.  The same section names
256 as the factor other fp8 attention kernels scale by before the cast; that
variant is mode 4.  Its closing question -- feed the e4m3 P straight to the
tensor-core P.V -- is mode 5: p~ = e4m3(p) as mode 2, and the operand that
multiplies the int8 V values is the float32 product p~ * v_scale rounded once
to f16 precision (11 significant bits, nearest-even).  V stays exact (an
int8 value is exact in f16); the per-token scale has to ride on the P side,
and one f16 operand holds p~ * v_scale only after that rounding.

Both formats are written from their definitions, not by bit tricks:
a value v >= 0 is rounded on the grid of its binade,

    quantum = 2^(max(floor(log2 v), emin) - mbits)
    round(v) = rint_half_even(v / quantum) * quantum

with (mbits, emin) = (7, -126) for bf16 and (3, -6) for e4m3.  The binade
floor at emin makes subnormals come out right.  e4m3 here is the OCP FP8
E4M3 format (bias 7, no infinities, largest finite 448, smallest subnormal
2^-9) with saturation to 448.  The division v / quantum is exact in float64
because quantum is a power of two.

P values are non-negative (they are exp of a non-positive number), so only
v >= 0 needs handling; negative inputs are rounded by symmetry anyway.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
P_MODES = {0: "f32", 1: "bf16", 2: "e4m3", 3: "e4m3x448", 4: "e4m3x256", 5: "e4m3direct"}
DIRECT = 5                                       # the mode whose P.V operand is rounded


def _round_grid(v, mbits: int, emin: int):
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(np.where(a > 0, a, 1.0))   # a = f * 2^e, f in [0.5, 1)
    e = np.maximum(e - 1, emin)                 # floor(log2 a), floored at emin
    quantum = np.ldexp(1.0, e - mbits)
    r = np.rint(a / quantum) * quantum          # ties to even
    return np.where(a > 0, np.copysign(r, v), v)


def bf16(v):
    """Round float32 values to bfloat16 (nearest, ties to even). float64 out."""
    return _round_grid(np.asarray(v, dtype=np.float32), 7, -126)


def e4m3(v):
    """Round to OCP FP8 E4M3 (nearest, ties to even, saturate to +-448)."""
    r = _round_grid(np.asarray(v, dtype=np.float32), 3, -6)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def f16_significand(v):
    """Round to 11 significant bits (the f16 significand), nearest-even, with
    no exponent range: the value a kernel gets by scaling into f16's normal
    range by a power of two, rounding to f16, and scaling back.  float64 out."""
    return _round_grid(np.asarray(v, dtype=np.float64), 10, -10**6)


def pv_operand(p_rounded, v_scale, mode: int):
    """The weight that multiplies key t's int8 V values: p~_t * v_scale_t.

    Modes 0-4 carry it exactly (float64 here); mode 5 rounds the float32
    product to 11 significant bits.  float64 out."""
    if mode == DIRECT:
        prod = np.multiply(np.asarray(p_rounded, np.float32), np.asarray(v_scale, np.float32),
                           dtype=np.float32)
        return f16_significand(prod)
    return np.asarray(p_rounded, np.float64) * np.asarray(v_scale, np.float64)


def round_p(p, mode: int):
    """The round_p variants, applied to float32 P values.

    mode 0: identity; 1: bf16(p); 2 and 5: e4m3(p);
    3: e4m3(f32(p * 448)) / 448 -- the product is rounded to float32 first
       (the kernel multiplies in float32), the final division is exact
       float64 arithmetic on the e4m3 value;
    4: e4m3(p * 256) / 256 -- both scalings by a power of two are exact.
    Returns float64.
    """
    p = np.asarray(p, dtype=np.float32)
    if mode == 0:
        return p.astype(np.float64)
    if mode == 1:
        return bf16(p)
    if mode == 2 or mode == DIRECT:
        return e4m3(p)
    if mode == 3:
        scaled = np.multiply(p, np.float32(E4M3_MAX), dtype=np.float32)
        return e4m3(scaled) / E4M3_MAX
    if mode == 4:
        return e4m3(np.float64(p) * 256.0) / 256.0
    raise ValueError(f"unknown p_mode {mode}")


def round_p_f32(p, mode: int):
    """round_p as the exact-mode sequence uses it: every value is a float32.

    Modes 0-2 give values that float32 holds exactly.  Mode 3 divides the
    e4m3 value by 448 with one float32 rounding (IEEE division), since the
    exact mode rounds every float32 operation separately.  Mode 5 has no
    exact-mode form (the sequential scan has no tensor-core operand).
    """
    if mode == DIRECT:
        raise ValueError("p_mode 5 (e4m3 P into the tensor-core P.V) is a fast-mode rounding")
    p = np.asarray(p, dtype=np.float32)
    if mode == 3:
        scaled = np.multiply(p, np.float32(E4M3_MAX), dtype=np.float32)
        return np.divide(e4m3(scaled).astype(np.float32), np.float32(E4M3_MAX),
                         dtype=np.float32)
    return round_p(p, mode).astype(np.float32)
