"""Pins for the oracle's P rounding ("在 agent 时代如何快速验证 kernel 对精度的影响",
section "注意力权重")."""

import itertools

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import rounding as R


def e4m3_values():
    """All non-negative finite OCP E4M3 values, decoded from their bit fields
    (bias 7; exponent field 0 = subnormal; S.1111.111 is NaN)."""
    vals = []
    for e, m in itertools.product(range(16), range(8)):
        if e == 15 and m == 7:
            continue
        vals.append((m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(sorted(vals))


def brute_nearest_even(v, grid, mant_of):
    """Nearest grid value; ties go to the value with an even mantissa."""
    d = np.abs(grid - v)
    best = np.flatnonzero(d == d.min())
    if len(best) == 1:
        return grid[best[0]]
    return [grid[i] for i in best if mant_of(grid[i]) % 2 == 0][0]


def test_e4m3_grid_facts():
    grid = e4m3_values()
    assert grid.max() == 448.0
    assert grid[1] == 2.0 ** -9
    assert len(grid) == 127


def test_e4m3_page_thresholds():
    g = read_golden("e4m3_thresholds.txt")
    assert R.e4m3(np.float32(1.0)) == 1.0
    assert R.e4m3(np.float32(448.0)) == float(g["e4m3_max"])
    smallest = R.e4m3(np.float32(0.002))
    assert smallest == 2.0 ** -9                       # "about 0.002"
    assert abs(smallest - float(g["smallest_positive_approx"])) < 1e-4
    assert R.e4m3(np.float32(2.0 ** -10)) == 0.0       # half of it: tie -> even (0)
    assert R.e4m3(np.float32(0.00098)) == 2.0 ** -9    # just above half
    assert R.e4m3(np.float32(0.0009)) == 0.0           # below "about 0.001"
    assert abs(2.0 ** -10 - float(g["flush_below_approx"])) < 1e-4
    # x448 variant: the smallest p that survives is just above 2^-10 / 448
    thr = 2.0 ** -10 / 448
    assert thr < float(g["x448_threshold_max"])        # "a few per million"
    assert R.round_p(np.float32(thr * 1.01), 3) > 0
    assert R.round_p(np.float32(thr * 0.99), 3) == 0


def test_e4m3_brute_force_nearest():
    grid = e4m3_values()

    def mant(v):
        i = int(np.flatnonzero(grid == v)[0])
        return i  # grid index parity equals mantissa-field parity
    rng = np.random.default_rng(3)
    vs = np.concatenate([rng.uniform(0, 448, 3000), rng.uniform(0, 0.02, 2000),
                         grid, (grid[1:] + grid[:-1]) / 2]).astype(np.float32)
    got = R.e4m3(vs)
    for v, g in zip(vs, got):
        assert g == brute_nearest_even(float(v), grid, mant), v


def test_e4m3_matches_torch_float8():
    rng = np.random.default_rng(4)
    vs = np.concatenate([rng.uniform(0, 448, 20000), rng.uniform(0, 0.05, 20000),
                         np.exp(rng.uniform(-20, 0, 20000))]).astype(np.float32)
    ref = torch.from_numpy(vs).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(R.e4m3(vs), ref)


def test_bf16_matches_torch_and_bit_rounding():
    rng = np.random.default_rng(5)
    vs = np.concatenate([rng.uniform(0, 1, 20000), np.exp(rng.uniform(-100, 0, 20000)),
                         np.array([1e-40, 3e-39, 1.0, 0.0])]).astype(np.float32)
    ref = torch.from_numpy(vs).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(R.bf16(vs), ref)
    # round-to-nearest-even on the bit pattern
    u = vs.view(np.uint32).astype(np.uint64)
    rne = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    assert np.array_equal(R.bf16(vs), rne.view(np.float32).astype(np.float64))


def test_round_p_modes():
    p = np.float32([1.0, 0.5, 0.3, 1e-3, 1e-7, 0.0])
    assert np.array_equal(R.round_p(p, 0), p.astype(np.float64))
    for mode in range(4):
        assert R.round_p(np.float32(1.0), mode) == 1.0   # p = 1 is kept by all
        assert R.round_p(np.float32(0.0), mode) == 0.0
    # x448: scale, round, unscale
    x = np.float32(0.3)
    assert R.round_p(x, 3) == R.e4m3(np.float32(x * np.float32(448))) / 448
    # exact-mode variant divides in float32
    assert R.round_p_f32(x, 3) == np.float32(np.float32(R.e4m3(x * np.float32(448))) / np.float32(448))


# -- mode 4: e4m3(p * 256) / 256 ("注意力权重" section: the factor other fp8
#    attention kernels scale by) -------------------------------------------------

def test_x256_matches_plain_e4m3_where_scaling_commutes():
    # For p >= 2^-6 both p and 256 p lie in e4m3's normal range below 448,
    # where scaling by a power of two commutes with rounding.
    rng = np.random.default_rng(4)
    p = np.concatenate([rng.uniform(2.0 ** -6, 1.0, 20000), [2.0 ** -6, 0.5, 1.0]]).astype(np.float32)
    assert np.array_equal(R.round_p(p, 4), R.round_p(p, 2))


def test_x256_threshold_and_ties():
    # smallest nonzero result 2^-9 / 256 = 2^-17; half of it is a tie to 0
    tiny = np.float32(2.0 ** -17)
    assert R.round_p(np.array([tiny]), 4)[0] == 2.0 ** -17
    assert R.round_p(np.array([np.float32(2.0 ** -18)]), 4)[0] == 0.0
    assert R.round_p(np.array([np.float32(3 * 2.0 ** -19)]), 4)[0] == 2.0 ** -17
    # p = 1 and the largest values stay exact (256 < 448: no saturation)
    assert R.round_p(np.array([np.float32(1.0)]), 4)[0] == 1.0


def test_x256_brute_force_against_the_e4m3_value_set():
    # every e4m3 value (positive, finite) / 256 is a fixed point, and a
    # value between two neighbours goes to the nearer one
    # E4M3 from its definition: subnormals m * 2^-9 (m = 1..7), normals
    # (8 + m) * 2^(e - 3) for e = -6..8, m = 0..7, up to 448
    vals = {m * 2.0 ** -9 for m in range(1, 8)}
    vals |= {(8 + m) * 2.0 ** (e - 3) for e in range(-6, 9) for m in range(8)}
    grid = np.array(sorted(v for v in vals if v <= 448.0)) / 256.0
    assert len(grid) == 126
    assert np.array_equal(R.round_p(grid.astype(np.float32), 4), grid)
    mids = (grid[1:-1] + grid[2:]) / 2 * (1 + 1e-6)           # just above a midpoint
    out = R.round_p(mids.astype(np.float32), 4)
    assert np.array_equal(out, grid[2:])
    assert np.array_equal(R.round_p_f32(grid.astype(np.float32), 4).astype(np.float64), grid)


# ---- mode 5: e4m3 P straight into the tensor-core P.V ("注意力权重", closing
# question).  Its operand p~ * v_scale is rounded to the f16 significand.

def test_f16_significand_matches_numpy_float16_in_its_normal_range():
    # numpy's float32 -> float16 cast rounds to nearest-even: in f16's normal
    # range it is the same 11-significant-bit rounding.
    rng = np.random.default_rng(50)
    v = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-14, 15, 20000)).astype(np.float32)
    ties = np.float32(1.0) + np.float32(2.0 ** -11) * np.arange(1, 64, 2, dtype=np.float32)
    v = np.concatenate([v, ties])
    want = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(R.f16_significand(v), want)


def test_f16_significand_has_no_exponent_floor():
    # Below f16's normal range the kernel scales by a power of two first, so
    # the rounding keeps 11 significant bits: equal to the float16 cast of the
    # value moved into the normal range and moved back.
    rng = np.random.default_rng(51)
    v = np.ldexp(rng.uniform(1.0, 2.0, 5000), rng.integers(-60, -15, 5000)).astype(np.float32)
    e = np.frexp(v.astype(np.float64))[1]
    k = 1 - e                                    # v * 2^k in [1, 2)
    want = np.ldexp(np.ldexp(v.astype(np.float64), k).astype(np.float16).astype(np.float64), -k)
    assert np.array_equal(R.f16_significand(v), want)
    assert np.all(np.abs(R.f16_significand(v) / v - 1.0) <= 2.0 ** -11)


def test_pv_operand_rounds_only_in_the_direct_mode():
    rng = np.random.default_rng(52)
    p = R.e4m3(rng.uniform(0.0, 1.0, 4000).astype(np.float32)).astype(np.float32)
    vs = rng.uniform(0.001, 0.9, 4000).astype(np.float32)
    prod32 = np.multiply(p, vs, dtype=np.float32)
    assert np.array_equal(R.pv_operand(p, vs, R.DIRECT), R.f16_significand(prod32))
    for mode in (0, 1, 2, 3, 4):
        assert np.array_equal(R.pv_operand(p, vs, mode), p.astype(np.float64) * vs.astype(np.float64))
    # a product that 11 bits hold exactly is unchanged: e4m3 values (<= 4
    # significant bits) times powers of two
    pw = np.ldexp(1.0, rng.integers(-8, 3, 4000)).astype(np.float32)
    assert np.array_equal(R.pv_operand(p, pw, R.DIRECT), p.astype(np.float64) * pw)
    assert np.array_equal(R.round_p(p, R.DIRECT), R.round_p(p, 2))


def test_direct_mode_has_no_exact_form():
    with pytest.raises(ValueError):
        R.round_p_f32(np.ones(3, np.float32), R.DIRECT)
