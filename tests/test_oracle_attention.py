"""Pins for the oracle's QK scores and decode attention.

Each test checks the oracle against something other than itself: brute force
in exact integers or in 40-digit arithmetic on tiny inputs, closed forms
(one key, identical keys, zero query, a dominating key), invariants (convex
combination, column j == M=1 at ctx+j) and the page's rounding semantics.
"""

import math

import mpmath
import numpy as np
import pytest

from oracle import attention as A
from oracle import quant as Q
from oracle import rounding as R


def tiny_case(rng, B=2, M=2, Hq=4, Hkv=2, d=8, ctx=(5, 3), gap=2, scale=1.0):
    ctx = np.array(ctx, np.int32)
    row_start = np.zeros(B, np.int64)
    pos = 1
    for b in range(B):
        row_start[b] = pos
        pos += int(ctx[b]) + M - 1 + gap
    cap = pos
    q = (rng.standard_normal((B, M, Hq, d)) * scale).astype(np.float32)
    k = (rng.standard_normal((cap, Hkv, d)) * scale).astype(np.float32)
    v = rng.standard_normal((cap, Hkv, d)).astype(np.float32)
    k8, ks = Q.quantize_kv(k)
    v8, vs = Q.quantize_kv(v)
    return q, k8, ks, v8, vs, row_start, ctx


# ----------------------------------------------------------------- QK ----

def test_qk_brute_force_python_ints():
    rng = np.random.default_rng(11)
    q8 = rng.integers(-127, 128, (3, 16)).astype(np.int8)
    k8 = rng.integers(-127, 128, (5, 16)).astype(np.int8)
    S = A.qk_int(q8, k8)
    for r in range(3):
        for t in range(5):
            assert S[r, t] == sum(int(a) * int(b) for a, b in zip(q8[r], k8[t]))


def test_qk_extreme_value():
    a = np.full((1, 128), 127, np.int8)
    assert A.qk_int(a, a)[0, 0] == 2064512
    assert A.qk_int(a, -a)[0, 0] == -2064512
    assert 2064512 < 2 ** 24   # so float32(S) is exact


def test_qk_scores_layout_and_gqa():
    rng = np.random.default_rng(12)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng)
    S, q8, qs = A.qk_scores(q, k8, rs, ctx)
    B, M, Hq, d = q.shape
    g = Hq // k8.shape[0]
    for b in range(B):
        for j in range(M):
            L = ctx[b] + j
            for h in range(Hq):
                for t in range(S.shape[-1]):
                    if t >= L:
                        assert S[b, j, h, t] == A.NO_SCORE
                        continue
                    row = k8[h // g, rs[b] + t]
                    assert S[b, j, h, t] == sum(int(x) * int(y) for x, y in zip(q8[b, j, h], row))


def test_default_sm_scale():
    mpmath.mp.dps = 40
    s = A.default_sm_scale(128)
    assert s.dtype == np.float32
    exact = 1 / mpmath.sqrt(128)
    # correctly rounded: no other float32 is closer
    up, dn = np.nextafter(s, np.float32(1)), np.nextafter(s, np.float32(0))
    e = abs(mpmath.mpf(float(s)) - exact)
    assert e <= abs(mpmath.mpf(float(up)) - exact) and e <= abs(mpmath.mpf(float(dn)) - exact)


# ----------------------------------------------------- reference mode ----

def brute_softmax_mp(s, vdeq):
    """sum_t e^{s_t} v_t / sum_t e^{s_t} at 40 digits, no max shift."""
    mpmath.mp.dps = 40
    w = [mpmath.exp(mpmath.mpf(float(x))) for x in s]
    den = sum(w)
    return np.array([float(sum(wt * mpmath.mpf(float(vdeq[t, i])) for t, wt in enumerate(w)) / den)
                     for i in range(vdeq.shape[1])])


def test_reference_against_brute_force():
    rng = np.random.default_rng(13)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, scale=2.0)
    out = A.decode(q, k8, ks, v8, vs, rs, ctx, mode="reference")
    q8, qs = Q.quantize_rows(q)
    sm = A.default_sm_scale(q.shape[-1])
    B, M, Hq, d = q.shape
    g = Hq // k8.shape[0]
    for b in range(B):
        for j in range(M):
            L = int(ctx[b]) + j
            for h in range(Hq):
                kh = h // g
                rows = range(rs[b], rs[b] + L)
                s = []
                for r in rows:
                    Sv = sum(int(x) * int(y) for x, y in zip(q8[b, j, h], k8[kh, r]))
                    s.append(np.float32(np.float32(np.float32(Sv) * np.float32(qs[b, j, h] * ks[kh, r])) * sm))
                vdeq = np.array([[float(vs[kh, r]) * int(v8[kh, r, i]) for i in range(d)] for r in rows])
                ref = brute_softmax_mp(s, vdeq)
                np.testing.assert_allclose(out[b, j, h], ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("p_mode", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("mode", ["reference", "exact"])
def test_single_key_returns_dequantized_row(p_mode, mode):
    rng = np.random.default_rng(14)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=1, M=1, ctx=(1,))
    out = A.decode(q, k8, ks, v8, vs, rs, ctx, mode=mode, p_mode=p_mode)
    g = q.shape[2] // k8.shape[0]
    for h in range(q.shape[2]):
        r = rs[0]
        expect = np.multiply(v8[h // g, r].astype(np.float32), vs[h // g, r], dtype=np.float32)
        assert np.array_equal(out[0, 0, h].astype(np.float32), expect)


@pytest.mark.parametrize("mode", ["reference", "exact"])
def test_identical_keys_give_mean_of_values(mode):
    rng = np.random.default_rng(15)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=1, M=1, ctx=(6,))
    k8[:] = k8[:, :1]
    ks[:] = ks[:, :1]
    out = A.decode(q, k8, ks, v8, vs, rs, ctx, mode=mode)
    g = q.shape[2] // k8.shape[0]
    for h in range(q.shape[2]):
        rows = slice(rs[0], rs[0] + 6)
        mean = (vs[h // g, rows, None].astype(np.float64) * v8[h // g, rows]).mean(axis=0)
        tol = 1e-15 if mode == "reference" else 2e-6
        np.testing.assert_allclose(out[0, 0, h], mean, rtol=tol, atol=tol)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(16)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=1, M=1, ctx=(7,))
    q[:] = 0
    out = A.decode(q, k8, ks, v8, vs, rs, ctx)
    rows = slice(rs[0], rs[0] + 7)
    g = q.shape[2] // k8.shape[0]
    for h in range(q.shape[2]):
        mean = (vs[h // g, rows, None].astype(np.float64) * v8[h // g, rows]).mean(axis=0)
        np.testing.assert_allclose(out[0, 0, h], mean, rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("mode", ["reference", "exact"])
def test_convex_combination(mode):
    rng = np.random.default_rng(17)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, ctx=(9, 4), scale=3.0)
    out = A.decode(q, k8, ks, v8, vs, rs, ctx, mode=mode)
    B, M, Hq, d = q.shape
    g = Hq // k8.shape[0]
    for b in range(B):
        for j in range(M):
            L = int(ctx[b]) + j
            for h in range(Hq):
                rows = slice(rs[b], rs[b] + L)
                vd = vs[h // g, rows, None].astype(np.float64) * v8[h // g, rows]
                slack = 1e-6 * np.abs(vd).max()
                assert np.all(out[b, j, h] >= vd.min(axis=0) - slack)
                assert np.all(out[b, j, h] <= vd.max(axis=0) + slack)


@pytest.mark.parametrize("mode,p_mode", [("reference", 0), ("reference", 2), ("exact", 0), ("exact", 3)])
def test_column_j_equals_single_column_decode(mode, p_mode):
    rng = np.random.default_rng(18)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=2, M=3, ctx=(6, 9))
    full = A.decode(q, k8, ks, v8, vs, rs, ctx, mode=mode, p_mode=p_mode, C=4, Bk=2)
    for j in range(3):
        one = A.decode(q[:, j:j + 1], k8, ks, v8, vs, rs, ctx + j, mode=mode, p_mode=p_mode, C=4, Bk=2)
        assert np.array_equal(full[:, j:j + 1], one)


# -------------------------------------------------- rounding mirror ----

def test_mirror_with_identity_rounding_is_the_softmax():
    rng = np.random.default_rng(19)
    s = (rng.standard_normal(300) * 3).astype(np.float32)
    vdeq = rng.standard_normal((300, 8))
    ref = A.row_softmax_f64(s, vdeq)
    for C, Bk in ((512, 64), (64, 16), (7, 3), (300, 300)):
        got = A.row_online_mirrored(s, vdeq, 0, C, Bk)
        # only the float32 rounding of p separates the two
        np.testing.assert_allclose(got, ref, rtol=3e-7, atol=3e-7 * np.abs(vdeq).max())


@pytest.mark.parametrize("p_mode", [1, 2, 3])
def test_mirror_when_first_key_holds_the_max(p_mode):
    # With the row max in the first block the running max never changes, so
    # every p is exp(s - max) and the blockwise result is the direct formula
    # sum round_p(p) v / sum p.
    rng = np.random.default_rng(20)
    s = (rng.standard_normal(200) * 2).astype(np.float32)
    s[0] = s.max() + 1
    vdeq = rng.standard_normal((200, 8))
    p = np.exp(s.astype(np.float64) - float(s[0])).astype(np.float32)
    direct = (R.round_p(p, p_mode) @ vdeq) / p.astype(np.float64).sum()
    got = A.row_online_mirrored(s, vdeq, p_mode, 10 ** 9, 16)
    np.testing.assert_allclose(got, direct, rtol=1e-12, atol=1e-13)


def test_mirror_rounds_relative_to_the_running_max():
    # Two blocks; the second holds a larger score.  Block 1's weights are
    # rounded relative to block 1's own max, then rescaled.
    s = np.array([0.0, -8.0, 5.0, 4.0], np.float32)
    vdeq = np.eye(4)
    got = A.row_online_mirrored(s, vdeq, 2, 4, 2)
    m1, m2 = 0.0, 5.0
    p_blk1 = np.exp(s[:2].astype(np.float64) - m1).astype(np.float32)
    p_blk2 = np.exp(s[2:].astype(np.float64) - m2).astype(np.float32)
    a = math.exp(m1 - m2)
    o = np.concatenate([R.e4m3(p_blk1) * a, R.e4m3(p_blk2)])
    l = p_blk1.astype(np.float64).sum() * a + p_blk2.astype(np.float64).sum()
    np.testing.assert_allclose(got, o / l, rtol=1e-15)
    assert R.e4m3(p_blk1)[1] == 0.0     # exp(-8) ~ 3.4e-4 flushes to zero


# ---------------------------------------------------------- exact mode ----

def test_exact_mode_dominating_key_returns_its_row():
    rng = np.random.default_rng(21)
    d = 8
    s = np.array([[0.0, 200.0, 10.0, -5.0]], np.float32)   # gaps > 104
    v8 = rng.integers(-127, 128, (4, d)).astype(np.int8)
    vs = np.float32([0.5, 0.25, 2.0, 1.0])
    out = A.rows_exact_f32(s, v8, vs, 0)
    assert np.array_equal(out[0], np.multiply(v8[1].astype(np.float32), vs[1], dtype=np.float32))


def test_exact_mode_close_to_float64_reference():
    rng = np.random.default_rng(22)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=1, M=1, Hq=2, Hkv=1, d=16, ctx=(64,), scale=2.0)
    ex = A.decode(q, k8, ks, v8, vs, rs, ctx, mode="exact")
    ref = A.decode(q, k8, ks, v8, vs, rs, ctx, mode="reference")
    np.testing.assert_allclose(ex, ref, rtol=2e-5, atol=2e-6)


def test_exact_mode_is_sequential_float32():
    # Two keys worked by hand: every step a separate float32 rounding.
    s = np.array([[1.5, 0.25]], np.float32)
    v8 = np.array([[3, -7], [11, 5]], np.int8)
    vs = np.float32([0.1, 0.3])
    from oracle.expf_tang import expf_tang
    f = np.float32
    vd0 = f(f(3) * vs[0]), f(f(-7) * vs[0])
    vd1 = f(f(11) * vs[1]), f(f(5) * vs[1])
    # t = 0: m = 1.5, a = 0, p = 1
    l = f(1.0)
    o = [f(f(1.0) * vd0[0]), f(f(1.0) * vd0[1])]
    # t = 1: m stays 1.5
    a = expf_tang(f(0.0))
    p = expf_tang(f(f(0.25) - f(1.5)))
    l = f(f(l * a) + p)
    o = [f(f(o[i] * a) + f(p * vd1[i])) for i in range(2)]
    expect = np.array([f(o[0] / l), f(o[1] / l)], np.float32)
    assert np.array_equal(A.rows_exact_f32(s, v8, vs, 0)[0], expect)


# ---- mode 5: e4m3 P into the tensor-core P.V, operand p~ * vs rounded to the
# f16 significand.

def test_direct_mode_single_key_returns_the_rounded_scale_times_v8():
    # One key: p = 1, p~ = 1, the operand is f16_significand(vs), l = 1.
    rng = np.random.default_rng(60)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=1, M=1, ctx=(1,))
    out = A.decode(q, k8, ks, v8, vs, rs, ctx, p_mode=R.DIRECT)
    g = q.shape[2] // k8.shape[0]
    for h in range(q.shape[2]):
        r = rs[0]
        expect = R.f16_significand(np.float32(vs[h // g, r])) * v8[h // g, r].astype(np.float64)
        assert np.array_equal(out[0, 0, h], expect)


def test_direct_mode_equals_e4m3_when_every_scale_is_a_power_of_two():
    # e4m3 values have at most 4 significant bits, so p~ * 2^k is exact in 11
    # bits and mode 5 computes what mode 2 computes, bit for bit.
    rng = np.random.default_rng(61)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=2, M=2, ctx=(150, 70), d=16)
    vs = np.ldexp(1.0, rng.integers(-9, -2, vs.shape)).astype(np.float32)
    a = A.decode(q, k8, ks, v8, vs, rs, ctx, p_mode=R.DIRECT, C=64, Bk=16)
    b = A.decode(q, k8, ks, v8, vs, rs, ctx, p_mode=2, C=64, Bk=16)
    assert np.array_equal(a, b)


def test_direct_mode_stays_within_the_f16_rounding_of_e4m3():
    # Each PV term moves by at most 2^-11 relative, the row sum not at all.
    rng = np.random.default_rng(62)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=2, M=2, ctx=(300, 120), d=16, scale=2.0)
    a = A.decode(q, k8, ks, v8, vs, rs, ctx, p_mode=R.DIRECT, C=64, Bk=16)
    b = A.decode(q, k8, ks, v8, vs, rs, ctx, p_mode=2, C=64, Bk=16)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 0.0 < rel <= 2.0 ** -11


def test_direct_mode_has_no_exact_scan():
    rng = np.random.default_rng(63)
    q, k8, ks, v8, vs, rs, ctx = tiny_case(rng, B=1, M=1, ctx=(4,))
    with pytest.raises(ValueError):
        A.decode(q, k8, ks, v8, vs, rs, ctx, p_mode=R.DIRECT, mode="exact")
