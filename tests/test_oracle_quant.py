"""Pins for the oracle's absmax/127 int8 quantization."""

import numpy as np

from oracle import quant as Q


def test_absmax_element_maps_to_127():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((500, 128)).astype(np.float32) * 3
    q, s = Q.quantize_rows(x)
    i = np.argmax(np.abs(x), axis=1)
    rows = np.arange(len(x))
    assert np.array_equal(np.abs(q[rows, i]), np.full(len(x), 127))
    assert np.array_equal(np.sign(q[rows, i]), np.sign(x[rows, i]).astype(np.int8))


def test_error_within_half_step():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((300, 128)).astype(np.float32)
    x[:, :4] *= 20
    q, s = Q.quantize_rows(x)
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * s[:, None])
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))


def test_zero_row_and_scale_definition():
    x = np.zeros((3, 128), np.float32)
    x[1, 5] = -2.5
    q, s = Q.quantize_rows(x)
    assert s[0] == 0 and not q[0].any()
    assert s[1] == np.float32(np.float32(2.5) / np.float32(127))
    assert q[1, 5] == -127 and np.count_nonzero(q[1]) == 1


def test_ties_round_to_even():
    # amax = 127 gives scale exactly 1, so x / scale = x exactly.
    x = np.zeros((1, 128), np.float32)
    x[0, :8] = [127, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5]
    q, s = Q.quantize_rows(x)
    assert s[0] == 1.0
    assert list(q[0, :8]) == [127, 2, 4, -2, -4, 0, 2, 0]


def test_kv_layout():
    rng = np.random.default_rng(3)
    rows = rng.standard_normal((7, 3, 128)).astype(np.float32)
    qk, sk = Q.quantize_kv(rows)
    assert qk.shape == (3, 7, 128) and sk.shape == (3, 7)
    q2, s2 = Q.quantize_rows(rows[4, 2])
    assert np.array_equal(qk[2, 4], q2) and sk[2, 4] == s2
