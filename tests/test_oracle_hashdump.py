"""Pins of the oracle's FNV-1a 64 row hashes ("Kestrel_VLLM - 18" §3.4).

The definition is pinned by published FNV-1a 64 test vectors; the
vectorised row hashing by the one-byte-at-a-time definition.
"""

import numpy as np

from oracle import hashdump as H


def test_published_fnv1a64_vectors():
    assert H.fnv1a64(b"") == 0xCBF29CE484222325          # the offset basis
    assert H.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert H.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_page_basis_is_a_truncation_of_the_published_one():
    # the page's 1469598103934665603 lost the last digit of the basis
    assert H.FNV_OFFSET == 14695981039346656037 == 0xCBF29CE484222325
    assert H.FNV_OFFSET // 10 == 1469598103934665603


def test_vectorised_rows_equal_the_definition():
    rng = np.random.default_rng(5)
    for shape, dt in (((7, 33), np.uint8), ((5, 128), np.float32), ((3, 4, 9), np.int32)):
        a = (rng.standard_normal(shape) * 100).astype(dt)
        got = H.hash_rows(a)
        rows = a.reshape(-1, shape[-1])
        assert [int(x) for x in got] == [H.fnv1a64(r.tobytes()) for r in rows]


def test_first_divergence_finds_the_first_changed_row():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((50, 16)).astype(np.float32)
    b = a.copy()
    assert H.first_divergence(H.hash_rows(a), H.hash_rows(b)) is None
    b[31, 7] = np.nextafter(b[31, 7], np.float32(np.inf))   # one ulp in one row
    b[40, 0] += 1
    assert H.first_divergence(H.hash_rows(a), H.hash_rows(b)) == 31
