"""FNV-1a 64 row hashes for parity dumps (oracle side; test infrastructure).

"Kestrel_VLLM - 18" §3.4 compares two runs by hashing the same buffers on
both sides with the same FNV-1a 64 and looking for the first tag whose
hashes differ.  Here a buffer is hashed row by row, so the first differing
row localises a divergence inside it.

FNV-1a 64: h = offset basis; for each byte b in order: h = (h XOR b) * prime
(mod 2^64), with offset basis 14695981039346656037 and prime 1099511628211.
The page prints the basis as 1469598103934665603, a truncation of it
(one digit lost in extraction); the published value is used here.
"""

from __future__ import annotations

import numpy as np

FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211
_MASK = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """The definition, one byte at a time in Python integers."""
    h = FNV_OFFSET
    for b in data:
        h = ((h ^ b) * FNV_PRIME) & _MASK
    return h


def hash_rows(a) -> np.ndarray:
    """FNV-1a 64 of every row of a (rows = all leading indices, bytes of the
    last dimension in memory order).  Returns uint64 [rows]."""
    a = np.ascontiguousarray(a)
    rows = a.reshape(-1, a.shape[-1]) if a.ndim > 1 else a.reshape(1, -1)
    b = rows.view(np.uint8).reshape(rows.shape[0], -1)
    h = np.full(b.shape[0], FNV_OFFSET, dtype=np.uint64)
    prime = np.uint64(FNV_PRIME)
    with np.errstate(over="ignore"):
        for j in range(b.shape[1]):               # uint64 arithmetic wraps mod 2^64
            h = (h ^ b[:, j].astype(np.uint64)) * prime
    return h


def first_divergence(a_hashes, b_hashes):
    """Index of the first row whose hashes differ, or None."""
    a = np.asarray(a_hashes, dtype=np.uint64).ravel()
    b = np.asarray(b_hashes, dtype=np.uint64).ravel()
    if a.shape != b.shape:
        raise ValueError("hash lists of different lengths")
    d = np.nonzero(a != b)[0]
    return int(d[0]) if d.size else None
