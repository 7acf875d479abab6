"""Per-row int8 quantization (oracle).

The pages use int8 K/V rows with one float scale per row ("Kestrel_VLLM - 18",
§四 lists the per-layer fields _k _ks _v _vs) and an int8 query with a
per-head scale (§3.3).  They do not print the formula; the reading used here
is the plain absmax one:

    scale = f32(max_i |x_i|) / 127            (IEEE float32 division)
    q_i   = clamp(rint_half_even(x_i / scale), -127, 127)
    scale == 0 (all-zero row)  =>  q = 0

Every operation is a single float32 rounding (numpy float32 ufuncs).
Inputs must be finite.
"""

from __future__ import annotations

import numpy as np


def quantize_rows(x) -> tuple:
    """Quantize the last axis of ``x``.

    Returns (q int8 with x's shape, scale float32 with x.shape[:-1]).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)                      # exact
    scale = np.divide(amax, np.float32(127.0), dtype=np.float32)
    zero = scale == 0
    safe = np.where(zero, np.float32(1.0), scale).astype(np.float32)
    ratio = np.divide(x, safe[..., None], dtype=np.float32)  # one f32 rounding
    q = np.clip(np.rint(ratio), -127, 127)                 # ties to even
    q = np.where(zero[..., None], 0, q)
    return q.astype(np.int8), scale.astype(np.float32)


def quantize_kv(rows) -> tuple:
    """K or V rows in arrival layout [n_rows][Hkv][d] -> cache layout.

    Returns (q int8 [Hkv][n_rows][d], scale float32 [Hkv][n_rows]).
    """
    q, s = quantize_rows(rows)
    return np.ascontiguousarray(q.transpose(1, 0, 2)), np.ascontiguousarray(s.T)


def quantize_queries(q) -> tuple:
    """Queries [B][M][Hq][d] -> (int8 [B][M][Hq][d], scale float32 [B][M][Hq])."""
    return quantize_rows(q)
