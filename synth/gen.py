"""Seeded generators (see the package docstring for layouts).

Host generation uses numpy's PCG64.  Large workloads (gigabytes of float32
K/V) can instead be drawn on a CUDA device with torch's Philox generator;
the tests then copy the float32 rows of the sequences they check back to
the host, so every value the oracle sees is a generator output.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD_DIM = 128
OUTLIER_CHANNELS = 4
OUTLIER_GAIN = 20.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-attention workload shape.

    ctx is either a fixed context length or a (kind, lo, hi) triple:
    ("uniform", lo, hi) draws integers uniformly in [lo, hi];
    ("loguniform", lo, hi) draws floor(exp(U(ln lo, ln hi))).
    ctx counts the keys column 0 attends to; column j attends to ctx + j.
    """

    name: str
    B: int
    M: int
    Hq: int
    Hkv: int
    ctx: object
    outliers: bool
    d: int = HEAD_DIM
    index: int = 0  # seed base: seed = index * 1000 + rep

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv


def _w(name, index, B, M, Hq, Hkv, ctx, outliers):
    return Workload(name=name, B=B, M=M, Hq=Hq, Hkv=Hkv, ctx=ctx,
                    outliers=outliers, index=index)


# The five workload families; sizes are those the decode path is specified on.
WORKLOADS = {
    # tiny single decode: GQA 4, ctx 256, no outliers
    "tiny": _w("tiny", 0, 1, 1, 8, 2, 256, False),
    # one Qwen3-30B-A3B attention layer at ctx 1024 with outlier channels
    "qwen_layer": _w("qwen_layer", 1, 1, 1, 32, 4, 1024, True),
    # speculative batch verify: 16 sequences x 5 draft columns
    "spec_verify": _w("spec_verify", 2, 16, 5, 32, 4, ("uniform", 1024, 4096), True),
    # long-context P-precision sweep
    "long_8k": _w("long_8k", 3, 4, 1, 32, 4, 8192, True),
    "long_32k": _w("long_32k", 3, 4, 1, 32, 4, 32768, True),
    "long_128k": _w("long_128k", 3, 4, 1, 32, 4, 131072, True),
    # serving sweep: ragged batches, log-uniform contexts
    "serving_b64_m1": _w("serving_b64_m1", 4, 64, 1, 32, 4, ("loguniform", 512, 32768), False),
    "serving_b128_m1": _w("serving_b128_m1", 4, 128, 1, 32, 4, ("loguniform", 512, 32768), False),
    "serving_b256_m1": _w("serving_b256_m1", 4, 256, 1, 32, 4, ("loguniform", 512, 32768), False),
    "serving_b64_m4": _w("serving_b64_m4", 4, 64, 4, 32, 4, ("loguniform", 512, 32768), False),
    "serving_b128_m4": _w("serving_b128_m4", 4, 128, 4, 32, 4, ("loguniform", 512, 32768), False),
    "serving_b256_m4": _w("serving_b256_m4", 4, 256, 4, 32, 4, ("loguniform", 512, 32768), False),
}


def make_lengths(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    """Per-sequence context lengths (int32, >= 1)."""
    if isinstance(wl.ctx, int):
        return np.full(wl.B, wl.ctx, dtype=np.int32)
    kind, lo, hi = wl.ctx
    if kind == "uniform":
        return rng.integers(lo, hi, size=wl.B, endpoint=True).astype(np.int32)
    if kind == "loguniform":
        u = rng.uniform(math.log(lo), math.log(hi), size=wl.B)
        return np.clip(np.floor(np.exp(u)), lo, hi).astype(np.int32)
    raise ValueError(f"unknown ctx kind {kind!r}")


def outlier_channels(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    """[Hkv][4] distinct channel indices per KV head (empty if no outliers)."""
    if not wl.outliers:
        return np.zeros((wl.Hkv, 0), dtype=np.int64)
    return np.stack([rng.choice(wl.d, size=OUTLIER_CHANNELS, replace=False)
                     for _ in range(wl.Hkv)]).astype(np.int64)


@dataclasses.dataclass
class Inputs:
    """A generated workload instance (host arrays unless stated)."""

    wl: Workload
    seed: int
    ctx: np.ndarray        # int32 [B]
    row_start: np.ndarray  # int64 [B]
    cap_rows: int
    channels: np.ndarray   # int64 [Hkv][n_outlier]
    q: object              # float32 [B][M][Hq][d]  (numpy or torch)
    k_rows: object         # float32 [cap_rows][Hkv][d]
    v_rows: object         # float32 [cap_rows][Hkv][d]

    @property
    def max_ctx(self) -> int:
        return int(self.ctx.max())

    def rows_of(self, b: int) -> tuple:
        """Row range [lo, hi) of sequence b in the cache (ctx + M - 1 rows)."""
        lo = int(self.row_start[b])
        return lo, lo + int(self.ctx[b]) + self.wl.M - 1


def _layout(wl: Workload, ctx: np.ndarray, rng: np.random.Generator):
    """Pack sequences one after another with 0-3 unused rows between them,
    so sequence starts land on arbitrary (odd, unaligned) row indices."""
    gaps = rng.integers(0, 4, size=wl.B)
    row_start = np.zeros(wl.B, dtype=np.int64)
    pos = 0
    for b in range(wl.B):
        pos += int(gaps[b])
        row_start[b] = pos
        pos += int(ctx[b]) + wl.M - 1
    return row_start, pos + int(rng.integers(0, 4))


def make_workload(wl: Workload, rep: int = 0, device: Optional[str] = None,
                  ctx_override: Optional[np.ndarray] = None) -> Inputs:
    """Draw one instance of a workload.

    device=None draws everything on the host with numpy PCG64.  device="cuda"
    draws the (large) K/V rows and Q on that device with torch's generator
    seeded from the same seed; lengths, layout and outlier channels always
    come from numpy so they are identical on both routes.
    """
    seed = wl.index * 1000 + rep
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = make_lengths(wl, rng) if ctx_override is None else np.asarray(ctx_override, np.int32)
    row_start, cap = _layout(wl, ctx, rng)
    ch = outlier_channels(wl, rng)
    gain = np.ones((wl.Hkv, wl.d), dtype=np.float32)
    for h in range(wl.Hkv):
        gain[h, ch[h]] = OUTLIER_GAIN
    qgain = np.repeat(gain, wl.g, axis=0)  # q head h uses kv head h // g

    if device is None:
        q = rng.standard_normal((wl.B, wl.M, wl.Hq, wl.d), dtype=np.float32) * qgain
        k = rng.standard_normal((cap, wl.Hkv, wl.d), dtype=np.float32) * gain
        v = rng.standard_normal((cap, wl.Hkv, wl.d), dtype=np.float32) * gain
        q, k, v = (np.ascontiguousarray(a, dtype=np.float32) for a in (q, k, v))
    else:
        import torch
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        tg = torch.from_numpy(gain).to(device)
        tq = torch.from_numpy(qgain).to(device)
        q = torch.randn((wl.B, wl.M, wl.Hq, wl.d), generator=gen, device=device) * tq
        k = torch.empty((cap, wl.Hkv, wl.d), device=device, dtype=torch.float32)
        v = torch.empty_like(k)
        step = 1 << 18  # rows per chunk keeps the temporaries small
        for r0 in range(0, cap, step):
            r1 = min(cap, r0 + step)
            k[r0:r1] = torch.randn((r1 - r0, wl.Hkv, wl.d), generator=gen, device=device) * tg
            v[r0:r1] = torch.randn((r1 - r0, wl.Hkv, wl.d), generator=gen, device=device) * tg
    return Inputs(wl=wl, seed=seed, ctx=ctx, row_start=row_start, cap_rows=int(cap),
                  channels=ch, q=q, k_rows=k, v_rows=v)
