"""Shared helpers for the GPU parity tests (inputs come from ``synth``; the
expected values come from ``oracle``; the CUDA path is reached only through
the C ABI binding ``int8_kv_decode_gb300``)."""

from __future__ import annotations

import dataclasses

import numpy as np

import oracle
from synth import Workload, make_workload

F32_MAX_ABS = 1e-4      # fast mode, f32 P: max |delta|
F32_REL_L2 = 1e-5       # fast mode, f32 P: relative L2
ROUNDED_REL_L2 = 2e-3   # rounded-P modes against the oracle with the same rounding

# The rounding points of the rounded-P modes: spans of C = 128 keys at fixed
# positions, online-softmax blocks of Bk = 32 keys.  The oracle mirrors them
# from these constants; the library must report the same tiling, so a change
# to the kernels' tiling fails the tests instead of being followed silently.
SPAN_C = 128
BLOCK_BK = 32


def pinned_tiling():
    """(C, Bk) for the oracle's rounded-P mirror, after checking that the
    library under test reports exactly that tiling."""
    import int8_kv_decode_gb300 as K
    assert K.get_tiling() == (SPAN_C, BLOCK_BK), K.get_tiling()
    return SPAN_C, BLOCK_BK


@dataclasses.dataclass
class GpuCase:
    x: object            # synth Inputs (host arrays)
    k8: object           # torch int8 [Hkv][cap][d] on the device
    v8: object
    ks: object
    vs: object
    q: object
    rs: object
    ctx: object
    ok8: np.ndarray      # oracle's quantized cache (host)
    oks: np.ndarray
    ov8: np.ndarray
    ovs: np.ndarray


def custom(name, B, M, Hq, Hkv, ctx, outliers=True, index=9):
    return Workload(name=name, B=B, M=M, Hq=Hq, Hkv=Hkv, ctx=ctx, outliers=outliers, index=index)


def upload(wl, rep=0, ctx_override=None, device="cuda"):
    """Host-generated workload, quantized on the GPU and by the oracle."""
    import torch
    import int8_kv_decode_gb300 as K
    x = make_workload(wl, rep=rep, ctx_override=ctx_override)
    dev = torch.device(device)
    k8 = torch.empty((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device=dev)
    v8 = torch.empty_like(k8)
    ks = torch.empty((wl.Hkv, x.cap_rows), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    K.quantize_kv(torch.from_numpy(x.k_rows).to(dev), k8, ks)
    K.quantize_kv(torch.from_numpy(x.v_rows).to(dev), v8, vs)
    ok8, oks = oracle.quant.quantize_kv(x.k_rows)
    ov8, ovs = oracle.quant.quantize_kv(x.v_rows)
    return GpuCase(x=x, k8=k8, v8=v8, ks=ks, vs=vs, q=torch.from_numpy(x.q).to(dev),
                   rs=torch.from_numpy(x.row_start).to(dev),
                   ctx=torch.from_numpy(x.ctx).to(dev), ok8=ok8, oks=oks, ov8=ov8, ovs=ovs)


def device_upload(wl, rep=0):
    """A workload drawn and quantized on the GPU (large shapes), as a GpuCase
    without the oracle's caches (ok8 .. ovs are None)."""
    import torch
    import int8_kv_decode_gb300 as K
    x = make_workload(wl, rep=rep, device="cuda")
    k8 = torch.empty((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty((wl.Hkv, x.cap_rows), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    K.quantize_kv(x.k_rows, k8, ks)
    K.quantize_kv(x.v_rows, v8, vs)
    x.k_rows = x.v_rows = None
    return GpuCase(x=x, k8=k8, v8=v8, ks=ks, vs=vs, q=x.q,
                   rs=torch.from_numpy(x.row_start).cuda(), ctx=torch.from_numpy(x.ctx).cuda(),
                   ok8=None, oks=None, ov8=None, ovs=None)


def run(c: GpuCase, **kw):
    import int8_kv_decode_gb300 as K
    return K.decode(c.q, c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx, c.x.max_ctx, **kw)


def oracle_decode(c: GpuCase, **kw):
    x = c.x
    return oracle.attention.decode(x.q, c.ok8, c.oks, c.ov8, c.ovs, x.row_start, x.ctx, **kw)


def assert_f32_tolerance(got, ref, mask=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= F32_MAX_ABS and rel <= F32_REL_L2, (err, rel)
    return err, rel


def rel_l2(got, ref, mask=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def sample_rows(x, n, seed=0):
    """n distinct (b, j, h) rows, always including the first and last."""
    rng = np.random.default_rng(seed)
    B, M, Hq = x.wl.B, x.wl.M, x.wl.Hq
    rows = {(0, 0, 0), (B - 1, M - 1, Hq - 1)}
    while len(rows) < min(n, B * M * Hq):
        rows.add((int(rng.integers(B)), int(rng.integers(M)), int(rng.integers(Hq))))
    return sorted(rows)


def row_mask(shape, rows):
    m = np.zeros(shape[:3], dtype=bool)
    for (b, j, h) in rows:
        m[b, j, h] = True
    return m


def bits(a):
    """float32 array as its uint32 bit patterns (byte-for-byte comparisons)."""
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32)


def device_case(name, rep=0):
    """A full-size workload drawn on the GPU and quantized there:
    (inputs, k8, ks, v8, vs, row_start, ctx) with the caches and the two
    index arrays on the device."""
    import torch
    import int8_kv_decode_gb300 as K
    from synth import WORKLOADS
    wl = WORKLOADS[name]
    x = make_workload(wl, rep=rep, device="cuda")
    k8 = torch.empty((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty((wl.Hkv, x.cap_rows), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    K.quantize_kv(x.k_rows, k8, ks)
    K.quantize_kv(x.v_rows, v8, vs)
    rs = torch.from_numpy(x.row_start).cuda()
    ctx = torch.from_numpy(x.ctx).cuda()
    return x, k8, ks, v8, vs, rs, ctx


def oracle_sequence_cache(x, b, k8=None, ks=None, v8=None, vs=None):
    """The oracle's own quantized cache of sequence b of a device-drawn
    workload, from the generator's float32 rows (copied to the host).  When
    the device caches are given, their bytes for the sequence must equal the
    oracle's (quantization parity)."""
    lo, hi = x.rows_of(b)
    ok8, oks = oracle.quant.quantize_kv(x.k_rows[lo:hi].cpu().numpy())
    ov8, ovs = oracle.quant.quantize_kv(x.v_rows[lo:hi].cpu().numpy())
    if k8 is not None:
        assert np.array_equal(k8[:, lo:hi].cpu().numpy(), ok8)
        assert np.array_equal(bits(ks[:, lo:hi].cpu().numpy()), bits(oks))
        assert np.array_equal(v8[:, lo:hi].cpu().numpy(), ov8)
        assert np.array_equal(bits(vs[:, lo:hi].cpu().numpy()), bits(ovs))
    return ok8, oks, ov8, ovs


def oracle_sequence_rows(x, b, cache, rows, **kw):
    """Oracle outputs of sequence b alone (its cache from oracle_sequence_cache)
    for the (j, h) pairs in rows: an array [M][Hq][d], NaN elsewhere."""
    q = x.q[b:b + 1]
    q = q.cpu().numpy() if hasattr(q, "cpu") else np.asarray(q)
    ok8, oks, ov8, ovs = cache
    out = oracle.attention.decode(q, ok8, oks, ov8, ovs, np.array([0]), x.ctx[b:b + 1],
                                  rows=[(0, j, h) for (j, h) in rows], **kw)
    return out[0]
