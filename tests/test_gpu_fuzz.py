"""Seeded random shapes through the whole fast path, each checked three ways.

Every case draws a batch size, draft columns M, GQA group g, kv heads, a
context mix (1 key up to several windows, ragged), outlier channels, a P
mode, and the cache layout (contiguous or paged with random page order).
Checks:

- sampled rows against the oracle: f32 P within the fast-mode tolerance,
  rounded P within the rounded-mode bound of the same-rounding oracle;
- draft column j equals, byte for byte, an M = 1 decode at ctx + j
  ("Kestrel_VLLM - 18", §二);
- a sub-batch decoded alone equals, byte for byte, its rows in the whole batch;
- the device error word stays clear;
- every third case with contexts up to 3000 (and a P mode with an exact form):
  exact mode equals the oracle's float32 emulation, byte for byte, on sampled
  rows.

The P mode is drawn over all six, e4m3 fed straight to the P.V MMA included.

("海光 DCU 实测" §4: one shape being right proves nothing about the others.)
"""

import numpy as np
import pytest

from helpers import (ROUNDED_REL_L2, assert_f32_tolerance, custom, oracle_decode,
                     pinned_tiling, rel_l2, row_mask, sample_rows, upload)
from synth.paging import page_layout, paged_copy

pytestmark = pytest.mark.gpu

N_CASES = 48


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def bits(a):
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32)


def draw_case(i):
    rng = np.random.default_rng(7000 + i)
    while True:
        g = int(rng.choice([1, 2, 4, 8]))
        M = int(rng.integers(1, 9))
        if g * M <= 64:
            break
    Hkv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 24))
    kind = rng.integers(0, 3)
    if kind == 0:
        ctx = rng.integers(1, 200, B)                             # within one window
    elif kind == 1:
        ctx = rng.integers(1, 3000, B)                            # a few windows
    else:
        ctx = np.exp(rng.uniform(0, np.log(6000), B)).astype(np.int64) + 1   # ragged, long
    return dict(B=B, M=M, g=g, Hkv=Hkv, ctx=ctx.astype(np.int32), p_mode=int(rng.integers(0, 6)),
                outliers=bool(rng.integers(0, 2)), page=int(rng.choice([0, 32, 64, 128])),
                seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i):
    import torch
    import int8_kv_decode_gb300 as K
    d = draw_case(i)
    B, M, g, Hkv = d["B"], d["M"], d["g"], d["Hkv"]
    Hq = g * Hkv
    wl = custom(f"fuzz{i}", B, M, Hq, Hkv, ("uniform", 1, 2), outliers=d["outliers"],
                index=30 + i)
    c = upload(wl, ctx_override=d["ctx"])
    max_ctx = c.x.max_ctx
    ws = K.alloc_workspace(B, M, Hq, max_ctx)

    if d["page"]:
        L = page_layout(c.x.ctx, c.x.row_start, M, d["page"], seed=d["seed"] % 1000)
        kp, ksp, vp, vsp = paged_copy(L, c.k8, c.ks, c.v8, c.vs, seed=d["seed"] % 997)
        bt = torch.from_numpy(L.block_table).cuda()

        def dec(q, sel, ctx, mc, p_mode):
            return K.decode_paged(q, kp, ksp, vp, vsp, bt[sel].contiguous(), d["page"], ctx, mc,
                                  p_mode=p_mode, workspace=K.alloc_workspace(
                                      q.shape[0], q.shape[1], Hq, mc))
    else:
        def dec(q, sel, ctx, mc, p_mode):
            return K.decode(q, c.k8, c.ks, c.v8, c.vs, c.rs[sel].contiguous(), ctx, mc,
                            p_mode=p_mode, workspace=K.alloc_workspace(
                                q.shape[0], q.shape[1], Hq, mc))

    every = torch.arange(B, device="cuda")
    if d["page"]:
        full = K.decode_paged(c.q, kp, ksp, vp, vsp, bt, d["page"], c.ctx, max_ctx,
                              p_mode=d["p_mode"], workspace=ws).cpu().numpy()
    else:
        full = K.decode(c.q, c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx, max_ctx, p_mode=d["p_mode"],
                        workspace=ws).cpu().numpy()
    assert K.get_device_status(ws) == 0
    assert np.isfinite(full).all()

    # 1. sampled rows against the oracle
    rows = sample_rows(c.x, 12, seed=i)
    C, Bk = pinned_tiling()
    ref = oracle_decode(c, rows=rows, p_mode=d["p_mode"], C=C, Bk=Bk)
    m = row_mask(full.shape, rows)
    if d["p_mode"] == 0:
        assert_f32_tolerance(full[m], ref[m])
    else:
        assert rel_l2(full[m], ref[m]) <= ROUNDED_REL_L2

    # 2. column j against an M = 1 decode at ctx + j
    j = int(np.random.default_rng(i).integers(0, M))
    one = dec(c.q[:, j:j + 1].contiguous(), every, (c.ctx + j).contiguous(), max_ctx + j,
              d["p_mode"]).cpu().numpy()
    assert np.array_equal(bits(full[:, j:j + 1]), bits(one)), j

    # 3. a sub-batch alone
    lo = int(np.random.default_rng(i + 1).integers(0, B))
    hi = min(B, lo + 3)
    sel = torch.arange(lo, hi, device="cuda")
    sub = dec(c.q[lo:hi].contiguous(), sel, c.ctx[lo:hi].contiguous(),
              int(c.x.ctx[lo:hi].max()), d["p_mode"]).cpu().numpy()
    assert np.array_equal(bits(full[lo:hi]), bits(sub)), (lo, hi)

    # 4. exact mode on sampled rows (p_mode 5 has no exact form)
    if i % 3 == 0 and int(c.x.ctx.max()) <= 3000 and d["p_mode"] != 5:
        if d["page"]:
            ex = K.decode_paged(c.q, kp, ksp, vp, vsp, bt, d["page"], c.ctx, max_ctx,
                                p_mode=d["p_mode"], exact_mode=True).cpu().numpy()
        else:
            ex = K.decode(c.q, c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx, max_ctx, p_mode=d["p_mode"],
                          exact_mode=True).cpu().numpy()
        xr = sample_rows(c.x, 6, seed=100 + i)
        ref = oracle_decode(c, rows=xr, p_mode=d["p_mode"], mode="exact")
        mk = row_mask(ex.shape, xr)
        assert np.array_equal(bits(ex[mk]), bits(ref[mk]))
