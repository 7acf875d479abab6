"""Paged KV (kattn_decode_paged) on the GPU.

A paged cache holds the same rows as a contiguous one, at the same key
positions of the fixed tiling, so the decode must return the same bytes:
the fast path against kattn_decode on the contiguous cache (itself held to
the oracle by test_gpu_parity.py), exact mode against the oracle directly.
Pages are shuffled over the pool, the unused rows hold random bytes and the
unused table entries are -1, so a read of anything else shows up.
"""

import numpy as np
import pytest

from helpers import custom, device_upload, oracle_decode, run, upload
from synth import WORKLOADS, make_workload
from synth.paging import page_layout, paged_copy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def bits(a):
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32)


class Paged:
    def __init__(self, c, P, seed=0):
        import torch
        x = c.x
        self.layout = page_layout(x.ctx, x.row_start, x.wl.M, P, seed=seed)
        self.k8, self.ks, self.v8, self.vs = paged_copy(self.layout, c.k8, c.ks, c.v8, c.vs,
                                                        seed=seed)
        self.bt = torch.from_numpy(self.layout.block_table).to(c.k8.device)
        self.P = P

    def decode(self, c, bt=None, ctx=None, **kw):
        import int8_kv_decode_gb300 as K
        return K.decode_paged(c.q, self.k8, self.ks, self.v8, self.vs,
                              self.bt if bt is None else bt, self.P,
                              c.ctx if ctx is None else ctx, c.x.max_ctx, **kw)


@pytest.mark.parametrize("p_mode", [0, 2, 3])
@pytest.mark.parametrize("name,P", [("tiny", 32), ("qwen_layer", 128), ("spec_verify", 32),
                                    ("spec_verify", 256)])
def test_paged_equals_contiguous_bytes(name, P, p_mode):
    import int8_kv_decode_gb300 as K
    c = upload(WORKLOADS[name])
    ref = run(c, p_mode=p_mode).cpu().numpy()
    pc = Paged(c, P, seed=P + p_mode)
    wl = c.x.wl
    ws = K.alloc_workspace(wl.B, wl.M, wl.Hq, c.x.max_ctx)
    got = pc.decode(c, p_mode=p_mode, workspace=ws).cpu().numpy()
    assert np.array_equal(bits(got), bits(ref))
    assert K.get_device_status(ws) == 0          # no -1 entry or spare page was read


@pytest.mark.parametrize("name,P,p_mode", [("tiny", 32, 0), ("tiny", 64, 2), ("qwen_layer", 128, 0),
                                           ("qwen_layer", 32, 3)])
def test_paged_exact_mode_bit_exact(name, P, p_mode):
    c = upload(WORKLOADS[name])
    got = Paged(c, P, seed=7).decode(c, p_mode=p_mode, exact_mode=True).cpu().numpy()
    ref = oracle_decode(c, mode="exact", p_mode=p_mode)
    assert np.array_equal(bits(got), bits(ref))


def test_paged_full_size_serving_m4_equals_contiguous():
    # B = 64 sequences of 512..32768 keys, M = 4 (R = 32 rows per kv head),
    # 64-row pages: about 8000 pages shuffled over the pool.
    import torch
    import int8_kv_decode_gb300 as K
    wl = WORKLOADS["serving_b64_m4"]
    x = make_workload(wl, device="cuda")
    k8 = torch.empty((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty((wl.Hkv, x.cap_rows), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    K.quantize_kv(x.k_rows, k8, ks)
    K.quantize_kv(x.v_rows, v8, vs)
    rs = torch.as_tensor(x.row_start, device="cuda")
    ctx = torch.as_tensor(x.ctx, device="cuda")
    q = torch.as_tensor(x.q, device="cuda")
    ref = K.decode(q, k8, ks, v8, vs, rs, ctx, x.max_ctx)
    L = page_layout(x.ctx, x.row_start, wl.M, 64, seed=11)
    kp, ksp, vp, vsp = paged_copy(L, k8, ks, v8, vs, seed=11)
    del k8, v8
    bt = torch.from_numpy(L.block_table).cuda()
    ws = K.alloc_workspace(wl.B, wl.M, wl.Hq, x.max_ctx)
    got = K.decode_paged(q, kp, ksp, vp, vsp, bt, 64, ctx, x.max_ctx, workspace=ws)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    assert K.get_device_status(ws) == 0


# R = 8: the one-tile kernel; R = 32 with 6 sequences: its row groups; R = 32
# with 48 long sequences (more work items than the row-group bound): tcgen05
@pytest.mark.parametrize("M,Hq,B,ctx", [(2, 8, 6, ("uniform", 100, 900)),
                                        (4, 16, 6, ("uniform", 100, 900)),
                                        (4, 16, 48, ("uniform", 20000, 30000))])
def test_paged_bad_tables_are_flagged_without_touching_other_sequences(M, Hq, B, ctx):
    import torch
    import int8_kv_decode_gb300 as K
    wl = custom(f"paged_bad_m{M}_b{B}", B, M, Hq, 2, ctx, outliers=False)
    c = upload(wl) if B <= 8 else device_upload(wl)
    pc = Paged(c, 64, seed=3)
    ws = K.alloc_workspace(wl.B, wl.M, wl.Hq, c.x.max_ctx)
    clean = pc.decode(c, workspace=ws).cpu().numpy()
    assert K.get_device_status(ws) == 0
    n_pages = (c.x.ctx + wl.M - 1 + 63) // 64
    # a table too narrow for the longest sequences: those get NaN rows
    cols = int(np.median(n_pages))
    narrow = pc.bt[:, :cols].contiguous()
    out = pc.decode(c, bt=narrow, workspace=ws).cpu().numpy()
    short = n_pages > cols
    assert short.any() and (~short).any()
    assert np.isnan(out[short]).all()
    assert np.array_equal(bits(out[~short]), bits(clean[~short]))
    assert K.get_device_status(ws) == 1          # KATTN_DEVERR_BAD_SEQUENCE
    # entries outside the pool (one too large, one negative): flagged, page 0 read instead
    bad = pc.bt.clone()
    bad[1, 0] = pc.layout.n_pages + 5
    bad[4, n_pages[4] - 1] = -3
    out = pc.decode(c, bt=bad, workspace=ws).cpu().numpy()
    others = [b for b in range(wl.B) if b not in (1, 4)]
    assert np.array_equal(bits(out[others]), bits(clean[others]))
    assert np.isfinite(out[[1, 4]]).all()
    assert K.get_device_status(ws) == 4          # KATTN_DEVERR_BAD_PAGE
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,P,p_mode", [("spec_verify", 32, 0), ("spec_verify", 64, 3),
                                           ("qwen_layer", 128, 0)])
def test_paged_append_equals_separate_calls_and_the_oracle(name, P, p_mode):
    # kattn_decode_paged_append: the step's K/V rows quantized into the pool at
    # the physical rows of each sequence's M newest keys, then the paged
    # decode, in one launch chain.  The same bytes as the two row appends and
    # kattn_decode_paged; the oracle quantizes the rows itself and decodes its
    # contiguous copy of the cache.
    import torch
    import int8_kv_decode_gb300 as K
    import oracle
    from helpers import ROUNDED_REL_L2, assert_f32_tolerance, pinned_tiling, rel_l2
    C, Bk = pinned_tiling()
    c = upload(WORKLOADS[name], rep=3)
    wl, x = c.x.wl, c.x
    fused, separate = Paged(c, P, seed=5), Paged(c, P, seed=5)
    seqs = np.repeat(np.arange(wl.B), wl.M)
    keys = np.concatenate([np.arange(int(n) - 1, int(n) - 1 + wl.M) for n in x.ctx])
    bt = fused.layout.block_table
    phys = bt[seqs, keys // P].astype(np.int64) * P + keys % P
    fresh = make_workload(wl, rep=4)
    knew = np.ascontiguousarray(fresh.k_rows[:len(phys)])
    vnew = np.ascontiguousarray(fresh.v_rows[:len(phys)])
    tk, tv = torch.from_numpy(knew).cuda(), torch.from_numpy(vnew).cuda()
    dst = torch.from_numpy(phys).cuda()
    ws = K.alloc_workspace(wl.B, wl.M, wl.Hq, x.max_ctx)
    got = K.decode_paged_append(c.q, tk, tv, dst, fused.k8, fused.ks, fused.v8, fused.vs,
                                fused.bt, P, c.ctx, x.max_ctx, p_mode=p_mode,
                                workspace=ws).cpu().numpy()
    assert K.get_device_status(ws) == 0
    K.quantize_kv_rows(tk, dst, separate.k8, separate.ks)
    K.quantize_kv_rows(tv, dst, separate.v8, separate.vs)
    ref = separate.decode(c, p_mode=p_mode).cpu().numpy()
    assert np.array_equal(bits(got), bits(ref))
    for a, b in ((fused.k8, separate.k8), (fused.ks, separate.ks), (fused.v8, separate.v8),
                 (fused.vs, separate.vs)):
        assert torch.equal(a, b)
    # the oracle: its own contiguous cache with the new rows at the same keys
    ok8, oks, ov8, ovs = c.ok8.copy(), c.oks.copy(), c.ov8.copy(), c.ovs.copy()
    rows = x.row_start[seqs] + keys
    nk8, nks = oracle.quant.quantize_kv(knew)
    nv8, nvs = oracle.quant.quantize_kv(vnew)
    ok8[:, rows], oks[:, rows], ov8[:, rows], ovs[:, rows] = nk8, nks, nv8, nvs
    want = oracle.attention.decode(x.q, ok8, oks, ov8, ovs, x.row_start, x.ctx, p_mode=p_mode,
                                   C=C, Bk=Bk)
    if p_mode == 0:
        assert_f32_tolerance(got, want)
    else:
        assert rel_l2(got, want) <= ROUNDED_REL_L2
