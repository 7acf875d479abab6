"""Context-parallel decode on one GPU: the shards of a sequence's keys are
decoded by separate kattn_decode_shard calls (each with a cache holding only
its own keys), their partials stacked as an all-gather leaves them, and
kattn_merge_shards must return, byte for byte, what kattn_decode returns on
one cache holding every key (kattn_decode is held to the oracle by
test_gpu_parity.py; the merged output is also checked against the oracle).
Ranks are emulated as consecutive calls on one device: no kernel waits on
another.
"""

import numpy as np
import pytest

from helpers import assert_f32_tolerance, custom, device_upload, oracle_decode, run, upload
from int8_kv_decode_gb300 import context_parallel as cp
from synth import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def bits(a):
    return np.ascontiguousarray(np.asarray(a, np.float32)).view(np.uint32)


def shard_cache(c, M, shard, ws, seed):
    """This shard's keys of every sequence, packed one sequence after another
    with 0..3 spare rows of random bytes in between; row_start of sequences
    without a key in the shard is -7 (it must not be read)."""
    import torch
    x = c.x
    k0, k1 = cp.shard_key_range(x.ctx, M, shard, ws)
    n = np.maximum(k1 - k0, 0)
    rng = np.random.default_rng(seed)
    gaps = rng.integers(0, 4, len(n))
    starts = np.concatenate([[0], np.cumsum(n + gaps)[:-1]]).astype(np.int64)
    cap = int((n + gaps).sum()) + 1
    Hkv, _, d = c.k8.shape
    g = torch.Generator(device=c.k8.device)
    g.manual_seed(seed)
    k8 = torch.randint(-127, 128, (Hkv, cap, d), generator=g, device=c.k8.device, dtype=torch.int8)
    v8 = torch.randint(-127, 128, (Hkv, cap, d), generator=g, device=c.k8.device, dtype=torch.int8)
    ks = torch.rand((Hkv, cap), generator=g, device=c.k8.device) + 0.5
    vs = torch.rand((Hkv, cap), generator=g, device=c.k8.device) + 0.5
    for b in range(len(n)):
        if n[b] == 0:
            continue
        src = slice(int(x.row_start[b] + k0[b]), int(x.row_start[b] + k1[b]))
        dst = slice(int(starts[b]), int(starts[b] + n[b]))
        k8[:, dst] = c.k8[:, src]
        v8[:, dst] = c.v8[:, src]
        ks[:, dst] = c.ks[:, src]
        vs[:, dst] = c.vs[:, src]
    rs = torch.from_numpy(np.where(n > 0, starts, -7)).to(c.k8.device)
    return k8, ks, v8, vs, rs


def cp_decode(c, n_shards, p_mode=0, seed=0, ctx=None, check_status=True):
    import torch
    import int8_kv_decode_gb300 as K
    wl = c.x.wl
    ctx = c.ctx if ctx is None else ctx
    ws = cp.plan_shards(c.x.max_ctx, wl.M, n_shards)
    parts = []
    for s in range(n_shards):
        k8, ks, v8, vs, rs = shard_cache(c, wl.M, s, ws, seed + 101 * s)
        wsp = K.alloc_workspace(wl.B, wl.M, wl.Hq, c.x.max_ctx)
        parts.append(K.decode_shard(c.q, k8, ks, v8, vs, rs, ctx, c.x.max_ctx, s, ws,
                                    p_mode=p_mode, workspace=wsp))
        if check_status:
            assert K.get_device_status(wsp) == 0
    allp = torch.stack(parts)                    # what an all-gather leaves
    mws = torch.zeros(256, dtype=torch.uint8, device=c.q.device)
    out = K.merge_shards(allp, ctx, wl.M, wl.Hq, c.x.max_ctx, workspace=mws)
    return out, mws


@pytest.mark.parametrize("n_shards", [2, 3])
@pytest.mark.parametrize("p_mode", [0, 2])
def test_spec_verify_shards_equal_single_gpu_bytes(n_shards, p_mode):
    import int8_kv_decode_gb300 as K
    c = upload(WORKLOADS["spec_verify"])        # B 16, M 5, ctx 1024..4096, outliers
    ref = run(c, p_mode=p_mode).cpu().numpy()
    out, mws = cp_decode(c, n_shards, p_mode=p_mode, seed=n_shards)
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))
    assert K.get_device_status(mws) == 0


@pytest.mark.parametrize("n_shards,B", [(2, 8), (3, 8), (2, 48)])
def test_r32_shards_equal_single_gpu_bytes(n_shards, B):
    # 32 query rows per kv head (M = 4, GQA 8): the window partials in shard
    # mode, gathered and merged, give the single-GPU bytes.  8 sequences take
    # row groups; 48 long ones (more work items than the row-group bound) the
    # tcgen05 kernel.
    import int8_kv_decode_gb300 as K
    if B <= 8:
        c = upload(custom("cp_r32", B, 4, 16, 2, ("uniform", 300, 5000), outliers=True))
    else:
        c = device_upload(custom("cp_r32_big", B, 4, 16, 2, ("uniform", 20000, 30000),
                                 outliers=True))
    ref = run(c).cpu().numpy()
    out, mws = cp_decode(c, n_shards, seed=70 + n_shards)
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))
    assert K.get_device_status(mws) == 0


def test_short_and_single_window_sequences():
    # sequences of 1 key, one window, exactly one window, and long ones; with
    # 4 shards most sequences have no key in the last shards
    wl = custom("cp_mix", 7, 2, 8, 2, ("uniform", 1, 2))
    ctx = np.array([1, 300, 511, 512, 1500, 5000, 2049], dtype=np.int32)
    c = upload(wl, ctx_override=ctx)
    ref = run(c).cpu().numpy()
    for n in (2, 4):
        out, _ = cp_decode(c, n, seed=40 + n)
        assert np.array_equal(bits(out.cpu().numpy()), bits(ref))
    assert_f32_tolerance(out.cpu().numpy(), oracle_decode(c))


def test_more_than_64_windows_per_row():
    # 80 windows: the merge's 32-warps-per-row shape reads across shards
    wl = custom("cp_long", 2, 1, 32, 4, ("uniform", 1, 2))
    ctx = np.array([40500, 3000], dtype=np.int32)
    c = upload(wl, ctx_override=ctx)
    ref = run(c).cpu().numpy()
    out, _ = cp_decode(c, 3, seed=9)
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


def test_bad_context_length_gives_nan_rows_only():
    import torch
    import int8_kv_decode_gb300 as K
    wl = custom("cp_bad", 4, 1, 8, 2, ("uniform", 600, 1800))
    c = upload(wl)
    ref = run(c).cpu().numpy()
    bad = c.ctx.clone()
    bad[2] = c.x.max_ctx + 1                     # beyond max_ctx: invalid everywhere
    out, mws = cp_decode(c, 2, ctx=bad, check_status=False)
    out = out.cpu().numpy()
    assert np.isnan(out[2]).all()
    keep = [0, 1, 3]
    assert np.array_equal(bits(out[keep]), bits(ref[keep]))
    assert K.get_device_status(mws) == 1         # KATTN_DEVERR_BAD_SEQUENCE
    torch.cuda.synchronize()
