"""Full-size parity: the specified workloads at their full sizes, decoded in
the launch configuration the benchmark times, against the CPU oracle.

The oracle cannot decode a whole full-size batch in seconds, so it checks
sampled rows, chosen to reach every sequence, every kv head, the first and
the last query head of a GQA group and (with draft columns) every column.
The oracle quantizes the generator's float32 rows itself; the device caches
must hold the same bytes.

* Long-context P-precision sweep: B = 4, 32q/4kv, ctx 8192 / 32768 / 131072
  with outlier channels, every P mode against the oracle with the same
  rounding ("在 agent 时代如何快速验证 kernel 对精度的影响", section
  "注意力权重"); exact mode bit for bit at 8192 and 32768.
* Serving sweep: 256 ragged sequences (ctx log-uniform in [512, 32768]) at
  M = 1 and M = 4 against the oracle, and batch invariance across batch
  sizes 64, 128 and 256: the same sequences decoded inside batches of each
  size give the same bytes ("Kestrel_VLLM - 18", §二).
* The fused KV append (the benchmark's step): the appended rows quantized by
  the oracle, the cache bytes and the decode against the oracle.
* The tcgen05 kernel at 20 and 24 rows (many work items), and every rounded-P
  mode on diffuse attention at 8k, where the rounding moves the output
  measurably and the kernel must follow the same-rounding oracle.
"""

import numpy as np
import pytest

import oracle
from helpers import (ROUNDED_REL_L2, assert_f32_tolerance, bits, custom, device_case, oracle_decode,
                     oracle_sequence_cache, oracle_sequence_rows, pinned_tiling, rel_l2, upload)
from synth import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _compare(got, ref, p_mode):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all()
    if p_mode == 0:
        return assert_f32_tolerance(got, ref)
    r = rel_l2(got, ref)
    assert r <= ROUNDED_REL_L2, r
    return None, r


def _long_rows(B, Hkv, g):
    """Per sequence b: one head of every kv head, the first or the last of
    the group alternately, so the four sequences cover both for every kv
    head."""
    return {b: [(0, kh * g + (0 if (b + kh) % 2 == 0 else g - 1)) for kh in range(Hkv)]
            for b in range(B)}


# ------------------------------------------------------ long-context sweep --

@pytest.mark.parametrize("name", ["long_8k", "long_32k", "long_128k"])
def test_long_context_every_p_mode_against_the_oracle(name):
    import int8_kv_decode_gb300 as K
    C, Bk = pinned_tiling()
    x, k8, ks, v8, vs, rs, ctx = device_case(name)
    wl = x.wl
    rows = _long_rows(wl.B, wl.Hkv, wl.g)
    caches = {b: oracle_sequence_cache(x, b, k8, ks, v8, vs) for b in rows}
    for p_mode in range(6):
        out = K.decode(x.q, k8, ks, v8, vs, rs, ctx, x.max_ctx, p_mode=p_mode).cpu().numpy()
        assert np.isfinite(out).all(), p_mode
        got, ref = [], []
        for b, rr in rows.items():
            o = oracle_sequence_rows(x, b, caches[b], rr, p_mode=p_mode, C=C, Bk=Bk)
            for (j, h) in rr:
                got.append(out[b, j, h])
                ref.append(o[j, h])
        _compare(np.array(got), np.array(ref), p_mode)


@pytest.mark.parametrize("name,p_mode", [("long_8k", 0), ("long_8k", 3), ("long_32k", 0)])
def test_long_context_exact_mode_bit_exact(name, p_mode):
    import int8_kv_decode_gb300 as K
    x, k8, ks, v8, vs, rs, ctx = device_case(name)
    wl = x.wl
    out = K.decode(x.q, k8, ks, v8, vs, rs, ctx, x.max_ctx, exact_mode=True,
                   p_mode=p_mode).cpu().numpy()
    picks = {0: [(0, 0), (0, wl.Hq - 1)], wl.B - 1: [(0, wl.g), (0, 2 * wl.g - 1)]}
    if name == "long_8k":
        picks[1] = [(0, 2 * wl.g + 3)]
        picks[2] = [(0, 3 * wl.g + 5)]
    for b, rr in picks.items():
        cache = oracle_sequence_cache(x, b)
        o = oracle_sequence_rows(x, b, cache, rr, mode="exact", p_mode=p_mode)
        for (j, h) in rr:
            assert np.array_equal(bits(out[b, j, h]), bits(o[j, h])), (b, j, h)


# ----------------------------------------------------------- serving sweep --

def _serving_rows(x, n_seq, seed):
    """Sampled (b, [(j, h)]) over n_seq sequences, always including the
    longest and the shortest, every draft column and every kv head."""
    wl = x.wl
    rng = np.random.default_rng(seed)
    seqs = [int(np.argmax(x.ctx)), int(np.argmin(x.ctx)), 0, wl.B - 1]
    while len(set(seqs)) < n_seq:
        seqs.append(int(rng.integers(wl.B)))
    out = {}
    for i, b in enumerate(dict.fromkeys(seqs)):
        rr = []
        for kh in range(wl.Hkv):
            j = (i + kh) % wl.M
            first_or_last = 0 if (i + kh) % 2 == 0 else wl.g - 1
            rr.append((j, kh * wl.g + first_or_last))
        out[b] = rr
    return out


@pytest.mark.parametrize("name", ["serving_b256_m1", "serving_b256_m4"])
def test_serving_full_size_against_the_oracle(name):
    import int8_kv_decode_gb300 as K
    x, k8, ks, v8, vs, rs, ctx = device_case(name)
    out = K.decode(x.q, k8, ks, v8, vs, rs, ctx, x.max_ctx).cpu().numpy()
    assert np.isfinite(out).all()
    got, ref = [], []
    for b, rr in _serving_rows(x, 10, seed=11).items():
        cache = oracle_sequence_cache(x, b, k8, ks, v8, vs)
        o = oracle_sequence_rows(x, b, cache, rr)
        for (j, h) in rr:
            got.append(out[b, j, h])
            ref.append(o[j, h])
    _compare(np.array(got), np.array(ref), 0)


@pytest.mark.parametrize("name", ["serving_b256_m1", "serving_b256_m4"])
def test_batch_invariance_across_batch_sizes_64_128_256(name):
    # The same sequences decoded inside batches of 256, 128 and 64 (in
    # order, and gathered from across the batch in shuffled order): every
    # row has the same bytes whatever batch it sits in.
    import torch
    import int8_kv_decode_gb300 as K
    x, k8, ks, v8, vs, rs, ctx = device_case(name)
    full = K.decode(x.q, k8, ks, v8, vs, rs, ctx, x.max_ctx).cpu().numpy()
    rng = np.random.default_rng(21)
    picks = [np.arange(0, 128), np.arange(128, 192), rng.permutation(256)[:128],
             rng.permutation(256)[:64]]
    for sel in picks:
        idx = torch.from_numpy(sel.astype(np.int64)).cuda()
        sub = K.decode(x.q[idx].contiguous(), k8, ks, v8, vs, rs[idx].contiguous(),
                       ctx[idx].contiguous(), int(x.ctx[sel].max())).cpu().numpy()
        assert np.array_equal(bits(sub), bits(full[sel])), len(sel)


# -------------------------------------------------------------- KV append --

def _append_case(name, rep=5):
    """A workload whose cache holds the prefill rows, plus the step's new K/V
    rows (the next instance of the same generator) for the M newest rows of
    every sequence: row_start + ctx - 1 + j."""
    wl = WORKLOADS[name] if name != "r32" else custom("append_r32", 6, 4, 16, 2,
                                                       ("uniform", 200, 3000), outliers=True)
    x = make_workload(wl, rep=rep)
    dst = np.array([int(x.row_start[b]) + int(x.ctx[b]) - 1 + j
                    for b in range(wl.B) for j in range(wl.M)], np.int64)
    fresh = make_workload(wl, rep=rep + 1)
    n = len(dst)
    assert fresh.cap_rows >= n
    knew = np.ascontiguousarray(fresh.k_rows[:n])
    vnew = np.ascontiguousarray(fresh.v_rows[:n])
    return x, dst, knew, vnew


@pytest.mark.parametrize("name,p_mode", [("spec_verify", 0), ("spec_verify", 3), ("qwen_layer", 0),
                                         ("r32", 0), ("r32", 2)])
def test_decode_append_against_the_oracle(name, p_mode):
    # kattn_decode_append quantizes the step's K/V rows into the cache and
    # decodes in one launch chain.  The oracle quantizes the same rows
    # itself, writes them into its copy of the cache and decodes.
    import torch
    import int8_kv_decode_gb300 as K
    C, Bk = pinned_tiling()
    x, dst, knew, vnew = _append_case(name)
    wl = x.wl
    dev = "cuda"
    k8 = torch.empty((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device=dev)
    v8 = torch.empty_like(k8)
    ks = torch.empty((wl.Hkv, x.cap_rows), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    K.quantize_kv(torch.from_numpy(x.k_rows).to(dev), k8, ks)     # the prefill
    K.quantize_kv(torch.from_numpy(x.v_rows).to(dev), v8, vs)
    out = K.decode_append(torch.from_numpy(x.q).to(dev), torch.from_numpy(knew).to(dev),
                          torch.from_numpy(vnew).to(dev), torch.from_numpy(dst).to(dev),
                          k8, ks, v8, vs, torch.from_numpy(x.row_start).to(dev),
                          torch.from_numpy(x.ctx).to(dev), x.max_ctx,
                          p_mode=p_mode).cpu().numpy()
    ok8, oks = oracle.quant.quantize_kv(x.k_rows)
    ov8, ovs = oracle.quant.quantize_kv(x.v_rows)
    nk8, nks = oracle.quant.quantize_kv(knew)
    nv8, nvs = oracle.quant.quantize_kv(vnew)
    ok8[:, dst], oks[:, dst], ov8[:, dst], ovs[:, dst] = nk8, nks, nv8, nvs
    assert np.array_equal(k8.cpu().numpy(), ok8)
    assert np.array_equal(bits(ks.cpu().numpy()), bits(oks))
    assert np.array_equal(v8.cpu().numpy(), ov8)
    assert np.array_equal(bits(vs.cpu().numpy()), bits(ovs))
    ref = oracle.attention.decode(x.q, ok8, oks, ov8, ovs, x.row_start, x.ctx, p_mode=p_mode,
                                  C=C, Bk=Bk)
    _compare(out, ref, p_mode)


def test_quantize_kv_rows_against_the_oracle():
    # Scattered destination rows, two of them outside the cache (skipped on
    # the device); every other row keeps its old bytes.
    import torch
    import int8_kv_decode_gb300 as K
    x, dst, knew, _ = _append_case("spec_verify", rep=8)
    wl = x.wl
    dst = dst.copy()
    dst[3] = -1
    dst[7] = x.cap_rows
    q8 = torch.full((wl.Hkv, x.cap_rows, wl.d), 99, dtype=torch.int8, device="cuda")
    sc = torch.full((wl.Hkv, x.cap_rows), -1.0, dtype=torch.float32, device="cuda")
    K.quantize_kv_rows(torch.from_numpy(knew).cuda(), torch.from_numpy(dst).cuda(), q8, sc)
    nk8, nks = oracle.quant.quantize_kv(knew)
    want_q = np.full((wl.Hkv, x.cap_rows, wl.d), 99, np.int8)
    want_s = np.full((wl.Hkv, x.cap_rows), -1.0, np.float32)
    keep = (dst >= 0) & (dst < x.cap_rows)
    want_q[:, dst[keep]] = nk8[:, keep]
    want_s[:, dst[keep]] = nks[:, keep]
    assert np.array_equal(q8.cpu().numpy(), want_q)
    assert np.array_equal(bits(sc.cpu().numpy()), bits(want_s))


@pytest.mark.parametrize("g,M", [(8, 3), (4, 5)])
def test_tcgen05_kernel_at_24_and_20_rows(g, M):
    # 17..32 query rows per kv head with more work items than the row-group
    # bound (48 sequences x about 50 windows x 2 kv heads > 4096): the tcgen05
    # kernel.  Every draft column equals the M = 1 decode byte for byte, and
    # sampled rows meet the oracle.
    import torch
    import int8_kv_decode_gb300 as K
    wl = custom(f"tc_r{g * M}", 48, M, 2 * g, 2, ("uniform", 20000, 30000), outliers=True,
                index=31)
    x = make_workload(wl, device="cuda")
    windows = (int(x.ctx.max()) + M - 1 + 511) // 512
    assert wl.B * windows * wl.Hkv > 4096
    k8 = torch.empty((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device="cuda")
    v8 = torch.empty_like(k8)
    ks = torch.empty((wl.Hkv, x.cap_rows), dtype=torch.float32, device="cuda")
    vs = torch.empty_like(ks)
    K.quantize_kv(x.k_rows, k8, ks)
    K.quantize_kv(x.v_rows, v8, vs)
    rs = torch.from_numpy(x.row_start).cuda()
    ctx = torch.from_numpy(x.ctx).cuda()
    out = K.decode(x.q, k8, ks, v8, vs, rs, ctx, x.max_ctx).cpu().numpy()
    for j in range(M):
        one = K.decode(x.q[:, j:j + 1].contiguous(), k8, ks, v8, vs, rs, ctx + j,
                       x.max_ctx + j).cpu().numpy()
        assert np.array_equal(bits(out[:, j:j + 1]), bits(one)), j
    got, ref = [], []
    for b in (0, int(np.argmax(x.ctx)), wl.B - 1):
        rr = [(j, (j + kh) % g + kh * g) for j in range(M) for kh in range(wl.Hkv)]
        o = oracle_sequence_rows(x, b, oracle_sequence_cache(x, b, k8, ks, v8, vs), rr)
        for (j, h) in rr:
            got.append(out[b, j, h])
            ref.append(o[j, h])
    _compare(np.array(got), np.array(ref), 0)


@pytest.mark.parametrize("p_mode", [1, 2, 3, 4, 5])
def test_rounded_p_acts_on_diffuse_attention_at_8k(p_mode):
    # No outlier channels: attention spreads over thousands of keys, so every
    # rounded-P mode moves the output measurably.  The kernel must sit within
    # the rounded-mode bound of the oracle with the same rounding, and far
    # closer to it than to the unrounded (f32 P) oracle.
    import int8_kv_decode_gb300 as K
    C, Bk = pinned_tiling()
    wl = custom("diffuse_8k", 2, 1, 32, 4, 8192, outliers=False, index=41)
    c = upload(wl)
    got = K.decode(c.q, c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx, c.x.max_ctx,
                   p_mode=p_mode).cpu().numpy()
    rows = [(b, 0, h) for b in range(wl.B) for h in (0, 7, 13, 20, 31)]
    same = oracle_decode(c, rows=rows, p_mode=p_mode, C=C, Bk=Bk)
    plain = oracle_decode(c, rows=rows)
    m = np.zeros(got.shape[:3], bool)
    for (b, j, h) in rows:
        m[b, j, h] = True
    effect = rel_l2(same[m], plain[m])
    dist = rel_l2(got[m], same[m])
    assert dist <= ROUNDED_REL_L2, dist
    assert effect > 1e-5, effect
    assert dist < 0.25 * effect, (dist, effect)
