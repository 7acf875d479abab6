"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: bit-exact for quantized bytes, integer QK scores and exact mode;
max|delta| <= 1e-4 and relative L2 <= 1e-5 for fast mode with f32 P;
relative L2 <= 2e-3 for the rounded-P modes against the oracle applying the
same rounding at the same points; bit-identical run to run and across
columns / batch sizes.
"""

import numpy as np
import pytest

import oracle
from helpers import (ROUNDED_REL_L2, assert_f32_tolerance, bits, custom, oracle_decode,
                     pinned_tiling, rel_l2, row_mask, run, sample_rows, upload)
from synth import WORKLOADS, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


# ----------------------------------------------------------- quantization --

@pytest.mark.parametrize("name", ["tiny", "qwen_layer", "spec_verify"])
def test_quantize_kv_bytes(name):
    c = upload(WORKLOADS[name])
    assert np.array_equal(c.k8.cpu().numpy(), c.ok8)
    assert np.array_equal(c.v8.cpu().numpy(), c.ov8)
    assert np.array_equal(bits(c.ks.cpu()), bits(c.oks))
    assert np.array_equal(bits(c.vs.cpu()), bits(c.ovs))


def test_quantize_kv_offset_zero_rows_and_ties():
    import torch
    import int8_kv_decode_gb300 as K
    rng = np.random.default_rng(5)
    rows = rng.standard_normal((9, 3, 128)).astype(np.float32)
    rows[2, 1] = 0.0                               # zero row -> scale 0, zeros
    rows[4, 0] = 0.0
    rows[4, 0, :6] = [127, 2.5, -2.5, 3.5, 0.5, -1.5]   # scale exactly 1: ties
    cap, r0 = 20, 7
    q8 = torch.full((3, cap, 128), 99, dtype=torch.int8, device="cuda")
    sc = torch.full((3, cap), -1.0, dtype=torch.float32, device="cuda")
    K.quantize_kv(torch.from_numpy(rows).cuda(), q8, sc, dst_row0=r0)
    oq, os_ = oracle.quant.quantize_kv(rows)
    assert np.array_equal(q8.cpu().numpy()[:, r0:r0 + 9], oq)
    assert np.array_equal(bits(sc.cpu().numpy()[:, r0:r0 + 9]), bits(os_))
    assert (q8.cpu().numpy()[:, :r0] == 99).all() and (q8.cpu().numpy()[:, r0 + 9:] == 99).all()
    assert list(q8.cpu().numpy()[0, r0 + 4, :6]) == [127, 2, -2, 4, 0, -2]


# --------------------------------------------------------------- QK scores --

@pytest.mark.parametrize("name", ["tiny", "qwen_layer", "spec_verify"])
def test_qk_scores_bit_exact(name):
    import int8_kv_decode_gb300 as K
    c = upload(WORKLOADS[name])
    S, q8, qs = K.qk_scores_debug(c.q, c.k8, c.ks, c.rs, c.ctx, c.x.max_ctx, want_q=True)
    S = S.cpu().numpy()
    oS, oq8, oqs = oracle.attention.qk_scores(c.x.q, c.ok8, c.x.row_start, c.x.ctx)
    valid = oS != oracle.attention.NO_SCORE
    assert np.array_equal(S[valid], oS[valid].astype(np.int32))
    assert np.all(S[~valid] == -2 ** 31)          # entries t >= L_j untouched
    assert np.array_equal(q8.cpu().numpy(), oq8)
    assert np.array_equal(bits(qs.cpu()), bits(oqs))


# -------------------------------------------------------------- exact mode --

@pytest.mark.parametrize("name,p_mode", [("tiny", 0), ("tiny", 1), ("tiny", 2), ("tiny", 3),
                                         ("tiny", 4),
                                         ("qwen_layer", 0), ("qwen_layer", 3)])
def test_exact_mode_bit_exact(name, p_mode):
    c = upload(WORKLOADS[name])
    got = run(c, exact_mode=True, p_mode=p_mode).cpu().numpy()
    ref = oracle_decode(c, mode="exact", p_mode=p_mode)
    assert np.array_equal(bits(got), bits(ref))


def test_exact_mode_spec_verify_sampled():
    c = upload(WORKLOADS["spec_verify"])
    got = run(c, exact_mode=True).cpu().numpy()
    rows = [(b, j, h) for b in (0, 15) for j in range(5) for h in (0, 3, 29)]
    ref = oracle_decode(c, mode="exact", rows=rows)
    m = row_mask(got.shape, rows)
    assert np.array_equal(bits(got[m]), bits(ref[m]))


# --------------------------------------------------------------- fast mode --

@pytest.mark.parametrize("name", ["tiny", "qwen_layer"])
def test_fast_f32_within_tolerance(name):
    c = upload(WORKLOADS[name])
    got = run(c).cpu().numpy()
    assert_f32_tolerance(got, oracle_decode(c))


def test_fast_f32_spec_verify_sampled():
    c = upload(WORKLOADS["spec_verify"])
    got = run(c).cpu().numpy()
    rows = sample_rows(c.x, 60, seed=1)
    ref = oracle_decode(c, rows=rows)
    assert_f32_tolerance(got, ref, row_mask(got.shape, rows))


@pytest.mark.parametrize("p_mode", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("name", ["tiny", "qwen_layer"])
def test_fast_rounded_p_modes(name, p_mode):
    import int8_kv_decode_gb300 as K
    C, Bk = pinned_tiling()
    c = upload(WORKLOADS[name])
    got = run(c, p_mode=p_mode).cpu().numpy()
    same = oracle_decode(c, p_mode=p_mode, C=C, Bk=Bk)
    assert rel_l2(got, same) <= ROUNDED_REL_L2
    # Where the rounding moves the result measurably, the kernel must apply
    # it: its distance to the same-rounding oracle is far below the size of
    # the rounding's own effect.  (With very peaked attention -- the outlier
    # channels -- p is ~1 or ~0 and no rounding changes anything.)
    effect = rel_l2(same, oracle_decode(c))
    if effect > 1e-5:
        assert rel_l2(got, same) < 0.25 * effect, (rel_l2(got, same), effect)


def test_fast_deterministic_run_to_run():
    c = upload(WORKLOADS["spec_verify"])
    for p_mode in (0, 2):
        a = run(c, p_mode=p_mode).cpu().numpy()
        for _ in range(2):
            assert np.array_equal(bits(run(c, p_mode=p_mode).cpu().numpy()), bits(a))


@pytest.mark.parametrize("exact", [False, True])
def test_columns_equal_single_column_decodes(exact):
    # "Kestrel_VLLM - 18" §二: batch-verify column j must equal, byte for
    # byte, an M=1 decode that saw the same tokens (ctx + j keys).
    import int8_kv_decode_gb300 as K
    c = upload(WORKLOADS["spec_verify"])
    full = run(c, exact_mode=exact).cpu().numpy()
    for j in range(c.x.wl.M):
        qj = c.q[:, j:j + 1].contiguous()
        one = K.decode(qj, c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx + j, c.x.max_ctx + j,
                       exact_mode=exact).cpu().numpy()
        assert np.array_equal(bits(full[:, j:j + 1]), bits(one)), j


def test_batch_size_invariance():
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
    rs = torch.from_numpy(x.row_start).cuda()
    ctx = torch.from_numpy(x.ctx).cuda()
    full = K.decode(x.q, k8, ks, v8, vs, rs, ctx, x.max_ctx).cpu().numpy()
    # (a single long sequence takes the other launch shape of the window merge)
    bl = int(np.argmax(x.ctx))
    for lo, hi in ((0, 1), (5, 9), (10, 26), (63, 64), (bl, bl + 1)):
        sub = K.decode(x.q[lo:hi].contiguous(), k8, ks, v8, vs, rs[lo:hi].contiguous(),
                       ctx[lo:hi].contiguous(), int(x.ctx[lo:hi].max()) + 7).cpu().numpy()
        assert np.array_equal(bits(full[lo:hi]), bits(sub)), (lo, hi)
    # the same sequence moved to another place in another cache
    b = 11
    r0, r1 = x.rows_of(b)
    n = r1 - r0
    k2 = torch.zeros((wl.Hkv, n + 37, wl.d), dtype=torch.int8, device="cuda")
    v2, ks2, vs2 = torch.zeros_like(k2), torch.zeros((wl.Hkv, n + 37), device="cuda"), None
    vs2 = torch.zeros_like(ks2)
    k2[:, 37:] = k8[:, r0:r1]
    v2[:, 37:] = v8[:, r0:r1]
    ks2[:, 37:] = ks[:, r0:r1]
    vs2[:, 37:] = vs[:, r0:r1]
    one = K.decode(x.q[b:b + 1].contiguous(), k2, ks2, v2, vs2,
                   torch.tensor([37], dtype=torch.int64, device="cuda"),
                   ctx[b:b + 1].contiguous(), int(x.ctx[b])).cpu().numpy()
    assert np.array_equal(bits(full[b:b + 1]), bits(one))


@pytest.mark.parametrize("g,M", [(1, 1), (4, 1), (8, 1), (1, 8), (4, 3), (8, 2), (4, 5), (8, 3),
                                 (8, 4), (8, 5), (8, 8), (3, 8), (16, 2), (32, 1)])
def test_shape_sweep(g, M):
    # ctx around the block and split sizes ("海光 DCU 实测" §4: one shape being
    # exact proves nothing about the others).
    import int8_kv_decode_gb300 as K
    C, Bk = pinned_tiling()
    ctxs = np.array([1, 2, Bk - 1, Bk, Bk + 1, C - 1, C, C + 1, 2 * C + 3], np.int32)
    wl = custom(f"sweep_g{g}_m{M}", len(ctxs), M, 2 * g, 2, 1, outliers=True)
    c = upload(wl, ctx_override=ctxs)
    got = run(c).cpu().numpy()
    assert_f32_tolerance(got, oracle_decode(c))
    for j in range(M):
        one = K.decode(c.q[:, j:j + 1].contiguous(), c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx + j,
                       c.x.max_ctx + j).cpu().numpy()
        assert np.array_equal(bits(got[:, j:j + 1]), bits(one))
    ex = run(c, exact_mode=True, p_mode=2).cpu().numpy()
    rows = [(b, j, h) for b in range(len(ctxs)) for j in (0, M - 1) for h in (0, 2 * g - 1)]
    ref = oracle_decode(c, mode="exact", p_mode=2, rows=rows)
    m = row_mask(ex.shape, rows)
    assert np.array_equal(bits(ex[m]), bits(ref[m]))


@pytest.mark.parametrize("g,M", [(1, 3), (3, 1), (1, 5)])
def test_odd_row_count_over_several_windows(g, M):
    # R = g * M odd and sequences longer than one 512-key window: the
    # per-window partial rows must stay 16-byte aligned for any R.
    import int8_kv_decode_gb300 as K
    ctxs = np.array([513, 1500, 2049, 700], np.int32)
    wl = custom(f"odd_g{g}_m{M}", len(ctxs), M, 2 * g, 2, 1, outliers=True)
    c = upload(wl, ctx_override=ctxs)
    got = run(c).cpu().numpy()
    assert_f32_tolerance(got, oracle_decode(c))
    for j in range(M):
        one = K.decode(c.q[:, j:j + 1].contiguous(), c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx + j,
                       c.x.max_ctx + j).cpu().numpy()
        assert np.array_equal(bits(got[:, j:j + 1]), bits(one))


@pytest.mark.parametrize("B,M,Hq", [(1000, 1, 8), (2100, 1, 8), (2100, 4, 16)])
def test_many_short_sequences(B, M, Hq):
    # Many short sequences: most work items are one short window, so warps
    # of a CTA reach the next item at very different times.  Above 2048
    # sequences the work list is written by its own kernel rather than by
    # the query-packing launch.  Sampled rows against the oracle, and the
    # bytes of each half of the batch decoded alone.
    import int8_kv_decode_gb300 as K
    wl = custom(f"many{B}_m{M}", B, M, Hq, 2, ("uniform", 1, 1200), outliers=False)
    c = upload(wl)
    got = run(c).cpu().numpy()
    rows = sample_rows(c.x, 40, seed=3)
    assert_f32_tolerance(got, oracle_decode(c, rows=rows), row_mask(got.shape, rows))
    for lo, hi in ((0, B // 2), (B // 2, B)):
        half = K.decode(c.q[lo:hi].contiguous(), c.k8, c.ks, c.v8, c.vs, c.rs[lo:hi].contiguous(),
                        c.ctx[lo:hi].contiguous(), int(c.x.ctx[lo:hi].max())).cpu().numpy()
        assert np.array_equal(bits(got[lo:hi]), bits(half)), (lo, hi)


@pytest.mark.parametrize("shape", ["spec_verify", "r32"])   # row groups at R = 40 and R = 32
def test_decode_replays_in_a_cuda_graph(shape):
    # The three launches of a fast decode, captured once and replayed, give
    # the bytes of an ordinary call.
    import torch
    import int8_kv_decode_gb300 as K
    c = upload(WORKLOADS["spec_verify"] if shape == "spec_verify" else
               custom("graph_r32", 12, 4, 16, 2, ("uniform", 100, 3000), outliers=True))
    B, M, Hq, _ = c.q.shape
    ws = K.alloc_workspace(B, M, Hq, c.x.max_ctx)
    ref = run(c, workspace=ws).cpu().numpy()
    out = torch.full_like(c.q, float("nan"))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        K.decode(c.q, c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx, c.x.max_ctx, out=out, workspace=ws)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


def test_bad_sequence_is_flagged_without_touching_other_rows():
    import torch
    import int8_kv_decode_gb300 as K
    wl = custom("bad", 3, 2, 8, 2, 300, outliers=False)
    c = upload(wl)
    clean = run(c).cpu().numpy()
    ws = K.alloc_workspace(3, 2, 8, c.x.max_ctx)
    assert K.get_device_status(ws) == 0
    bad_ctx = c.ctx.clone()
    bad_ctx[1] = c.x.max_ctx + 1                       # breaks ctx <= max_ctx
    out = K.decode(c.q, c.k8, c.ks, c.v8, c.vs, c.rs, bad_ctx, c.x.max_ctx,
                   workspace=ws).cpu().numpy()
    assert np.isnan(out[1]).all()
    assert np.array_equal(bits(out[[0, 2]]), bits(clean[[0, 2]]))
    assert K.get_device_status(ws) == 1
    assert K.get_device_status(ws) == 0                # the read cleared it
    bad_rs = c.rs.clone()
    bad_rs[2] = c.x.cap_rows                           # rows past the cache
    ex = K.decode(c.q, c.k8, c.ks, c.v8, c.vs, bad_rs, c.ctx, c.x.max_ctx,
                  exact_mode=True).cpu().numpy()
    assert np.isnan(ex[2]).all() and np.isfinite(ex[:2]).all()
    torch.cuda.synchronize()


# ------------------------------------------------------------ fused append --

@pytest.mark.parametrize("name,p_mode", [("spec_verify", 0), ("spec_verify", 2), ("qwen_layer", 0),
                                         ("r32", 0)])
def test_decode_append_equals_separate_calls(name, p_mode):
    # kattn_decode_append: the M draft rows of every sequence quantized into
    # the cache inside the decode launch -- the same cache bytes and outputs
    # as kattn_quantize_kv_rows twice followed by kattn_decode.
    import torch
    import int8_kv_decode_gb300 as K
    # r32: 32 query rows per kv head (M = 4, GQA 8) over 6 sequences: row groups
    wl = WORKLOADS[name] if name != "r32" else custom("append_r32", 6, 4, 16, 2,
                                                       ("uniform", 200, 3000), outliers=True)
    x = make_workload(wl, rep=5)
    dev = "cuda"
    k_rows = torch.from_numpy(x.k_rows).to(dev)
    v_rows = torch.from_numpy(x.v_rows).to(dev)
    # the draft rows of sequence b: row_start + ctx - 1 + j (j < M)
    dst = torch.tensor([int(x.row_start[b]) + int(x.ctx[b]) - 1 + j
                        for b in range(wl.B) for j in range(wl.M)], dtype=torch.int64, device=dev)
    caches = []
    for _ in range(2):
        k8 = torch.zeros((wl.Hkv, x.cap_rows, wl.d), dtype=torch.int8, device=dev)
        v8 = torch.zeros_like(k8)
        ks = torch.zeros((wl.Hkv, x.cap_rows), dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        K.quantize_kv(k_rows, k8, ks)                 # the prefill, then stale draft rows
        K.quantize_kv(v_rows, v8, vs)
        caches.append((k8, ks, v8, vs))
    knew = torch.randn((dst.numel(), wl.Hkv, wl.d), device=dev) * 2
    vnew = torch.randn_like(knew)
    q = torch.from_numpy(x.q).to(dev)
    rs = torch.from_numpy(x.row_start).to(dev)
    ctx = torch.from_numpy(x.ctx).to(dev)
    k8, ks, v8, vs = caches[0]
    K.quantize_kv_rows(knew, dst, k8, ks)
    K.quantize_kv_rows(vnew, dst, v8, vs)
    ref = K.decode(q, k8, ks, v8, vs, rs, ctx, x.max_ctx, p_mode=p_mode).cpu().numpy()
    k8b, ksb, v8b, vsb = caches[1]
    got = K.decode_append(q, knew, vnew, dst, k8b, ksb, v8b, vsb, rs, ctx, x.max_ctx,
                          p_mode=p_mode).cpu().numpy()
    assert np.array_equal(bits(got), bits(ref))
    for a, b in zip(caches[0], caches[1]):
        assert torch.equal(a, b)


def test_row_hashes_match_the_oracle_and_find_a_planted_divergence():
    # kattn_hash_rows (FNV-1a 64 per row, "Kestrel_VLLM - 18" §3.4) against the
    # oracle's hashes of the same bytes: the quantized K cache, the exact-mode
    # output, and strided / misaligned row views.
    import torch
    import int8_kv_decode_gb300 as K
    from oracle import hashdump as H
    c = upload(WORKLOADS["qwen_layer"])
    k_bytes = c.k8.reshape(-1, 128)
    assert np.array_equal(K.hash_rows(k_bytes).cpu().numpy().view(np.uint64),
                          H.hash_rows(c.ok8.reshape(-1, 128)))
    ex = run(c, exact_mode=True)
    ref = oracle_decode(c, mode="exact").astype(np.float32)
    gh = K.hash_rows(ex.reshape(-1, 128)).cpu().numpy().view(np.uint64)
    assert H.first_divergence(gh, H.hash_rows(ref.reshape(-1, 128))) is None
    planted = ref.reshape(-1, 128).copy()
    planted[17, 3] = np.nextafter(planted[17, 3], np.float32(np.inf))
    assert H.first_divergence(gh, H.hash_rows(planted)) == 17
    # a strided view whose rows start 4 bytes past 16-byte boundaries
    view = ex.reshape(-1, 128)[:, 1:101]
    assert np.array_equal(K.hash_rows(view).cpu().numpy().view(np.uint64),
                          H.hash_rows(ex.reshape(-1, 128)[:, 1:101].cpu().numpy()))


@pytest.mark.parametrize("p_mode", [0, 2])
def test_long_rows_alone_equal_the_batch(p_mode):
    # Rows of up to 79 windows (several per merge slot), decoded in a batch
    # of 40 and in sub-batches of one and three sequences: the same bytes,
    # whichever launch shape the merge takes for each.
    import int8_kv_decode_gb300 as K
    wl = custom("long_mix", 40, 1, 32, 4, ("uniform", 600, 40000), outliers=True)
    c = upload(wl)
    assert K.decode_launch_count(40, 1, 32, 4, c.x.max_ctx) == 3
    ws = K.alloc_workspace(40, 1, 32, c.x.max_ctx)
    full = run(c, p_mode=p_mode, workspace=ws).cpu().numpy()
    assert K.get_device_status(ws) == 0
    for lo, hi in ((0, 1), (7, 10), (int(np.argmax(c.x.ctx)), int(np.argmax(c.x.ctx)) + 1)):
        mc = int(c.x.ctx[lo:hi].max())
        sub = K.decode(c.q[lo:hi].contiguous(), c.k8, c.ks, c.v8, c.vs, c.rs[lo:hi].contiguous(),
                       c.ctx[lo:hi].contiguous(), mc, p_mode=p_mode).cpu().numpy()
        assert np.array_equal(bits(full[lo:hi]), bits(sub)), (lo, hi)
    rows = sample_rows(c.x, 24, seed=5)
    if p_mode == 0:
        assert_f32_tolerance(full, oracle_decode(c, rows=rows), row_mask(full.shape, rows))


def test_e4m3_direct_mode_columns_and_oracle():
    # p_mode 5 (e4m3 P into the tensor-core P.V, one f16 operand): the M = 4
    # batch (32 rows per kv head over 5 sequences: row groups) against the oracle with
    # the same rounding, every draft column equal to the M = 1 decode (the
    # mma.sync kernel) byte for byte, and no exact-mode form.
    import int8_kv_decode_gb300 as K
    C, Bk = pinned_tiling()
    wl = custom("direct_m4", 5, 4, 16, 2, ("uniform", 300, 2500), outliers=True, index=77)
    c = upload(wl)
    got = run(c, p_mode=5).cpu().numpy()
    rows = sample_rows(c.x, 16, seed=5)
    same = oracle_decode(c, p_mode=5, C=C, Bk=Bk, rows=rows)
    m = row_mask(got.shape, rows)
    assert rel_l2(got[m], same[m]) <= ROUNDED_REL_L2
    for j in range(wl.M):
        one = K.decode(c.q[:, j:j + 1].contiguous(), c.k8, c.ks, c.v8, c.vs, c.rs, c.ctx + j,
                       c.x.max_ctx + j, p_mode=5).cpu().numpy()
        assert np.array_equal(bits(got[:, j:j + 1]), bits(one)), j
    with pytest.raises(Exception):
        run(c, p_mode=5, exact_mode=True)
