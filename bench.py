#!/usr/bin/env python3
"""Decode-attention benchmark: KV GB/s and queries/s on GB300, % of HBM roofline.

One step = one decode step of the hot path over one batch of synthetic
sequences: kattn_decode_append (kattn_decode_paged_append for the paged
layout) quantizes this step's appended K and V rows into the int8 cache and
decodes every sequence, in one call.  The
default workload is the serving mix: 256 ragged sequences, contexts
log-uniform in [512, 32768], 32 query / 4 KV heads, head_dim 128, M = 1,
float32 P, fast mode.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

With N > 1 (torchrun, one rank per GPU) every rank decodes its own batch
(weak scaling, no data-path collective); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "serving_b256_m1"
METRIC = "decode_attn_kv_GBps"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_BYTES_NOMINAL = 129 * 1024 * 1024
HEAD_DIM = 128
# The source files each decode kernel is built from: a traffic line stays
# valid while they are unchanged.
_COMMON_SOURCES = ["device_common.cuh", "kattn_internal.cuh"]
KERNEL_SOURCES = {
    "decode_fast_kernel": ["decode_fast.cu", "decode_split.cuh"] + _COMMON_SOURCES,
    "decode_tc_kernel": ["decode_fast.cu", "decode_split.cuh", "tcgen05_common.cuh",
                         "decode_tc.cu"] + _COMMON_SOURCES,
    "decode_exact_kernel": ["decode_exact.cu"] + _COMMON_SOURCES,
}


# ------------------------------------------------------------ accounting --

def kv_bytes(ctx, M: int, Hkv: int, d: int = HEAD_DIM) -> int:
    """Algorithmic KV bytes of one decode call: every visible (key, kv head)
    row once -- int8 K and V rows plus their two float32 scales."""
    return int(sum(Hkv * (int(c) + M - 1) * (2 * d + 8) for c in ctx))


def qo_bytes(B: int, M: int, Hq: int, d: int = HEAD_DIM) -> int:
    """float32 queries read plus float32 outputs written."""
    return 2 * B * M * Hq * d * 4


def append_rows(row_start, ctx, M: int):
    """Cache rows written by this step: the M newest rows of each sequence
    (draft column j's own key is row ctx + j - 1)."""
    rows = []
    for rs, c in zip(row_start, ctx):
        rows.extend(int(rs) + int(c) - 1 + j for j in range(M))
    return rows


def load_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


ROW_GROUP_MAX_ITEMS = 4096   # the library's bound on work items for row groups
WINDOW_KEYS = 512


def roofline_kernel(g: int, M: int, exact: bool, B: int = 1 << 20, max_ctx: int = 1 << 20,
                    Hkv: int = 1) -> str:
    """The decode kernel a call launches: exact mode; the one-tile mma.sync
    kernel for up to 8 query rows per (sequence, kv head), and for more rows
    when the batch has few work items (row groups); P.V on tcgen05 for 17..32
    rows; else the mma.sync split pass."""
    if exact:
        return "decode_exact_kernel"
    R = g * M
    items = B * ((max_ctx + M - 1 + WINDOW_KEYS - 1) // WINDOW_KEYS) * Hkv   # an upper bound
    if R > 8 and items <= ROW_GROUP_MAX_ITEMS:
        return "decode_fast_kernel"
    return "decode_tc_kernel" if 16 < R <= 32 else "decode_fast_kernel"


def _code_only(text: str) -> str:
    """C++ source without its comments and with whitespace collapsed, so that
    an edit of a comment does not change a kernel's hash."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(kernel: str = "decode_fast_kernel", paged: bool = False) -> str:
    """Hash of the code (comments dropped) of the files a decode kernel is built from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel] + (["decode_fast_paged.cu"] if paged else []):
        with open(os.path.join(ROOT, "int8_kv_decode_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_key(workload: str, page_rows: int = 0) -> str:
    """The name a workload's traffic line carries: the paged layout is its own."""
    return f"{workload}_paged{page_rows}" if page_rows else workload


def paged_rows(block_table, page_rows: int, seqs, keys):
    """Physical cache row of key keys[i] of sequence seqs[i] in a paged layout."""
    import numpy as np
    seqs = np.asarray(seqs, np.int64)
    keys = np.asarray(keys, np.int64)
    return block_table[seqs, keys // page_rows].astype(np.int64) * page_rows + keys % page_rows


def profiled_traffic(workload: str, sha: str):
    """DRAM bytes per launch of the decode kernel from a committed ncu summary
    line 'traffic_per_launch <workload> <source sha> <bytes>', if the kernel
    sources are unchanged since the capture; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name), encoding="utf-8") as f:
            for line in f:
                parts = line.strip().strip("`").split()
                if len(parts) == 4 and parts[0] == "traffic_per_launch" \
                        and parts[1] == workload and parts[2] == sha:
                    return float(parts[3])
    return None


# ------------------------------------------------------------- clocks ----

CLOCK_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def start_clock_sampler(gpu_id: str, path: str, period_ms: int = 20):
    try:
        f = open(path, "w")
        p = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                              "-i", gpu_id, "-lms", str(period_ms)], stdout=f,
                             stderr=subprocess.DEVNULL)
        return p, f
    except OSError:
        return None, None


def stop_clock_sampler(handle):
    p, f = handle
    if p is not None:
        p.terminate()
        try:
            p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            p.kill()
    if f is not None:
        f.close()


def parse_clocks(text: str, t0: float = None, t1: float = None):
    """Summarise nvidia-smi samples (CSV, no header, no units).  Samples whose
    timestamp falls in [t0, t1] (epoch seconds) are used when there are any;
    otherwise all samples are."""
    rows = []
    for line in text.splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) != 8:
            continue
        try:
            ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
            rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[4:]))
        except (ValueError, IndexError):
            continue
    if not rows:
        return None
    inside = [r for r in rows if t0 is not None and t0 - 0.05 <= r[0] <= t1 + 0.05]
    use = inside or rows
    reasons = sorted({REASON_NAMES[i] for r in use for i, v in enumerate(r[3])
                      if v.lower().startswith("active")})
    return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
            "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


# --------------------------------------------------------- distribution --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(local_bytes: float, local_queries: float, local_seconds: float, pg=None):
    """Whole-job totals: bytes and queries summed over ranks, time = max over
    ranks (the slowest rank bounds the job)."""
    if pg is None:
        return local_bytes, local_queries, local_seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_bytes, local_queries], dtype=torch.float64)
    m = torch.tensor([local_seconds], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t, m = t.cuda(), m.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(m, op=dist.ReduceOp.MAX)
    return float(t[0]), float(t[1]), float(m[0])


# ---------------------------------------------------------------- oracle --

def oracle_sample(wl, n_seq: int, seed_rep: int = 0):
    """Host inputs for the first n_seq context lengths of the workload (same
    length draw, fresh host values), quantized by the oracle."""
    import numpy as np
    import oracle
    from synth import make_lengths, make_workload
    import dataclasses
    rng = np.random.Generator(np.random.PCG64(wl.index * 1000 + seed_rep))
    ctx = make_lengths(wl, rng)[:n_seq]
    small = dataclasses.replace(wl, B=len(ctx))
    x = make_workload(small, rep=seed_rep, ctx_override=ctx)
    k8, ks = oracle.quant.quantize_kv(x.k_rows)
    v8, vs = oracle.quant.quantize_kv(x.v_rows)
    return x, (k8, ks, v8, vs)


def time_oracle(wl, budget_s: float, max_seq: int = 12):
    """Oracle reference decode (float64, f32 P) on whole sequences of the
    workload until budget_s of CPU time is spent.  Returns (GB/s, queries/s,
    seconds, sequences, cores)."""
    import contextlib
    import oracle
    try:
        from threadpoolctl import threadpool_limits
        limit = threadpool_limits(limits=1)
    except ImportError:
        limit = contextlib.nullcontext()
    x, (k8, ks, v8, vs) = oracle_sample(wl, max_seq)
    spent = 0.0
    nbytes = nq = n = 0
    with limit:
        while spent < budget_s:                   # passes over the sample until the budget
            for b in range(x.wl.B):
                t0 = time.perf_counter()
                oracle.attention.decode(x.q[b:b + 1], k8, ks, v8, vs, x.row_start[b:b + 1],
                                        x.ctx[b:b + 1])
                spent += time.perf_counter() - t0
                nbytes += kv_bytes(x.ctx[b:b + 1], wl.M, wl.Hkv)
                nq += wl.M
                n += 1
                if spent >= budget_s:
                    break
    return nbytes / spent / 1e9, nq / spent, spent, n, 1


def _oracle_worker(job):
    """One process of the all-cores oracle baseline: decode one sequence of
    the workload's length draw, repeatedly, for budget_s of its own time."""
    wl_name, i, budget_s = job
    import numpy as np
    import oracle
    from synth import WORKLOADS, make_lengths, make_workload
    import dataclasses
    wl = WORKLOADS[wl_name]
    rng = np.random.Generator(np.random.PCG64(wl.index * 1000))
    lengths = make_lengths(wl, rng)
    ctx = lengths[i % len(lengths):][:1]
    x = make_workload(dataclasses.replace(wl, B=1), rep=100 + i, ctx_override=ctx)
    k8, ks = oracle.quant.quantize_kv(x.k_rows)
    v8, vs = oracle.quant.quantize_kv(x.v_rows)
    spent, nbytes = 0.0, 0
    while spent < budget_s:
        t0 = time.perf_counter()
        oracle.attention.decode(x.q, k8, ks, v8, vs, x.row_start, x.ctx)
        spent += time.perf_counter() - t0
        nbytes += kv_bytes(x.ctx, wl.M, wl.Hkv)
    return nbytes, spent


def _one_thread():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"


def time_oracle_all_cores(wl, budget_s: float):
    """The oracle on every core this process may use: one spawned worker per
    core, each on its own sequence of the workload; GB/s = all their KV bytes
    / the longest worker's time."""
    import multiprocessing as mp
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    with mp.get_context("spawn").Pool(n, initializer=_one_thread) as pool:
        res = pool.map(_oracle_worker, [(wl.name, i % 12, budget_s) for i in range(n)])
    total = sum(r[0] for r in res)
    secs = max(r[1] for r in res)
    return total / secs / 1e9, n, secs


def run_reference(args):
    """The reference arm: the CPU oracle, timed as it stands, one bounded
    sample of the workload per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from synth import WORKLOADS
    import oracle
    wl = WORKLOADS[args.workload]
    x, (k8, ks, v8, vs) = oracle_sample(wl, args.ref_sequences)
    n_seq = x.wl.B
    bytes_per_step = kv_bytes(x.ctx, wl.M, wl.Hkv)

    def step():
        oracle.attention.decode(x.q, k8, ks, v8, vs, x.row_start, x.ctx)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = bytes_per_step / dt / 1e9
    sample = (f"{n_seq} sequences of the {wl.name} workload (first {n_seq} context lengths, "
              f"mean {float(x.ctx.mean()):.0f}), float64 reference, f32 P, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "queries_per_s": n_seq * wl.M / dt,
        "config": workload_config(wl, x.ctx, note="bounded sample"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, ctx, note=None, l2=None, launch=None, p_mode="f32", exact=False,
                    page_rows=0):
    import numpy as np
    c = {"workload": wl.name, "B": wl.B, "M": wl.M, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
         "ctx": wl.ctx if isinstance(wl.ctx, int) else f"{wl.ctx[0]}[{wl.ctx[1]},{wl.ctx[2]}]",
         "mean_ctx": float(np.mean(ctx)), "p_mode": p_mode, "exact_mode": bool(exact),
         "layout": f"paged, {page_rows}-row pages in shuffled order" if page_rows else "contiguous"}
    if l2:
        c["l2"] = l2
    if launch:
        c["launch"] = launch
    if note:
        c["note"] = note
    return c


# ------------------------------------------------------------------ ours --

def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import int8_kv_decode_gb300 as K
    from synth import WORKLOADS, make_workload

    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N>1 with torchrun")
    pg = None
    if world > 1:
        dist.init_process_group(backend="nccl")
        pg = dist.group.WORLD
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K.load()

    wl = WORKLOADS[args.workload]
    x = make_workload(wl, rep=rank, device=str(dev))
    B, M, Hq, Hkv, d = wl.B, wl.M, wl.Hq, wl.Hkv, wl.d
    kvb = kv_bytes(x.ctx, M, Hkv)
    qob = qo_bytes(B, M, Hq)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES_NOMINAL
    n_copies = max(1, math.ceil(3 * l2 / kvb))          # keep every step L2-cold
    caches = []
    for _ in range(n_copies):
        k8 = torch.empty((Hkv, x.cap_rows, d), dtype=torch.int8, device=dev)
        v8 = torch.empty_like(k8)
        ks = torch.empty((Hkv, x.cap_rows), dtype=torch.float32, device=dev)
        vs = torch.empty_like(ks)
        K.quantize_kv(x.k_rows, k8, ks)                   # the prefill, untimed
        K.quantize_kv(x.v_rows, v8, vs)
        caches.append((k8, ks, v8, vs))
    dst = torch.tensor(append_rows(x.row_start, x.ctx, M), dtype=torch.int64, device=dev)
    knew = x.k_rows[dst].contiguous()
    vnew = x.v_rows[dst].contiguous()
    P = int(args.page_rows)
    bt = None
    if P:
        # The same rows in a paged layout (shuffled pages): every cache copy is
        # re-laid out and the contiguous copy dropped; the step's appends go to
        # the paged rows of keys ctx - 1 .. ctx + M - 2.
        import numpy as np
        from synth.paging import page_layout, paged_copy
        L = page_layout(x.ctx, x.row_start, M, P, seed=rank)
        caches = [paged_copy(L, *cc, seed=c) for c, cc in enumerate(caches)]
        bt = torch.from_numpy(L.block_table).to(dev)
        seqs = np.repeat(np.arange(B), M)
        keys = np.concatenate([np.arange(int(c) - 1, int(c) - 1 + M) for c in x.ctx])
        dst = torch.from_numpy(paged_rows(L.block_table, P, seqs, keys)).to(dev)
    x.k_rows = x.v_rows = None                          # free the float32 prefill rows
    torch.cuda.empty_cache()
    q = x.q.contiguous()
    rs = torch.from_numpy(x.row_start).to(dev)
    ctx = torch.from_numpy(x.ctx).to(dev)
    max_ctx = int(x.ctx.max())
    ws = K.alloc_workspace(B, M, Hq, max_ctx, dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    pm = K.P_MODES[args.p_mode]
    exact = bool(args.exact)

    # The step's inputs (the queries, the new K/V rows, their cache rows and
    # the context lengths) and its output; the caches stay resident.
    io0 = dict(q=q, knew=knew, vnew=vnew, ctx=ctx, dst=dst, out=out)

    def decode(i, io=io0):
        k8, ks, v8, vs = caches[i % n_copies]
        if P:
            K.decode_paged(io["q"], k8, ks, v8, vs, bt, P, io["ctx"], max_ctx, out=io["out"],
                           workspace=None if exact else ws, p_mode=pm, exact_mode=exact)
            return
        K.decode(io["q"], k8, ks, v8, vs, rs, io["ctx"], max_ctx, out=io["out"],
                 workspace=None if exact else ws, p_mode=pm, exact_mode=exact)

    def step(i, io=io0):
        k8, ks, v8, vs = caches[i % n_copies]
        if exact:
            # exact mode has no fused append: the two appends, then the decode
            K.quantize_kv_rows(io["knew"], io["dst"], k8, ks)
            K.quantize_kv_rows(io["vnew"], io["dst"], v8, vs)
            decode(i, io)
            return
        # this step's K/V rows appended inside the decode call
        if P:
            K.decode_paged_append(io["q"], io["knew"], io["vnew"], io["dst"], k8, ks, v8, vs, bt,
                                  P, io["ctx"], max_ctx, out=io["out"], workspace=ws, p_mode=pm)
            return
        K.decode_append(io["q"], io["knew"], io["vnew"], io["dst"], k8, ks, v8, vs, rs,
                        io["ctx"], max_ctx, out=io["out"], workspace=ws, p_mode=pm)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # CUDA graphs per cache copy for the step and for the decode alone: one
    # graph holds a single step, another G consecutive steps on consecutive
    # cache copies (as a model step's graph holds a layer's attention call
    # between its other kernels, so the graph's own launch is not paid per
    # call).  A replay is one host call, so small steps are timed on the GPU
    # rather than on the Python launch path.  The graphs hold the same
    # launches as the eager calls above (the warm-up did the one-time set-up).
    G = max(1, int(args.graph_steps))
    run_steps = lambda i0, n: [step(i0 + k) for k in range(n)]       # noqa: E731
    run_decodes = lambda i0, n: [decode(i0 + k) for k in range(n)]   # noqa: E731
    if not args.no_graphs:
        graphs = {}
        for c in range(n_copies):
            for n in sorted({1, G}):
                gs, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, capture_error_mode="thread_local"):
                    run_steps(c, n)
                with torch.cuda.graph(gd, capture_error_mode="thread_local"):
                    run_decodes(c, n)
                graphs[(c, n)] = (gs, gd)
        run_steps = lambda i0, n: graphs[(i0 % n_copies, n)][0].replay()     # noqa: E731
        run_decodes = lambda i0, n: graphs[(i0 % n_copies, n)][1].replay()   # noqa: E731
        for i in range(args.warmup):
            run_steps(i, 1)
        torch.cuda.synchronize(dev)

    def timed(run, i0, k):
        """Exactly k steps from step index i0: graphs of G steps, then single ones."""
        i = 0
        while i < k:
            n = G if k - i >= G else 1
            run(i0 + i, n)
            i += n
    stream = torch.cuda.current_stream(dev)
    if pg is not None:
        dist.barrier()

    gpu_id = str(local)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    import tempfile
    clock_fd, clock_path = tempfile.mkstemp(prefix=f"kattn_bench_clocks_rank{rank}_", suffix=".csv")
    os.close(clock_fd)
    sampler = start_clock_sampler(gpu_id, clock_path) if rank == 0 else (None, None)
    time.sleep(0.3)                                       # sampler start-up

    # Timed region: K whole steps (append + decode).
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    if pg is not None:
        dist.barrier()
    wall0 = time.time()
    start.record(stream)
    timed(run_steps, args.warmup, args.steps)
    end.record(stream)
    torch.cuda.synchronize(dev)
    if pg is not None:
        dist.barrier()
    elapsed = start.elapsed_time(end) / 1e3

    # The decode alone, K launches back to back on the same rotating copies:
    # its average duration is the roofline's denominator.
    d_start, d_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    d_start.record(stream)
    timed(run_decodes, args.warmup, args.steps)
    d_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    decode_s = d_start.elapsed_time(d_end) / 1e3 / args.steps
    stop_clock_sampler(sampler)

    total_bytes, total_q, tmax = aggregate(kvb * args.steps, B * M * args.steps, elapsed, pg)

    # End to end through the public API: every step's inputs copied from
    # pinned host memory, every step's output read back to pinned host
    # memory.  As a serving loop does, the copies run on their own streams
    # against two sets of device buffers, so that step i + 1's inputs arrive
    # and step i - 1's output leaves while step i computes; a buffer is
    # refilled only after the step that used it is done and its output is out.
    # The inputs travel packed in one pinned buffer (one copy per step), each
    # at a 256-byte aligned offset; the device buffers are typed views of the
    # same layout.
    names = ("q", "knew", "vnew", "ctx", "dst")
    offs, pos = {}, 0
    for k in names:
        offs[k] = pos
        pos += (io0[k].numel() * io0[k].element_size() + 255) // 256 * 256
    h_pack = torch.empty(pos, dtype=torch.uint8).pin_memory()

    def views(raw):
        return {k: raw[offs[k]:offs[k] + io0[k].numel() * io0[k].element_size()]
                .view(io0[k].dtype).view(io0[k].shape) for k in names}

    for k, t in views(h_pack).items():
        t.copy_(io0[k].cpu())
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(io0[k].numel() * io0[k].element_size() for k in names)
    d2h = h_outs[0].numel() * 4
    d_packs = [torch.empty(pos, dtype=torch.uint8, device=dev) for _ in range(2)]
    bufs = [dict(views(d_packs[b]), out=torch.empty_like(out)) for b in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # buffer b's inputs landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the step on buffer b is done
    ev_out = [torch.cuda.Event() for _ in range(2)]    # buffer b's output is on the host
    torch.cuda.synchronize(dev)
    if pg is not None:
        dist.barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    s_in.wait_event(e_start)
    s_out.wait_event(e_start)
    for i in range(args.steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[b])            # step i - 2 has read buffer b
            d_packs[b].copy_(h_pack, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])               # step i - 2's output has left
        step(i, bufs[b])
        ev_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            h_outs[b].copy_(bufs[b]["out"], non_blocking=True)
            ev_out[b].record(s_out)
    for b in range(min(2, args.steps)):
        stream.wait_event(ev_out[b])
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e_elapsed = e_start.elapsed_time(e_end) / 1e3
    _, _, e_tmax = aggregate(0.0, 0.0, e_elapsed, pg)

    if rank != 0:
        dist.destroy_process_group() if pg is not None else None
        return 0

    peak, peak_kind = load_peak_hbm()
    algo = kvb + qob
    achieved = algo / decode_s / 1e9
    rkernel = roofline_kernel(wl.Hq // wl.Hkv, wl.M, exact, B, max_ctx, Hkv)
    sha = kernel_source_sha(rkernel, paged=bool(P) and not exact)
    clocks = None
    try:
        with open(clock_path) as f:
            clocks = parse_clocks(f.read(), wall0, wall1)
    except OSError:
        pass
    finally:
        try:
            os.unlink(clock_path)
        except OSError:
            pass

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        gbs, qps, secs, nseq, cores = time_oracle(wl, args.cpu_budget)
        cpu = {"value": gbs, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": (f"{nseq} sequence decodes ({secs:.1f} s single-threaded) over repeated "
                          f"passes on 12 whole sequences of {wl.name}, float64 reference, f32 P; "
                          f"GB/s = their KV bytes / time"),
               "queries_per_s": qps}
        if not args.no_cpu_all_cores:
            gbs_all, n_all, secs_all = time_oracle_all_cores(wl, args.cpu_budget / 2)
            cpu["all_cores"] = {"value": gbs_all, "unit": UNIT, "cores": n_all,
                                "sample": (f"{n_all} spawned processes, one sequence of {wl.name} "
                                           f"each, {secs_all:.1f} s; GB/s = their KV bytes / "
                                           f"the longest process's time")}

    line = {
        "metric": METRIC, "value": total_bytes / tmax / 1e9, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tmax / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8/f32", "data": "synthetic",
        "queries_per_s": total_q / tmax,
        "config": workload_config(
            wl, x.ctx, l2=(f"inputs larger than L2: {kvb / 1e9:.2f} GB KV per step x "
                           f"{n_copies} rotating cache copies vs {l2 / 2**20:.0f} MiB L2"),
            launch=("eager" if args.no_graphs else
                    "one CUDA graph replay per step" if G == 1 else
                    f"CUDA graphs of {G} consecutive steps on consecutive cache copies "
                    f"(a remainder of single-step graphs), {args.steps} steps timed"),
            p_mode=args.p_mode, exact=exact, page_rows=P),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_nominal_8000": achieved / NOMINAL_HBM_GBS,
                     "traffic": profiled_traffic(traffic_key(wl.name, P), sha),
                     "kernel": rkernel,
                     "algorithmic_bytes_per_launch": algo,
                     "avg_launch_us": decode_s * 1e6, "kernel_source_sha": sha},
        "kv_frac_of_step": (kvb / (elapsed / args.steps) / 1e9) / peak,
        "cpu_baseline": cpu,
        "e2e": {"value": total_bytes / e_tmax / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": ((3 if exact else K.decode_launch_count(B, M, Hq, Hkv, max_ctx))
                         * args.steps),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle CPU time for the cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-all-cores", action="store_true",
                    help="skip the all-cores oracle baseline (the single-threaded one stays)")
    ap.add_argument("--p-mode", default="f32", choices=["f32", "bf16", "e4m3", "e4m3x448",
                                                        "e4m3x256", "e4m3direct"],
                    help="rounding of the P that multiplies V")
    ap.add_argument("--exact", action="store_true",
                    help="time exact mode (token-order scan, table-driven exp) instead of fast mode")
    ap.add_argument("--page-rows", type=int, default=0,
                    help="time the paged layout: pages of this many rows (32 * 2^k) in shuffled "
                         "order (default: the contiguous cache)")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch every step eagerly instead of replaying CUDA graphs")
    ap.add_argument("--graph-steps", type=int, default=8,
                    help="steps captured in one CUDA graph (1: one graph replay per step)")
    ap.add_argument("--ref-sequences", type=int, default=2,
                    help="sequences per step of the reference arm")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
