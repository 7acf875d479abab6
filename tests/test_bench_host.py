"""Host-side logic of bench.py (no GPU): byte accounting, clock parsing, the
profile lookup, whole-job aggregation over 2 gloo ranks, and the reference
arm's JSON line."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_kv_bytes_and_queries():
    # 264 bytes per (key, kv head) at d = 128: 2 x 128 int8 + 2 float32 scales
    assert bench.kv_bytes([1024], 1, 4) == 4 * 1024 * 264
    assert bench.kv_bytes([10, 20], 3, 2) == 2 * (12 + 22) * 264
    assert bench.qo_bytes(2, 3, 4) == 2 * 2 * 3 * 4 * 128 * 4


def test_append_rows_are_each_columns_own_key():
    assert bench.append_rows([5, 100], [3, 7], 2) == [7, 8, 106, 107]


def test_parse_clocks_window_and_reasons():
    text = "\n".join([
        "2026/12/02 10:00:00.100, 1980, 2070, 700.1, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:01.100, 1900, 2070, 900.0, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:05.100, 1200, 2070, 300.0, Not Active, Active, Not Active, Not Active",
    ])
    import time
    t0 = time.mktime(time.strptime("2026/12/02 10:00:00", "%Y/%m/%d %H:%M:%S"))
    c = bench.parse_clocks(text, t0, t0 + 2)
    assert c["samples"] == 2 and c["in_timed_region"]
    assert c["sm_mhz"] == 1940 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clocks("garbage") is None


def test_profiled_traffic_lookup(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "x.md").write_text(
        "text\n`traffic_per_launch serving_b256_m1 abc123 2.5e9`\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("serving_b256_m1", "abc123") == 2.5e9
    assert bench.profiled_traffic("serving_b256_m1", "changed") is None


def _agg_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = bench.aggregate(100.0 * (rank + 1), 5.0, 0.5 + rank, dist.group.WORLD)
    q.put((rank, res))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_agg_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    for r in range(2):
        assert got[r] == (300.0, 10.0, 1.5)     # bytes summed, time = max


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_all_cores_oracle_baseline_runs_in_spawned_processes():
    import bench
    from synth import WORKLOADS
    gbs, cores, secs = bench.time_oracle_all_cores(WORKLOADS["tiny"], 0.2)
    assert cores >= 1 and secs >= 0.2 and gbs > 0


def test_roofline_kernel_follows_the_dispatch():
    # 17..32 query rows per (sequence, kv head) with many work items run the
    # tcgen05 P.V kernel; with few, row groups of the one-tile kernel.
    assert bench.roofline_kernel(8, 1, False) == "decode_fast_kernel"
    assert bench.roofline_kernel(8, 2, False) == "decode_fast_kernel"      # R = 16
    assert bench.roofline_kernel(8, 3, False) == "decode_tc_kernel"        # R = 24
    assert bench.roofline_kernel(8, 4, False) == "decode_tc_kernel"        # R = 32
    assert bench.roofline_kernel(8, 5, False) == "decode_fast_kernel"      # R = 40
    assert bench.roofline_kernel(8, 4, True) == "decode_exact_kernel"
    # few work items: more than 8 rows go to row groups of the one-tile kernel
    assert bench.roofline_kernel(8, 4, False, 6, 3000, 2) == "decode_fast_kernel"
    assert bench.roofline_kernel(8, 4, False, 64, 32768, 4) == "decode_tc_kernel"
    assert bench.roofline_kernel(8, 1, False, 6, 3000, 2) == "decode_fast_kernel"


def test_paged_rows_and_traffic_key():
    # Key t of sequence b lives at block_table[b][t // P] * P + t % P; the
    # paged layout's traffic line carries its own name.
    bt = np.array([[3, 1, -1], [0, 2, 4]], np.int32)
    got = bench.paged_rows(bt, 32, [0, 0, 1, 1], [0, 33, 64, 5])
    assert got.tolist() == [96, 33, 128, 5]
    assert bench.traffic_key("serving_b256_m4", 64) == "serving_b256_m4_paged64"
    assert bench.traffic_key("serving_b256_m4") == "serving_b256_m4"


def test_kernel_hash_ignores_comments_but_not_code():
    import bench
    src = "int f(int x) {  // the answer\n  return x + 1; /* one */\n}\n"
    same = "int f(int x) {\n  // changed words\n  return x + 1;\n}\n"
    other = "int f(int x) { return x + 2; }"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    assert len(bench.kernel_source_sha("decode_fast_kernel")) == 16


def test_committed_traffic_lines_match_the_kernel_sources():
    # Every workload with a traffic line in the committed ncu summary resolves
    # against the current sources of the kernel that runs it (the summary was
    # taken from these kernels), and its bytes are close to the algorithmic
    # bytes of a launch: no K/V byte read twice.
    import bench
    cases = [("serving_b256_m1", "decode_fast_kernel", False, 2323.93e6),
             ("long_128k", "decode_fast_kernel", False, 553.78e6),
             ("serving_b256_m4", "decode_tc_kernel", False, 2349.91e6),
             ("spec_verify", "decode_fast_kernel", False, 44.33e6),
             ("serving_b256_m1_paged64", "decode_fast_kernel", True, 2323.93e6)]
    for workload, kernel, paged, algorithmic in cases:
        got = bench.profiled_traffic(workload, bench.kernel_source_sha(kernel, paged=paged))
        assert got is not None, workload
        assert 0.9 * algorithmic <= got <= 1.15 * algorithmic, (workload, got)
