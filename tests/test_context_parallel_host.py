"""Context-parallel host logic without a GPU: the shard plan covers every key
of every sequence exactly once on window boundaries, the partials of 2 gloo
ranks are gathered rank-major (the layout kattn_merge_shards reads), and the
composite call refuses CPU tensors (no fallback)."""

import os

import numpy as np
import pytest
import torch

from int8_kv_decode_gb300 import context_parallel as cp
from int8_kv_decode_gb300.api import WINDOW_KEYS


@pytest.mark.parametrize("n_shards", [1, 2, 3, 8])
@pytest.mark.parametrize("M", [1, 5])
def test_shards_cover_every_key_once_on_window_boundaries(n_shards, M):
    rng = np.random.default_rng(n_shards * 10 + M)
    ctx = np.concatenate([[1, 511, 512, 513, 1024], rng.integers(1, 40000, 60)])
    max_ctx = int(ctx.max())
    ws = cp.plan_shards(max_ctx, M, n_shards)
    assert n_shards * ws >= cp.windows_of(max_ctx + M - 1)
    assert (n_shards - 1) * ws < cp.windows_of(max_ctx + M - 1) or n_shards == 1
    held = np.zeros(len(ctx), dtype=np.int64)
    prev_end = np.zeros(len(ctx), dtype=np.int64)
    for s in range(n_shards):
        k0, k1 = cp.shard_key_range(ctx, M, s, ws)
        assert np.all(k0 % WINDOW_KEYS == 0)
        n = np.maximum(k1 - k0, 0)
        has = n > 0
        assert np.all(k0[has] == prev_end[has])           # contiguous, in shard order
        prev_end = np.where(has, k1, prev_end)
        held += n
    assert np.array_equal(held, ctx + M - 1)              # every key exactly once


def test_plan_rejects_bad_sizes():
    with pytest.raises(ValueError):
        cp.plan_shards(100, 1, 0)
    assert cp.plan_shards(1, 1, 4) == 1                   # more shards than windows


def _gather_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, Ws, Hkv, stride = 3, 2, 2, 8
    local = torch.arange(B * Ws * Hkv * stride, dtype=torch.float32).reshape(B, Ws, Hkv, stride)
    local = local + 1000.0 * rank
    allp = cp.gather_partials(local)
    q.put((rank, allp.numpy()))
    dist.destroy_process_group()


def test_gather_is_rank_major_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_gather_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    base = np.arange(3 * 2 * 2 * 8, dtype=np.float32).reshape(3, 2, 2, 8)
    for r in range(2):
        a = got[r]
        assert a.shape == (2, 3, 2, 2, 8)
        assert np.array_equal(a[0], base) and np.array_equal(a[1], base + 1000.0)


def test_composite_call_refuses_cpu_tensors():
    q = torch.zeros(1, 1, 8, 128)
    k = torch.zeros(2, 16, 128, dtype=torch.int8)
    s = torch.zeros(2, 16)
    rs = torch.zeros(1, dtype=torch.int64)
    c = torch.ones(1, dtype=torch.int32)
    from int8_kv_decode_gb300 import api
    with pytest.raises(ValueError, match="CUDA"):
        api.decode_shard(q, k, s, k, s, rs, c, 16, 0, 1, workspace=torch.zeros(1024, dtype=torch.uint8))
