"""Context-parallel decode: one sequence's keys spread over several GPUs.

Every rank holds the keys of a contiguous run of 512-key windows of every
sequence, reduces them into window partials (kattn_decode_shard), the ranks
all-gather the partials, and each rank combines them (kattn_merge_shards) in
the same fixed order as a single-GPU decode.  The one exchange is that
all-gather of (m, l, o) per window and query row; because the merge order
depends only on each row's own window count, the result equals the
single-GPU decode byte for byte ("Kestrel_VLLM - 18", §二: the combine order
must not depend on how the work is split).

This module is host logic only: the shard plan, which keys a rank holds,
and the gather.  The arithmetic runs in the library's kernels.
"""

from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import api
from .api import WINDOW_KEYS


def windows_of(keys) -> np.ndarray:
    """Windows a row of `keys` keys spans (ceil(keys / 512)), elementwise."""
    k = np.asarray(keys, dtype=np.int64)
    return (k + WINDOW_KEYS - 1) // WINDOW_KEYS


def plan_shards(max_ctx: int, M: int, n_shards: int) -> int:
    """Windows per shard so that n_shards shards cover a context of max_ctx
    (plus the M - 1 draft keys): ceil(windows / n_shards)."""
    if n_shards < 1 or max_ctx < 1 or M < 1:
        raise ValueError("n_shards, max_ctx and M must be positive")
    total = int(windows_of(max_ctx + M - 1))
    return max(1, -(-total // n_shards))


def shard_key_range(ctx, M: int, shard: int, win_per_shard: int):
    """Keys [k0, k1) of every sequence that shard `shard` holds (k1 <= k0:
    none).  ctx: the global context lengths [B]."""
    ctx = np.asarray(ctx, dtype=np.int64)
    k0 = np.full_like(ctx, shard * win_per_shard * WINDOW_KEYS)
    k1 = np.minimum(ctx + M - 1, (shard + 1) * win_per_shard * WINDOW_KEYS)
    return k0, k1


def gather_partials(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather every rank's partials [B][Ws][Hkv][stride] into
    [world][B][Ws][Hkv][stride], rank-major (shard s = rank s)."""
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(local.shape), dtype=local.dtype, device=local.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(out, local.contiguous(), group=group)
    else:
        dist.all_gather(list(out.unbind(0)), local.contiguous(), group=group)
    return out


def decode_context_parallel(q, k, k_scale, v, v_scale, row_start, ctx_len, max_ctx: int,
                            win_per_shard: int, *, group=None, p_mode=0, sm_scale: float = 0.0,
                            workspace=None, out=None):
    """One decode over keys spread across the ranks of `group` (rank r is
    shard r).  This rank's cache holds its keys as decode_shard describes;
    q, ctx_len (global lengths), max_ctx and the modes are the same on every
    rank.  Returns out [B][M][Hq][128] on every rank.  The ranks together
    must cover every sequence's windows: world * win_per_shard >=
    ceil((max_ctx + M - 1) / 512)."""
    rank = dist.get_rank(group)
    B, M, Hq, _ = q.shape
    if workspace is None:
        workspace = api.alloc_workspace(B, M, Hq, max_ctx, q.device)
    part = api.decode_shard(q, k, k_scale, v, v_scale, row_start, ctx_len, max_ctx, rank,
                            win_per_shard, p_mode=p_mode, sm_scale=sm_scale, workspace=workspace)
    allp = gather_partials(part, group)
    return api.merge_shards(allp, ctx_len, M, Hq, max_ctx, out=out, workspace=workspace)
