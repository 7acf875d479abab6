"""Seeded synthetic inputs for int8-KV decode attention.

This module is shared by the tests, the benchmark and the smoke check.  It
draws random numbers and lays them out; it holds none of the method's
arithmetic (no quantization, no scores, no softmax), so both the CUDA path
and the CPU oracle can consume what it produces without sharing any code.

Workload shapes follow the pages' setting: Qwen3-30B-A3B attention
(32 query heads, 4 KV heads, head_dim 128; "Kestrel_VLLM - 18", header
line naming the environment) and contexts from 1k to 128k tokens
("在 agent 时代如何快速验证 kernel 对精度的影响", section on the experiment's
corpus).  No dataset is used: Q/K/V are standard normal draws, optionally
with a few outlier channels scaled up.

Layouts produced here (all row-major, float32):
  q        [B][M][Hq][d]       queries, one per (sequence, draft column, head)
  kv rows  [cap_rows][Hkv][d]  K and V rows as they arrive for appending;
                               sequence b owns rows
                               [row_start[b], row_start[b] + ctx[b] + M - 1)
"""

from .gen import (  # noqa: F401
    Workload,
    WORKLOADS,
    make_workload,
    make_lengths,
    outlier_channels,
)
