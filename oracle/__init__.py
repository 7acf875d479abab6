"""CPU oracle for int8-KV decode attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import anything from this package.  It shares no code with
the CUDA path (no kernels, headers, helpers, tables or constant generators)
and imports nothing from ``int8_kv_decode_gb300``.

It is plain and slow on purpose: numpy float32 where the method fixes f32
rounding, float64 (or exact rational arithmetic) everywhere else.

Sources (page title, then section):
  * "Kestrel_VLLM - 18 · 投机解码位级对拍收口" (wsisp.com) -- §3.3 gives the
    int8-query / int32-QK / per-token online softmax order and the
    table-driven expf; §二 gives the batch-column == M=1 invariant.
  * "在 agent 时代如何快速验证 kernel 对精度的影响" (susun-blog.com) --
    section "注意力权重：直接转 fp8 随上下文变差" gives the blockwise online
    softmax with round_p applied only to the P that multiplies V.

Modules:
  quant      -- per-row absmax/127 int8 quantization (K/V rows and queries)
  rounding   -- bf16 and fp8-e4m3 round-to-nearest-even, the round_p modes
  expf_tang  -- the table-driven exp (64-entry 2^(j/64) table, 3-term poly)
  attention  -- QK scores, reference decode (float64, with the rounding
                points mirrored for rounded-P modes) and the exact-mode
                float32 emulation
  hashdump   -- FNV-1a 64 row hashes and the first differing row (§3.4's
                parity-dump method)

Parity unpinned:
  * the absolute accuracy of the rounded-P modes against the infinitely
    precise softmax is not pinned by anything on the pages; only the
    same-rounding comparison is;
  * the order of the score scaling, s = ((f32(S) * (qs * ks)) * sm_scale),
    each product rounded once to float32: the pages are silent on it, so no
    pin outside the oracle fixes it (its tests restate it; the GPU path is
    held to it only through the end-to-end tolerances and exact mode).
"""

from . import quant, rounding, expf_tang, attention, hashdump  # noqa: F401
