"""kattn_decode_noalloc: the fast decode for callers that cannot allocate.

Callers such as an engine whose device memory belongs to its own arena, a
serving loop that must not pay cudaMalloc's latency between steps, or a
plugin interface that only passes input and output buffers cannot hand the
library a workspace.  This entry point keeps the scratch in a fixed device
array inside the library instead.  The test calls it through the C ABI twice
in a row and checks each result against kattn_decode with a workspace
allocated by the caller.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest

from helpers import assert_f32_tolerance, custom, run, upload
from synth import WORKLOADS


def _noalloc(c, out):
    import torch
    from int8_kv_decode_gb300 import _lib
    lib = _lib.load()
    B, M, Hq, d = c.q.shape
    Hkv, cap, _ = c.k8.shape
    return lib.kattn_decode_noalloc(
        c.q.data_ptr(), c.k8.data_ptr(), c.ks.data_ptr(), c.v8.data_ptr(), c.vs.data_ptr(),
        c.rs.data_ptr(), c.ctx.data_ptr(), B, M, Hq, Hkv, d, cap, c.x.max_ctx, 0.0, 0,
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["qwen_layer", "spec_verify", "r32"])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(name):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    # r32: 32 query rows per kv head (M = 4, GQA 8) over 6 sequences: row groups
    c = upload(WORKLOADS[name] if name != "r32" else
               custom("noalloc_r32", 6, 4, 16, 2, ("uniform", 200, 3000), outliers=True))
    ref = run(c).cpu().numpy()                  # kattn_decode, caller-owned workspace
    for _ in range(2):
        out = torch.full_like(c.q, float("nan"))
        assert _noalloc(c, out) == 0
        got = out.cpu().numpy()
        assert_f32_tolerance(got, ref)
        # the same kernel on the same inputs: deterministic to the byte
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.gpu
def test_noalloc_after_a_larger_call_leaks_nothing_into_a_smaller_one():
    # The shared array keeps everything the previous call wrote: its work
    # list, item count, packed queries and window partials.  A large call
    # (16 sequences, 5 draft columns, up to 9 windows each) followed by small
    # ones of another batch size, column count and GQA group must give the
    # bytes of kattn_decode with a freshly zeroed workspace.
    import torch
    import __graft_entry__
    __graft_entry__.build()
    big = upload(WORKLOADS["spec_verify"])
    small = [upload(custom("noalloc_small", 3, 1, 8, 2, ("uniform", 40, 1500), outliers=False)),
             upload(custom("noalloc_small_r32", 2, 4, 16, 2, ("uniform", 600, 1100),
                           outliers=True))]
    out_big = torch.full_like(big.q, float("nan"))
    assert _noalloc(big, out_big) == 0
    for c in small + [small[0]]:
        ref = run(c).cpu().numpy()              # fresh workspace, zeroed by torch
        out = torch.full_like(c.q, float("nan"))
        assert _noalloc(c, out) == 0
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    ref_big = run(big).cpu().numpy()
    assert np.array_equal(out_big.cpu().numpy().view(np.uint32), ref_big.view(np.uint32))


def test_noalloc_rejects_requests_beyond_its_scratch():
    # Checked on the host before any CUDA call: the pointers are never used.
    import __graft_entry__
    __graft_entry__.build()
    from int8_kv_decode_gb300 import _lib
    lib = _lib.load()
    fake = 0x100000
    st = lib.kattn_decode_noalloc(fake, fake, fake, fake, fake, fake, fake,
                                  4096, 8, 64, 8, 128, 1 << 20, 131072, 0.0, 0, fake, None)
    assert st == -4                               # KATTN_ERR_WORKSPACE
    need = lib.kattn_decode_workspace_size(4096, 8, 64, 131072)
    assert need > 16 * 1024 * 1024
