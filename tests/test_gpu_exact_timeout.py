"""Exact mode's bounded waits, made to run out on purpose.

The exact-mode kernel runs three thread groups per query row (two producer
groups and the consumers) that hand chunks of keys and running maxima to each
other through shared-memory barriers; every wait for a hand-off is bounded,
and one that runs out leaves the row NaN and sets KATTN_DEVERR_TIMEOUT in the
workspace's error word.  To exercise that path
without any wait that could block, this test loads a separate build of the
library (build.py, build_exact_timeout_variant) in which the waits give up
after 0 polls: every wait runs out at once, deterministically.  The test
checks that the call returns, every row is NaN, the error bit is set, and the
GPU context is still usable: the ordinary library then decodes the same
inputs bit-exactly against the oracle.
"""

import ctypes

import numpy as np
import pytest

from helpers import bits, custom, oracle_decode, run, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spin0_lib():
    from int8_kv_decode_gb300 import _lib, build
    path = build.build_exact_timeout_variant()
    lib = ctypes.CDLL(path)                       # its own handle: not the package's library
    for name in ("kattn_decode", "kattn_get_device_status"):
        res, args = _lib.SIGNATURES[name]
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


@pytest.mark.parametrize("ctx", [200, 1500])       # 2 and 12 chunks of 128 keys
def test_exact_mode_waits_that_run_out_give_nan_rows_and_a_timeout_flag(spin0_lib, ctx):
    import torch
    import int8_kv_decode_gb300 as K
    c = upload(custom(f"timeout_{ctx}", 2, 2, 8, 2, ctx, outliers=False))
    B, M, Hq, d = c.q.shape
    Hkv, cap, _ = c.k8.shape
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(c.q)
    st = spin0_lib.kattn_decode(
        c.q.data_ptr(), c.k8.data_ptr(), c.ks.data_ptr(), c.v8.data_ptr(), c.vs.data_ptr(),
        c.rs.data_ptr(), c.ctx.data_ptr(), B, M, Hq, Hkv, d, cap, c.x.max_ctx, 0.0, 0, 1,
        out.data_ptr(), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    err = ctypes.c_int()
    assert spin0_lib.kattn_get_device_status(ws.data_ptr(), ws.numel(), ctypes.byref(err),
                                             torch.cuda.current_stream().cuda_stream) == 0
    assert err.value == K.DEVERR_TIMEOUT
    # the context is unharmed: the library proper, exact mode, bit for bit
    ws2 = torch.zeros(256, dtype=torch.uint8, device="cuda")
    good = run(c, exact_mode=True, workspace=ws2).cpu().numpy()
    assert np.array_equal(bits(good), bits(oracle_decode(c, mode="exact")))
    assert K.get_device_status(ws2) == 0
