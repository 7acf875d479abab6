"""C ABI checks that need no GPU: the library builds and loads, exports every
symbol include/kattn.h declares, and rejects bad arguments on the host before
anything is launched.  No test here passes validation, so nothing runs on a
device.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kattn.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from int8_kv_decode_gb300 import _lib
    return _lib.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kattn_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    from int8_kv_decode_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == names      # binding covers the header exactly


def test_status_strings(lib):
    assert lib.kattn_status_string(0) == b"KATTN_OK"
    assert lib.kattn_status_string(-3) == b"KATTN_ERR_MISALIGNED"
    assert lib.kattn_status_string(123) == b"KATTN_UNKNOWN_STATUS"


def test_tiling(lib):
    c, bk = ctypes.c_int(), ctypes.c_int()
    assert lib.kattn_get_tiling(ctypes.byref(c), ctypes.byref(bk)) == 0
    # the constants the oracle's rounded-P mirror is built with in the tests
    from helpers import BLOCK_BK, SPAN_C
    assert (c.value, bk.value) == (SPAN_C, BLOCK_BK) == (128, 32)
    assert lib.kattn_get_tiling(None, None) == 0


def test_workspace_size(lib):
    n = lib.kattn_decode_workspace_size(4, 1, 32, 8192)
    n8 = lib.kattn_decode_workspace_size(8, 1, 32, 8192)
    assert n > 4 * 32 * (128 + 2) * 4          # at least one partial per row
    assert n % 256 == 0
    assert 1.9 * n < n8 < 2.1 * n                # partials grow with the batch
    assert lib.kattn_decode_workspace_size(0, 1, 32, 8192) == 0
    assert lib.kattn_decode_workspace_size(1, 9, 32, 8192) == 0
    assert lib.kattn_decode_workspace_size(4, 5, 32, 8192) > n


def test_expf_constants_match_oracle(lib):
    # The library derives its constants in double-double arithmetic; the
    # oracle uses the decimal module.  Independent derivations must agree.
    from oracle import expf_tang as E
    buf = (ctypes.c_double * 68)()
    assert lib.kattn_expf_constants(buf) == 0
    got = list(buf)
    assert got[:4] == [E.K, E.C2, E.C0, E.C1]
    assert got[4:] == list(E.TABLE)
    assert lib.kattn_expf_constants(None) == -1


def _decode(lib, **kw):
    a = dict(q=64, k=64, ks=64, v=64, vs=64, rs=64, ctx=64, B=1, M=1, Hq=8, Hkv=2, d=128,
             cap=256, max_ctx=256, sm=0.0, p_mode=0, exact=0, out=64, ws=0, ws_bytes=0,
             stream=0)
    a.update(kw)
    return lib.kattn_decode(a["q"], a["k"], a["ks"], a["v"], a["vs"], a["rs"], a["ctx"],
                            a["B"], a["M"], a["Hq"], a["Hkv"], a["d"], a["cap"], a["max_ctx"],
                            a["sm"], a["p_mode"], a["exact"], a["out"], a["ws"], a["ws_bytes"],
                            a["stream"])


def test_decode_validation(lib):
    INVALID, UNSUP, MISAL, WS = -1, -2, -3, -4
    assert _decode(lib, q=0) == INVALID
    assert _decode(lib, Hq=6, Hkv=4) == INVALID
    assert _decode(lib, d=64) == UNSUP
    assert _decode(lib, M=9) == UNSUP
    assert _decode(lib, Hq=128, Hkv=1, M=1) == UNSUP       # g*M = 128 > 64
    assert _decode(lib, q=0x1008) == MISAL
    assert _decode(lib, k=0x1004) == MISAL
    assert _decode(lib, rs=0x1004) == MISAL
    assert _decode(lib, p_mode=6) == INVALID
    assert _decode(lib, p_mode=-1) == INVALID
    assert _decode(lib, p_mode=5, exact=1) == INVALID     # e4m3 direct: fast mode only
    assert _decode(lib, exact=2) == INVALID
    assert _decode(lib, sm=float("nan")) == INVALID
    assert _decode(lib, max_ctx=0) == INVALID
    assert _decode(lib, cap=0) == INVALID
    assert _decode(lib, ws=0) == WS                        # fast mode needs one
    assert _decode(lib, ws=0x1100, ws_bytes=16) == WS      # too small
    assert _decode(lib, ws=0x1010, ws_bytes=1 << 30) == WS  # not 256-aligned
    assert _decode(lib, B=0) == 0                          # empty batch: no-op


def _decode_paged(lib, **kw):
    a = dict(q=64, k=64, ks=64, v=64, vs=64, bt=64, max_pages=8, page=32, ctx=64, B=1, M=1,
             Hq=8, Hkv=2, d=128, cap=256, max_ctx=256, sm=0.0, p_mode=0, exact=0, out=64,
             ws=0, ws_bytes=0, stream=0)
    a.update(kw)
    return lib.kattn_decode_paged(a["q"], a["k"], a["ks"], a["v"], a["vs"], a["bt"],
                                  a["max_pages"], a["page"], a["ctx"], a["B"], a["M"], a["Hq"],
                                  a["Hkv"], a["d"], a["cap"], a["max_ctx"], a["sm"],
                                  a["p_mode"], a["exact"], a["out"], a["ws"], a["ws_bytes"],
                                  a["stream"])


def test_decode_paged_validation(lib):
    # Checked on the host before any CUDA call: the pointers are never used.
    INVALID, UNSUP, MISAL, WS = -1, -2, -3, -4
    assert _decode_paged(lib, bt=0) == INVALID
    assert _decode_paged(lib, bt=0x1002) == MISAL          # int32 table
    assert _decode_paged(lib, max_pages=0) == INVALID
    assert _decode_paged(lib, page=0) == INVALID
    assert _decode_paged(lib, page=16) == UNSUP            # a 32-key block would cross pages
    assert _decode_paged(lib, page=96, cap=288) == UNSUP   # not a power of two
    assert _decode_paged(lib, page=64, cap=224) == INVALID  # pages do not tile the planes
    assert _decode_paged(lib, d=64) == UNSUP
    assert _decode_paged(lib, p_mode=6) == INVALID
    assert _decode_paged(lib, p_mode=5, exact=1) == INVALID
    assert _decode_paged(lib, ws=0) == WS
    assert _decode_paged(lib, B=0) == 0


def _paged_append(lib, **kw):
    a = dict(q=64, kn=64, vn=64, dst=64, n=2, stride=256, k=64, ks=64, v=64, vs=64, bt=64,
             max_pages=8, page=32, ctx=64, B=1, M=1, Hq=8, Hkv=2, d=128, cap=256, max_ctx=256,
             sm=0.0, p_mode=0, out=64, ws=0, ws_bytes=0, stream=0)
    a.update(kw)
    return lib.kattn_decode_paged_append(
        a["q"], a["kn"], a["vn"], a["dst"], a["n"], a["stride"], a["k"], a["ks"], a["v"],
        a["vs"], a["bt"], a["max_pages"], a["page"], a["ctx"], a["B"], a["M"], a["Hq"], a["Hkv"],
        a["d"], a["cap"], a["max_ctx"], a["sm"], a["p_mode"], a["out"], a["ws"], a["ws_bytes"],
        a["stream"])


def test_decode_paged_append_validation(lib):
    # Checked on the host before any CUDA call: the pointers are never used.
    INVALID, UNSUP, MISAL, WS = -1, -2, -3, -4
    assert _paged_append(lib, page=16) == UNSUP
    assert _paged_append(lib, page=64, cap=224) == INVALID
    assert _paged_append(lib, bt=0x1002) == MISAL
    assert _paged_append(lib, n=-1) == INVALID
    assert _paged_append(lib, stride=255) == INVALID          # < Hkv * d
    assert _paged_append(lib, kn=0) == INVALID
    assert _paged_append(lib, dst=0x1004) == MISAL            # int64 rows
    assert _paged_append(lib, stride=258) == MISAL
    assert _paged_append(lib, p_mode=6) == INVALID
    assert _paged_append(lib, ws=0) == WS
    assert _paged_append(lib, B=0, n=0) == 0                  # nothing at all: no-op


def test_quantize_validation(lib):
    f = lib.kattn_quantize_kv
    assert f(64, 4, 2, 64, 256, 64, 64, 0, 8, 0) == -2       # d != 128
    assert f(64, 4, 2, 128, 255, 64, 64, 0, 8, 0) == -1      # stride < n_kv*d
    assert f(64, 4, 2, 128, 258, 64, 64, 0, 8, 0) == -3      # stride not /4
    assert f(64, 4, 2, 128, 256, 64, 64, 6, 8, 0) == -1      # dst_row0 + n > cap
    assert f(0, 4, 2, 128, 256, 64, 64, 0, 8, 0) == -1       # null x
    assert f(64, 0, 2, 128, 256, 64, 64, 0, 8, 0) == 0       # no rows: no-op


def test_qk_debug_validation(lib):
    f = lib.kattn_qk_scores_debug
    assert f(64, 64, 64, 64, 64, 1, 1, 8, 2, 128, 256, 256, 0, 0, 0, 0) == -1   # scores null
    assert f(64, 64, 64, 64, 64, 1, 1, 8, 2, 128, 256, 256, 0x1002, 0, 0, 0) == -3
    assert f(64, 64, 64, 64, 64, 1, 1, 8, 2, 96, 256, 256, 64, 0, 0, 0) == -2


def test_device_status_validation(lib):
    err = ctypes.c_int()
    assert lib.kattn_get_device_status(None, 1024, ctypes.byref(err), None) == -1
    assert lib.kattn_get_device_status(0x1010, 1024, ctypes.byref(err), None) == -4


def _decode_shard(lib, **kw):
    a = dict(q=64, k=64, ks=64, v=64, vs=64, rs=64, ctx=64, B=1, M=1, Hq=8, Hkv=2, d=128,
             cap=256, max_ctx=2048, shard=0, ws_per=2, sm=0.0, p_mode=0, part=64, ws=0,
             ws_bytes=0, stream=0)
    a.update(kw)
    return lib.kattn_decode_shard(a["q"], a["k"], a["ks"], a["v"], a["vs"], a["rs"], a["ctx"],
                                  a["B"], a["M"], a["Hq"], a["Hkv"], a["d"], a["cap"],
                                  a["max_ctx"], a["shard"], a["ws_per"], a["sm"], a["p_mode"],
                                  a["part"], a["ws"], a["ws_bytes"], a["stream"])


def _merge_shards(lib, **kw):
    a = dict(part=64, ctx=64, B=1, M=1, Hq=8, Hkv=2, d=128, max_ctx=2048, n=2, ws_per=2,
             out=64, ws=0x1000, ws_bytes=0, stream=0)
    a.update(kw)
    return lib.kattn_merge_shards(a["part"], a["ctx"], a["B"], a["M"], a["Hq"], a["Hkv"],
                                  a["d"], a["max_ctx"], a["n"], a["ws_per"], a["out"], a["ws"],
                                  a["ws_bytes"], a["stream"])


def test_shard_validation(lib):
    # Checked on the host before any CUDA call: the pointers are never used.
    INVALID, UNSUP, MISAL, WS = -1, -2, -3, -4
    assert _decode_shard(lib, shard=-1) == INVALID
    assert _decode_shard(lib, ws_per=0) == INVALID
    assert _decode_shard(lib, shard=1 << 20, ws_per=1 << 10) == INVALID   # keys beyond int32
    assert _decode_shard(lib, part=0) == INVALID
    assert _decode_shard(lib, part=0x1008) == MISAL
    assert _decode_shard(lib, d=64) == UNSUP
    assert _decode_shard(lib, p_mode=6) == INVALID
    assert _decode_shard(lib, ws=0) == WS
    assert _decode_shard(lib, B=0) == 0
    assert _merge_shards(lib, n=0) == INVALID
    assert _merge_shards(lib, ws_per=0) == INVALID
    assert _merge_shards(lib, d=64) == UNSUP
    assert _merge_shards(lib, M=9) == UNSUP
    assert _merge_shards(lib, part=0x1004) == MISAL
    assert _merge_shards(lib, out=0) == INVALID
    assert _merge_shards(lib, ws=0x1000, ws_bytes=128) == WS               # < 256 bytes
    assert _merge_shards(lib, ws=0x1010, ws_bytes=256) == WS               # not 256-aligned
    assert _merge_shards(lib, B=0) == 0


def test_shard_partials_size(lib):
    # [B][Ws][Hkv][stride] float32, stride = R*128 + (2R rounded up to 4)
    assert lib.kattn_shard_partials_size(3, 1, 8, 2, 5) == 3 * 5 * 2 * (4 * 128 + 8) * 4
    assert lib.kattn_shard_partials_size(2, 5, 32, 4, 1) == 2 * 4 * (40 * 128 + 80) * 4
    assert lib.kattn_shard_partials_size(2, 9, 32, 4, 1) == 0
    assert lib.kattn_shard_partials_size(2, 1, 6, 4, 1) == 0
    from int8_kv_decode_gb300 import api
    assert api.partial_stride(40) == 40 * 128 + 80
    assert api.partial_stride(3) == 3 * 128 + 8


def test_window_constant_matches_header():
    from int8_kv_decode_gb300 import api
    text = open(HEADER, encoding="utf-8").read()
    assert int(re.search(r"#define KATTN_WINDOW_KEYS (\d+)", text).group(1)) == api.WINDOW_KEYS


def test_device_error_bits_match_header():
    from int8_kv_decode_gb300 import api
    text = open(HEADER, encoding="utf-8").read()
    for name in ("BAD_SEQUENCE", "TIMEOUT", "BAD_PAGE"):
        val = int(re.search(rf"#define KATTN_DEVERR_{name} (0x[0-9a-f]+)u", text).group(1), 16)
        assert getattr(api, f"DEVERR_{name}") == val, name


def test_exact_mode_workspace_validation(lib):
    # exact mode: the workspace is optional, but one that is given must hold
    # the 256-byte error word and be 256-byte aligned
    WS = -4
    assert _decode(lib, exact=1, ws=0x1010, ws_bytes=256) == WS
    assert _decode(lib, exact=1, ws=0x1100, ws_bytes=128) == WS


def test_launch_count_validation(lib):
    f = lib.kattn_decode_launch_count
    assert f(0, 1, 32, 4, 1024) == 0          # no sequences
    assert f(4, 9, 32, 4, 1024) == 0          # M > KATTN_MAX_M
    assert f(4, 1, 30, 4, 1024) == 0          # Hq not a multiple of Hkv
    assert f(4, 1, 32, 4, 0) == 0
    assert f(1, 1, 8, 2, 256) == 2            # one window: packing + split pass, no merge
    assert f(4096, 1, 32, 4, 8192) == 4       # work list launch and merge launch
