"""ctypes loader for libkattn.so (the C ABI declared in include/kattn.h).

The library is required: importing a compute entry point without it raises.
There is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkattn.so")

c_int, c_int64, c_size_t, c_float, c_void_p = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                               ctypes.c_float, ctypes.c_void_p)

# name -> (restype, argtypes); mirrors include/kattn.h one to one.
SIGNATURES = {
    "kattn_status_string": (ctypes.c_char_p, [c_int]),
    "kattn_get_tiling": (c_int, [ctypes.POINTER(c_int), ctypes.POINTER(c_int)]),
    "kattn_decode_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "kattn_decode_launch_count": (c_int, [c_int, c_int, c_int, c_int, c_int]),
    "kattn_quantize_kv": (c_int, [c_void_p, c_int, c_int, c_int, c_int64, c_void_p, c_void_p,
                                  c_int64, c_int, c_void_p]),
    "kattn_quantize_kv_rows": (c_int, [c_void_p, c_int, c_int, c_int, c_int64, c_void_p,
                                       c_void_p, c_void_p, c_int, c_void_p]),
    "kattn_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                             c_float, c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "kattn_decode_paged": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_int, c_int, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                   c_int, c_int, c_float, c_int, c_int, c_void_p, c_void_p,
                                   c_size_t, c_void_p]),
    "kattn_decode_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int64,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                    c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "kattn_decode_paged_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int64,
                                          c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                          c_int, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                          c_int, c_int, c_float, c_int, c_void_p, c_void_p,
                                          c_size_t, c_void_p]),
    "kattn_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                     c_int, c_int, c_float, c_int, c_void_p, c_void_p]),
    "kattn_shard_partials_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "kattn_decode_shard": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                   c_int, c_int, c_float, c_int, c_void_p, c_void_p, c_size_t,
                                   c_void_p]),
    "kattn_merge_shards": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                   c_int, c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    "kattn_qk_scores_debug": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                      c_int, c_int, c_int, c_int, c_int, c_int, c_void_p,
                                      c_void_p, c_void_p, c_void_p]),
    "kattn_expf_constants": (c_int, [ctypes.POINTER(ctypes.c_double)]),
    "kattn_hash_rows": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p]),
    "kattn_get_device_status": (c_int, [c_void_p, c_size_t, ctypes.POINTER(c_int), c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkattn.so once and attach the signatures.  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libkattn.so not found at {path}: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class KattnError(RuntimeError):
    """A kattn entry point returned a non-zero status."""

    def __init__(self, fn: str, status: int):
        name = load().kattn_status_string(status).decode()
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != 0:
        raise KattnError(fn, status)
