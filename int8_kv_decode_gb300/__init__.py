"""int8-KV decode attention for NVIDIA GB300 (sm_103a).

The compute lives in libkattn.so (hand-written CUDA kernels behind the C ABI
in include/kattn.h); this package is a thin torch-facing binding.
"""

from .api import (  # noqa: F401
    DEVERR_BAD_PAGE,
    DEVERR_BAD_SEQUENCE,
    DEVERR_TIMEOUT,
    P_MODES,
    WINDOW_KEYS,
    alloc_workspace,
    decode,
    decode_append,
    decode_launch_count,
    decode_paged,
    decode_paged_append,
    decode_shard,
    decode_workspace_size,
    expf_constants,
    get_device_status,
    get_tiling,
    hash_rows,
    merge_shards,
    partial_stride,
    qk_scores_debug,
    quantize_kv,
    quantize_kv_rows,
    shard_partials_size,
)
from ._lib import KattnError, LIB_PATH, load  # noqa: F401
