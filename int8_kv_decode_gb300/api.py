"""Python binding over the kattn C ABI (argument marshalling only).

Every function takes torch CUDA tensors, checks dtypes/shapes/contiguity,
and passes raw device pointers plus torch's current CUDA stream to the
library.  All computation happens in the library's CUDA kernels.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib

P_MODES = {"f32": 0, "bf16": 1, "e4m3": 2, "e4m3x448": 3, "e4m3x256": 4, "e4m3direct": 5}

# Device error bits (KATTN_DEVERR_* in kattn.h), as get_device_status returns them.
DEVERR_BAD_SEQUENCE = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_BAD_PAGE = 0x4


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def get_tiling() -> tuple:
    lib = _lib.load()
    c, bk = ctypes.c_int(), ctypes.c_int()
    lib.kattn_get_tiling(ctypes.byref(c), ctypes.byref(bk))
    return c.value, bk.value


def expf_constants() -> list:
    """The library's exact-mode exp constants: [K, C2, C0, C1, T[0..63]]."""
    lib = _lib.load()
    buf = (ctypes.c_double * 68)()
    _lib.check("kattn_expf_constants", lib.kattn_expf_constants(buf))
    return list(buf)


def decode_workspace_size(B: int, M: int, Hq: int, max_ctx: int) -> int:
    return int(_lib.load().kattn_decode_workspace_size(B, M, Hq, max_ctx))


def decode_launch_count(B: int, M: int, Hq: int, Hkv: int, max_ctx: int) -> int:
    """Kernels one fast-mode decode launches for these sizes on the current
    device (kattn_decode_launch_count)."""
    return int(_lib.load().kattn_decode_launch_count(B, M, Hq, Hkv, max_ctx))


def alloc_workspace(B: int, M: int, Hq: int, max_ctx: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for kattn_decode (allocated by torch, not the library)."""
    n = decode_workspace_size(B, M, Hq, max_ctx)
    if n == 0:
        raise ValueError("invalid sizes for a decode workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def quantize_kv(x: torch.Tensor, out_q: torch.Tensor, out_scale: torch.Tensor,
                dst_row0: int = 0) -> None:
    """x [n_rows][Hkv][d] float32 -> out_q [Hkv][cap][d] int8, out_scale [Hkv][cap]."""
    _need(x, torch.float32, "x", 3)
    _need(out_q, torch.int8, "out_q", 3)
    _need(out_scale, torch.float32, "out_scale", 2)
    n_rows, n_kv, d = x.shape
    cap = out_q.shape[1]
    if out_q.shape[0] != n_kv or out_q.shape[2] != d or tuple(out_scale.shape) != (n_kv, cap):
        raise ValueError("cache shapes do not match x")
    lib = _lib.load()
    _lib.check("kattn_quantize_kv", lib.kattn_quantize_kv(
        _ptr(x), n_rows, n_kv, d, n_kv * d, _ptr(out_q), _ptr(out_scale), dst_row0, cap,
        _stream(x.device)))


def quantize_kv_rows(x: torch.Tensor, dst_rows: torch.Tensor, out_q: torch.Tensor,
                     out_scale: torch.Tensor) -> None:
    """Append form: row r of x [n_rows][Hkv][d] goes to cache row dst_rows[r]."""
    _need(x, torch.float32, "x", 3)
    _need(dst_rows, torch.int64, "dst_rows", 1)
    _need(out_q, torch.int8, "out_q", 3)
    _need(out_scale, torch.float32, "out_scale", 2)
    n_rows, n_kv, d = x.shape
    cap = out_q.shape[1]
    if dst_rows.numel() != n_rows:
        raise ValueError("dst_rows must have one entry per row of x")
    if out_q.shape[0] != n_kv or out_q.shape[2] != d or tuple(out_scale.shape) != (n_kv, cap):
        raise ValueError("cache shapes do not match x")
    lib = _lib.load()
    _lib.check("kattn_quantize_kv_rows", lib.kattn_quantize_kv_rows(
        _ptr(x), n_rows, n_kv, d, n_kv * d, _ptr(dst_rows), _ptr(out_q), _ptr(out_scale), cap,
        _stream(x.device)))


def decode(q, k, k_scale, v, v_scale, row_start, ctx_len, max_ctx: int, *,
           out=None, p_mode=0, exact_mode=False, sm_scale: float = 0.0, workspace=None):
    """Decode attention; returns out [B][M][Hq][d] float32.

    q [B][M][Hq][d] f32; k, v [Hkv][cap][d] int8; k_scale, v_scale [Hkv][cap]
    f32; row_start [B] int64; ctx_len [B] int32 (all on the same CUDA device).
    p_mode: an int or a name of P_MODES -- "f32", "bf16", "e4m3", "e4m3x448",
    "e4m3x256", or "e4m3direct" (e4m3 P fed straight to the P.V MMA as one
    f16 operand p~ * v_scale; fast mode only).
    workspace: a zeroed uint8 tensor of decode_workspace_size(...) bytes
    (fast mode); allocated here with torch if None.  Exact mode needs none; a
    zeroed one of at least 256 bytes, if given, receives the device error bits.
    """
    _need(q, torch.float32, "q", 4)
    _need(k, torch.int8, "k", 3)
    _need(v, torch.int8, "v", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    _need(row_start, torch.int64, "row_start", 1)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    B, M, Hq, d = q.shape
    Hkv, cap, _ = k.shape
    if tuple(v.shape) != tuple(k.shape) or tuple(k_scale.shape) != (Hkv, cap) \
            or tuple(v_scale.shape) != (Hkv, cap):
        raise ValueError("k/v/scales shapes disagree")
    if row_start.numel() != B or ctx_len.numel() != B:
        raise ValueError("row_start / ctx_len must have B entries")
    mode = P_MODES.get(p_mode, p_mode) if isinstance(p_mode, str) else int(p_mode)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, torch.float32, "out", 4)
    ws_bytes = 0
    if not exact_mode and workspace is None:
        workspace = alloc_workspace(B, M, Hq, max_ctx, q.device)
    if workspace is not None:                 # exact mode: optional, for the error word
        _need(workspace, torch.uint8, "workspace", 1)
        ws_bytes = workspace.numel()
    lib = _lib.load()
    _lib.check("kattn_decode", lib.kattn_decode(
        _ptr(q), _ptr(k), _ptr(k_scale), _ptr(v), _ptr(v_scale), _ptr(row_start), _ptr(ctx_len),
        B, M, Hq, Hkv, d, cap, int(max_ctx), float(sm_scale), mode, 1 if exact_mode else 0,
        _ptr(out), _ptr(workspace), ws_bytes, _stream(q.device)))
    return out


def decode_paged(q, k, k_scale, v, v_scale, block_table, page_rows: int, ctx_len, max_ctx: int,
                 *, out=None, p_mode=0, exact_mode=False, sm_scale: float = 0.0, workspace=None):
    """Decode attention over a paged cache; returns out [B][M][Hq][d] float32.

    Key t of sequence b is row block_table[b][t // page_rows] * page_rows +
    t % page_rows of every kv-head plane of k, v [Hkv][cap][d] (int8) and
    k_scale, v_scale [Hkv][cap] (f32).  block_table: int32 [B][max_pages];
    page_rows: 32 * 2^k, dividing cap.  Otherwise as decode().
    """
    _need(q, torch.float32, "q", 4)
    _need(k, torch.int8, "k", 3)
    _need(v, torch.int8, "v", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    _need(block_table, torch.int32, "block_table", 2)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    B, M, Hq, d = q.shape
    Hkv, cap, _ = k.shape
    if tuple(v.shape) != tuple(k.shape) or tuple(k_scale.shape) != (Hkv, cap) \
            or tuple(v_scale.shape) != (Hkv, cap):
        raise ValueError("k/v/scales shapes disagree")
    if block_table.shape[0] != B or ctx_len.numel() != B:
        raise ValueError("block_table / ctx_len must have B rows")
    mode = P_MODES.get(p_mode, p_mode) if isinstance(p_mode, str) else int(p_mode)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, torch.float32, "out", 4)
    ws_bytes = 0
    if not exact_mode and workspace is None:
        workspace = alloc_workspace(B, M, Hq, max_ctx, q.device)
    if workspace is not None:                 # exact mode: optional, for the error word
        _need(workspace, torch.uint8, "workspace", 1)
        ws_bytes = workspace.numel()
    lib = _lib.load()
    _lib.check("kattn_decode_paged", lib.kattn_decode_paged(
        _ptr(q), _ptr(k), _ptr(k_scale), _ptr(v), _ptr(v_scale), _ptr(block_table),
        int(block_table.shape[1]), int(page_rows), _ptr(ctx_len), B, M, Hq, Hkv, d, cap,
        int(max_ctx), float(sm_scale), mode, 1 if exact_mode else 0, _ptr(out),
        _ptr(workspace), ws_bytes, _stream(q.device)))
    return out


def decode_append(q, k_new, v_new, dst_rows, k, k_scale, v, v_scale, row_start, ctx_len,
                  max_ctx: int, *, out=None, p_mode=0, sm_scale: float = 0.0, workspace=None):
    """Append rows k_new / v_new [n][Hkv][d] f32 at cache rows dst_rows [n]
    (int64), then decode (fast mode): one call of kattn_decode_append."""
    _need(q, torch.float32, "q", 4)
    _need(k_new, torch.float32, "k_new", 3)
    _need(v_new, torch.float32, "v_new", 3)
    _need(dst_rows, torch.int64, "dst_rows", 1)
    _need(k, torch.int8, "k", 3)
    _need(v, torch.int8, "v", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    _need(row_start, torch.int64, "row_start", 1)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    B, M, Hq, d = q.shape
    Hkv, cap, _ = k.shape
    n_new = k_new.shape[0]
    if tuple(v_new.shape) != tuple(k_new.shape) or dst_rows.numel() != n_new \
            or k_new.shape[1] != Hkv or k_new.shape[2] != d:
        raise ValueError("k_new / v_new / dst_rows shapes disagree with the cache")
    if tuple(v.shape) != tuple(k.shape) or tuple(k_scale.shape) != (Hkv, cap) \
            or tuple(v_scale.shape) != (Hkv, cap):
        raise ValueError("k/v/scales shapes disagree")
    mode = P_MODES.get(p_mode, p_mode) if isinstance(p_mode, str) else int(p_mode)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, torch.float32, "out", 4)
    if workspace is None:
        workspace = alloc_workspace(B, M, Hq, max_ctx, q.device)
    _need(workspace, torch.uint8, "workspace", 1)
    lib = _lib.load()
    _lib.check("kattn_decode_append", lib.kattn_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(dst_rows), n_new, Hkv * d, _ptr(k), _ptr(k_scale),
        _ptr(v), _ptr(v_scale), _ptr(row_start), _ptr(ctx_len), B, M, Hq, Hkv, d, cap,
        int(max_ctx), float(sm_scale), mode, _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(q.device)))
    return out


def decode_paged_append(q, k_new, v_new, dst_rows, k, k_scale, v, v_scale, block_table,
                        page_rows: int, ctx_len, max_ctx: int, *, out=None, p_mode=0,
                        sm_scale: float = 0.0, workspace=None):
    """Append rows k_new / v_new [n][Hkv][d] f32 at PHYSICAL pool rows
    dst_rows [n] (int64), then decode the paged cache (fast mode): one call of
    kattn_decode_paged_append.  Paging arguments as decode_paged()."""
    _need(q, torch.float32, "q", 4)
    _need(k_new, torch.float32, "k_new", 3)
    _need(v_new, torch.float32, "v_new", 3)
    _need(dst_rows, torch.int64, "dst_rows", 1)
    _need(k, torch.int8, "k", 3)
    _need(v, torch.int8, "v", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    _need(block_table, torch.int32, "block_table", 2)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    B, M, Hq, d = q.shape
    Hkv, cap, _ = k.shape
    n_new = k_new.shape[0]
    if tuple(v_new.shape) != tuple(k_new.shape) or dst_rows.numel() != n_new \
            or k_new.shape[1] != Hkv or k_new.shape[2] != d:
        raise ValueError("k_new / v_new / dst_rows shapes disagree with the cache")
    if tuple(v.shape) != tuple(k.shape) or tuple(k_scale.shape) != (Hkv, cap) \
            or tuple(v_scale.shape) != (Hkv, cap):
        raise ValueError("k/v/scales shapes disagree")
    if block_table.shape[0] != B or ctx_len.numel() != B:
        raise ValueError("block_table / ctx_len must have B rows")
    mode = P_MODES.get(p_mode, p_mode) if isinstance(p_mode, str) else int(p_mode)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, torch.float32, "out", 4)
    if workspace is None:
        workspace = alloc_workspace(B, M, Hq, max_ctx, q.device)
    _need(workspace, torch.uint8, "workspace", 1)
    lib = _lib.load()
    _lib.check("kattn_decode_paged_append", lib.kattn_decode_paged_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(dst_rows), n_new, Hkv * d, _ptr(k), _ptr(k_scale),
        _ptr(v), _ptr(v_scale), _ptr(block_table), int(block_table.shape[1]), int(page_rows),
        _ptr(ctx_len), B, M, Hq, Hkv, d, cap, int(max_ctx), float(sm_scale), mode, _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(q.device)))
    return out


WINDOW_KEYS = 512   # KATTN_WINDOW_KEYS: keys per window, the unit of a shard


def shard_partials_size(B: int, M: int, Hq: int, Hkv: int, win_per_shard: int) -> int:
    """Bytes of one shard's partials array (kattn_shard_partials_size)."""
    return int(_lib.load().kattn_shard_partials_size(B, M, Hq, Hkv, win_per_shard))


def partial_stride(R: int) -> int:
    """Floats per (sequence, window, kv head) partial: o[R][128], m[R], l[R],
    padded to a multiple of 4."""
    return R * 128 + (2 * R + 3) // 4 * 4


def decode_shard(q, k, k_scale, v, v_scale, row_start, ctx_len, max_ctx: int, shard: int,
                 win_per_shard: int, *, partials=None, p_mode=0, sm_scale: float = 0.0,
                 workspace=None):
    """Window partials of context-parallel shard `shard` (kattn_decode_shard).

    The cache k, v [Hkv][cap][d] (int8) and k_scale, v_scale [Hkv][cap] hold
    key t of sequence b, for the shard's keys t in [512 * shard * Ws,
    min(512 * (shard + 1) * Ws, ctx_len[b] + M - 1)), at row row_start[b] + t -
    512 * shard * Ws; ctx_len holds the global context lengths.  Returns
    partials float32 [B][Ws][Hkv][partial_stride(g * M)].
    """
    _need(q, torch.float32, "q", 4)
    _need(k, torch.int8, "k", 3)
    _need(v, torch.int8, "v", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    _need(row_start, torch.int64, "row_start", 1)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    B, M, Hq, d = q.shape
    Hkv, cap, _ = k.shape
    if tuple(v.shape) != tuple(k.shape) or tuple(k_scale.shape) != (Hkv, cap) \
            or tuple(v_scale.shape) != (Hkv, cap):
        raise ValueError("k/v/scales shapes disagree")
    if row_start.numel() != B or ctx_len.numel() != B:
        raise ValueError("row_start / ctx_len must have B entries")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    stride = partial_stride(Hq // Hkv * M)
    shape = (B, win_per_shard, Hkv, stride)
    if partials is None:
        partials = torch.empty(shape, dtype=torch.float32, device=q.device)
    else:
        _need(partials, torch.float32, "partials", 4)
        if tuple(partials.shape) != shape:
            raise ValueError(f"partials must have shape {shape}")
    if workspace is None:
        workspace = alloc_workspace(B, M, Hq, max_ctx, q.device)
    _need(workspace, torch.uint8, "workspace", 1)
    mode = P_MODES.get(p_mode, p_mode) if isinstance(p_mode, str) else int(p_mode)
    lib = _lib.load()
    _lib.check("kattn_decode_shard", lib.kattn_decode_shard(
        _ptr(q), _ptr(k), _ptr(k_scale), _ptr(v), _ptr(v_scale), _ptr(row_start), _ptr(ctx_len),
        B, M, Hq, Hkv, d, cap, int(max_ctx), int(shard), int(win_per_shard), float(sm_scale),
        mode, _ptr(partials), _ptr(workspace), workspace.numel(), _stream(q.device)))
    return partials


def merge_shards(partials, ctx_len, M: int, Hq: int, max_ctx: int, *, out=None, workspace=None):
    """Combine gathered shard partials [n_shards][B][Ws][Hkv][stride] into
    out [B][M][Hq][128] float32 (kattn_merge_shards)."""
    _need(partials, torch.float32, "partials", 5)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    n_shards, B, Ws, Hkv, stride = partials.shape
    if ctx_len.numel() != B:
        raise ValueError("ctx_len must have B entries")
    if Hq % Hkv != 0 or stride != partial_stride(Hq // Hkv * M):
        raise ValueError("partials do not match M, Hq")
    if out is None:
        out = torch.empty((B, M, Hq, 128), dtype=torch.float32, device=partials.device)
    else:
        _need(out, torch.float32, "out", 4)
        if tuple(out.shape) != (B, M, Hq, 128):
            raise ValueError("out must have shape [B][M][Hq][128]")
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=partials.device)
    _need(workspace, torch.uint8, "workspace", 1)
    lib = _lib.load()
    _lib.check("kattn_merge_shards", lib.kattn_merge_shards(
        _ptr(partials), _ptr(ctx_len), B, int(M), int(Hq), Hkv, 128, int(max_ctx), n_shards, Ws,
        _ptr(out), _ptr(workspace), workspace.numel(), _stream(partials.device)))
    return out


def hash_rows(x: torch.Tensor) -> torch.Tensor:
    """FNV-1a 64 of every row of x (a CUDA tensor whose last dimension is
    contiguous; rows = all leading indices).  Returns int64 [rows] holding
    the uint64 hash bits (kattn_hash_rows)."""
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    x2 = x.reshape(-1, x.shape[-1]) if x.dim() > 1 else x.reshape(1, -1)
    if x2.stride(-1) != 1:
        raise ValueError("the last dimension of x must be contiguous")
    out = torch.empty(x2.shape[0], dtype=torch.int64, device=x.device)
    row_bytes = x2.shape[1] * x2.element_size()
    stride = x2.stride(0) * x2.element_size()
    lib = _lib.load()
    _lib.check("kattn_hash_rows", lib.kattn_hash_rows(
        _ptr(x2), x2.shape[0], row_bytes, stride, _ptr(out), _stream(x.device)))
    return out


def qk_scores_debug(q, k, k_scale, row_start, ctx_len, max_ctx: int, *, scores=None,
                    want_q=False):
    """Integer QK scores [B][M][Hq][max_ctx + M - 1] (int32); entries t >= L_j
    keep their prior contents (filled with INT32_MIN when allocated here).
    With want_q, also returns (q_i8, q_scale)."""
    _need(q, torch.float32, "q", 4)
    _need(k, torch.int8, "k", 3)
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(row_start, torch.int64, "row_start", 1)
    _need(ctx_len, torch.int32, "ctx_len", 1)
    B, M, Hq, d = q.shape
    Hkv, cap, _ = k.shape
    width = int(max_ctx) + M - 1
    if scores is None:
        scores = torch.full((B, M, Hq, width), -2 ** 31, dtype=torch.int32, device=q.device)
    else:
        _need(scores, torch.int32, "scores", 4)
    q_i8 = q_scale = None
    if want_q:
        q_i8 = torch.zeros((B, M, Hq, d), dtype=torch.int8, device=q.device)
        q_scale = torch.zeros((B, M, Hq), dtype=torch.float32, device=q.device)
    lib = _lib.load()
    _lib.check("kattn_qk_scores_debug", lib.kattn_qk_scores_debug(
        _ptr(q), _ptr(k), _ptr(k_scale), _ptr(row_start), _ptr(ctx_len), B, M, Hq, Hkv, d, cap,
        int(max_ctx), _ptr(scores), _ptr(q_i8), _ptr(q_scale), _stream(q.device)))
    return (scores, q_i8, q_scale) if want_q else scores


def get_device_status(workspace: torch.Tensor) -> int:
    """Read and clear the device error bits of a decode workspace."""
    _need(workspace, torch.uint8, "workspace", 1)
    lib = _lib.load()
    err = ctypes.c_int(0)
    _lib.check("kattn_get_device_status", lib.kattn_get_device_status(
        _ptr(workspace), workspace.numel(), ctypes.byref(err), _stream(workspace.device)))
    return err.value
