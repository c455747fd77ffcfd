"""Thin ctypes binding of libsa.so (include/sa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libsa.so.  torch supplies device memory and streams.  There is no
fallback: if the library cannot be loaded, or a call returns an error status,
a ``RuntimeError`` is raised.

The C entry points are exposed under their C names (``sa_sparse_attn_fwd``,
``sa_topk_mask_shape``, ``sa_build_topk_mask`` ...) taking raw pointers and
sizes, and wrapped by tensor-level helpers ``sparse_attn``,
``topk_mask_shape`` and ``build_topk_mask``.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SA_OK = 0
_STATUS = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_SHAPE", 3: "SA_ERR_ALIGNMENT",
           4: "SA_ERR_WORKSPACE", 5: "SA_ERR_UNSUPPORTED_DEVICE", 6: "SA_ERR_CUDA"}

EXPORTS = ("sa_status_string", "sa_sparse_attn_num_splits", "sa_sparse_attn_workspace_size",
           "sa_sparse_attn_fwd", "sa_sparse_attn_fwd_splits", "sa_topk_mask_shape",
           "sa_build_topk_mask", "sa_device_error", "sa_sparse_attn_fwd_static_ws",
           "sa_sparse_attn_launch_count", "sa_selftest_wait_timeout", "sa_selftest_wait_drain", "sa_sparse_attn_fwd_topk_length",
           "sa_masked_dense_attn_fwd", "sa_masked_dense_attn_workspace_size", "sa_masked_dense_attn_launch_count",
           "sa_sparse_attn_fwd_fp8", "sa_sparse_attn_fp8_launch_count", "sa_build_topk_mask_window",
           "sa_masked_dense_attn_fwd_window", "sa_topk_mask_chunk_rows", "sa_topk_masked_attn_fwd",
           "sa_topk_masked_attn_workspace_size", "sa_sparse_attn_fwd_extra", "sa_sparse_attn_fwd_fp8_extra",
           "sa_probe_row_gather")

_lock = threading.Lock()
_lib = None


class SAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {_STATUS.get(code, code)}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libsa.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run deepseek_top_sparse_gb300.build.build()")
        lib = ctypes.CDLL(path)
        p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.sa_status_string.argtypes = [i32]
        lib.sa_status_string.restype = ctypes.c_char_p
        lib.sa_sparse_attn_num_splits.argtypes = [i64] * 5
        lib.sa_sparse_attn_num_splits.restype = i32
        lib.sa_sparse_attn_launch_count.argtypes = [i64] * 5 + [i32]
        lib.sa_sparse_attn_launch_count.restype = i32
        lib.sa_sparse_attn_workspace_size.argtypes = [i64] * 5 + [i32]
        lib.sa_sparse_attn_workspace_size.restype = sz
        lib.sa_sparse_attn_fwd.argtypes = [p, p, p, p, ctypes.c_float, p] + [i64] * 6 + [p, sz, p]
        lib.sa_sparse_attn_fwd.restype = i32
        lib.sa_sparse_attn_fwd_splits.argtypes = [p, p, p, p, ctypes.c_float, p] + [i64] * 6 + [i32, p, sz, p]
        lib.sa_sparse_attn_fwd_splits.restype = i32
        lib.sa_sparse_attn_fwd_topk_length.argtypes = [p, p, p, p, p, ctypes.c_float, p] + [i64] * 6 + [i32, p, sz, p]
        lib.sa_sparse_attn_fwd_topk_length.restype = i32
        lib.sa_topk_mask_shape.argtypes = [i64, i64, i64, i32, p]
        lib.sa_topk_mask_shape.restype = i32
        lib.sa_build_topk_mask.argtypes = [p, i64, p, i64, i64, i64, i64, p, p, p, p]
        lib.sa_build_topk_mask.restype = i32
        lib.sa_sparse_attn_fwd_static_ws.argtypes = [p, p, p, p, ctypes.c_float, p] + [i64] * 6 + [i32, p]
        lib.sa_sparse_attn_fwd_static_ws.restype = i32
        lib.sa_masked_dense_attn_fwd.argtypes = [p, p, p, p, i64, i64, i32, ctypes.c_float, p] + [i64] * 5 + \
            [i32, p, sz, p]
        lib.sa_masked_dense_attn_fwd.restype = i32
        lib.sa_masked_dense_attn_workspace_size.argtypes = [i64] * 5 + [i32]
        lib.sa_masked_dense_attn_workspace_size.restype = sz
        lib.sa_masked_dense_attn_launch_count.argtypes = [i64] * 5 + [i32]
        lib.sa_masked_dense_attn_launch_count.restype = i32
        lib.sa_sparse_attn_fwd_fp8.argtypes = [p, p, p, p, p, ctypes.c_float, p] + [i64] * 5 + [i32, p, sz, p]
        lib.sa_sparse_attn_fwd_fp8.restype = i32
        lib.sa_sparse_attn_fwd_extra.argtypes = [p, p, p, p, p, p, p, p, ctypes.c_float, p] + [i64] * 8 + [i32, p, sz, p]
        lib.sa_sparse_attn_fwd_extra.restype = i32
        lib.sa_sparse_attn_fwd_fp8_extra.argtypes = ([p, p, p, p, p, p, p, p, ctypes.c_float, p] + [i64] * 7 +
                                                     [i32, p, sz, p])
        lib.sa_sparse_attn_fwd_fp8_extra.restype = i32
        lib.sa_sparse_attn_fp8_launch_count.argtypes = [i64] * 4 + [i32]
        lib.sa_sparse_attn_fp8_launch_count.restype = i32
        lib.sa_build_topk_mask_window.argtypes = [p, i64, p, i64, i64, i64, i64, i64, p, p, p, p, p]
        lib.sa_build_topk_mask_window.restype = i32
        lib.sa_masked_dense_attn_fwd_window.argtypes = [p, p, p, p, i64, i64, i32, p, ctypes.c_float, p] + \
            [i64] * 7 + [i32, p, sz, p]
        lib.sa_masked_dense_attn_fwd_window.restype = i32
        lib.sa_topk_mask_chunk_rows.argtypes = [i64, i64, i64, i32, i64]
        lib.sa_topk_mask_chunk_rows.restype = i64
        lib.sa_topk_masked_attn_fwd.argtypes = [p, p, p, p, i64, p, p, p, ctypes.c_float, p] + [i64] * 8 + \
            [p, sz, p, sz, p]
        lib.sa_topk_masked_attn_fwd.restype = i32
        lib.sa_topk_masked_attn_workspace_size.argtypes = [i64] * 6 + [i32, i64]
        lib.sa_topk_masked_attn_workspace_size.restype = sz
        lib.sa_selftest_wait_timeout.argtypes = [ctypes.c_longlong]
        lib.sa_selftest_wait_timeout.restype = i32
        lib.sa_selftest_wait_drain.argtypes = [i32, ctypes.c_longlong, ctypes.POINTER(ctypes.c_float)]
        lib.sa_selftest_wait_drain.restype = i32
        lib.sa_probe_row_gather.argtypes = [p, i64, i64, i64, p, i64, i64, p]
        lib.sa_probe_row_gather.restype = i32
        lib.sa_device_error.argtypes = [i32]
        lib.sa_device_error.restype = i32
        _lib = lib
        return lib


# ------------------------------------------------------------------ C names

def sa_status_string(code: int) -> str:
    return load().sa_status_string(int(code)).decode()


def sa_sparse_attn_num_splits(B, S, H, D, K) -> int:
    return int(load().sa_sparse_attn_num_splits(B, S, H, D, K))


def sa_sparse_attn_launch_count(B, S, H, D, K, num_splits=0) -> int:
    return int(load().sa_sparse_attn_launch_count(B, S, H, D, K, num_splits))


def sa_sparse_attn_workspace_size(B, S, H, D, K, num_splits=0) -> int:
    return int(load().sa_sparse_attn_workspace_size(B, S, H, D, K, num_splits))


def sa_sparse_attn_fwd(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T, K,
                       workspace, workspace_bytes, stream) -> int:
    return int(load().sa_sparse_attn_fwd(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T, K,
                                          workspace, workspace_bytes, stream))


def sa_sparse_attn_fwd_splits(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T, K,
                              num_splits, workspace, workspace_bytes, stream) -> int:
    return int(load().sa_sparse_attn_fwd_splits(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T,
                                                 K, num_splits, workspace, workspace_bytes, stream))


def sa_sparse_attn_fwd_topk_length(q, kv, attn_sink, topk_idxs, topk_length, softmax_scale, o, B, S, H, D, T, K,
                                   num_splits, workspace, workspace_bytes, stream) -> int:
    return int(load().sa_sparse_attn_fwd_topk_length(q, kv, attn_sink, topk_idxs, topk_length, softmax_scale, o,
                                                      B, S, H, D, T, K, num_splits, workspace, workspace_bytes,
                                                      stream))


def sa_sparse_attn_fwd_static_ws(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T, K, num_splits,
                                 stream) -> int:
    """Allocation-free sparse_attn (workspace inside the library); same
    arguments as sa_sparse_attn_fwd_splits without the workspace pair."""
    return int(load().sa_sparse_attn_fwd_static_ws(q, kv, attn_sink, topk_idxs, softmax_scale, o, B, S, H, D, T, K,
                                                   num_splits, stream))


def sa_sparse_attn_fwd_fp8(q, kv_fp8, attn_sink, topk_idxs, topk_length, softmax_scale, o, B, S, H, T, K,
                           num_splits, workspace, workspace_bytes, stream) -> int:
    return int(load().sa_sparse_attn_fwd_fp8(q, kv_fp8, attn_sink, topk_idxs, topk_length, softmax_scale, o, B, S, H,
                                              T, K, num_splits, workspace, workspace_bytes, stream))


def sa_sparse_attn_fp8_launch_count(B, S, H, K, num_splits=0) -> int:
    return int(load().sa_sparse_attn_fp8_launch_count(B, S, H, K, num_splits))


def sa_masked_dense_attn_workspace_size(B, S, H, D, T, num_splits=0) -> int:
    return int(load().sa_masked_dense_attn_workspace_size(B, S, H, D, T, num_splits))


def sa_masked_dense_attn_launch_count(B, S, H, D, T, num_splits=0) -> int:
    return int(load().sa_masked_dense_attn_launch_count(B, S, H, D, T, num_splits))


def sa_masked_dense_attn_fwd(q, kv, attn_sink, mask, mask_rows, mask_words, key_start_word, softmax_scale, o,
                             B, S, H, D, T, num_splits, workspace, workspace_bytes, stream) -> int:
    return int(load().sa_masked_dense_attn_fwd(q, kv, attn_sink, mask, mask_rows, mask_words, key_start_word,
                                                softmax_scale, o, B, S, H, D, T, num_splits, workspace,
                                                workspace_bytes, stream))


def sa_topk_mask_shape(batch, max_query_len, max_key_len, reserve_key_starts_word) -> tuple[int, int, int]:
    out = (ctypes.c_int64 * 3)()
    rc = load().sa_topk_mask_shape(batch, max_query_len, max_key_len, int(bool(reserve_key_starts_word)), out)
    if rc != SA_OK:
        raise SAError("sa_topk_mask_shape", rc)
    return int(out[0]), int(out[1]), int(out[2])


def sa_build_topk_mask(topk, topk_rows, cu_q_lens, B, max_q_len, max_key_len, K, key_starts, mask,
                       mask_shape, stream) -> int:
    shp = (ctypes.c_int64 * 3)(*[int(v) for v in mask_shape])
    return int(load().sa_build_topk_mask(topk, topk_rows, cu_q_lens, B, max_q_len, max_key_len, K, key_starts,
                                         mask, shp, stream))


def sa_build_topk_mask_window(topk, topk_rows, cu_q_lens, B, q0, q_rows, max_key_len, K, key_starts, key_ends,
                              mask, mask_shape, stream) -> int:
    shp = (ctypes.c_int64 * 3)(*[int(v) for v in mask_shape])
    return int(load().sa_build_topk_mask_window(topk, topk_rows, cu_q_lens, B, q0, q_rows, max_key_len, K,
                                                 key_starts, key_ends, mask, shp, stream))


def sa_masked_dense_attn_fwd_window(q, kv, attn_sink, mask, mask_rows, mask_words, key_start_word, key_ends,
                                    softmax_scale, o, B, S_total, q0, S, H, D, T, num_splits, workspace,
                                    workspace_bytes, stream) -> int:
    return int(load().sa_masked_dense_attn_fwd_window(q, kv, attn_sink, mask, mask_rows, mask_words, key_start_word,
                                                       key_ends, softmax_scale, o, B, S_total, q0, S, H, D, T,
                                                       num_splits, workspace, workspace_bytes, stream))


def sa_topk_mask_chunk_rows(batch, max_query_len, max_key_len, reserve_key_starts_word, cap_bytes=0) -> int:
    return int(load().sa_topk_mask_chunk_rows(batch, max_query_len, max_key_len, int(bool(reserve_key_starts_word)),
                                              cap_bytes))


def sa_topk_masked_attn_fwd(q, kv, attn_sink, topk, topk_rows, cu_q_lens, key_starts, key_ends, softmax_scale, o, B,
                            max_q_len, H, D, T, max_key_len, K, cap_bytes, mask_buf, mask_buf_bytes, workspace,
                            workspace_bytes, stream) -> int:
    return int(load().sa_topk_masked_attn_fwd(q, kv, attn_sink, topk, topk_rows, cu_q_lens, key_starts, key_ends,
                                               softmax_scale, o, B, max_q_len, H, D, T, max_key_len, K, cap_bytes,
                                               mask_buf, mask_buf_bytes, workspace, workspace_bytes, stream))


def sa_topk_masked_attn_workspace_size(B, max_q_len, H, D, T, max_key_len, reserve_key_starts_word,
                                       cap_bytes=0) -> int:
    return int(load().sa_topk_masked_attn_workspace_size(B, max_q_len, H, D, T, max_key_len,
                                                          int(bool(reserve_key_starts_word)), cap_bytes))


def sa_selftest_wait_timeout(max_cycles: int) -> int:
    return int(load().sa_selftest_wait_timeout(int(max_cycles)))


def sa_selftest_wait_drain(ctas: int, first_cycles: int) -> tuple[int, float]:
    """(code, elapsed ms) of the fast-drain self-test (see include/sa.h)."""
    ms = ctypes.c_float(0.0)
    code = int(load().sa_selftest_wait_drain(int(ctas), int(first_cycles), ctypes.byref(ms)))
    return code, float(ms.value)


def sa_probe_row_gather(table, rows, row_bytes, part_bytes, idx, ctas, tiles, stream) -> int:
    return int(load().sa_probe_row_gather(table, rows, row_bytes, part_bytes, idx, ctas, tiles, stream))


def sa_device_error(clear: bool = True) -> int:
    return int(load().sa_device_error(int(bool(clear))))


# ------------------------------------------------------------------ tensor helpers

def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else int(t.data_ptr())


def _check(fn: str, rc: int):
    if rc != SA_OK:
        raise SAError(fn, rc)


def probe_row_gather(table: torch.Tensor, row_bytes: int, part_bytes: int, idx: torch.Tensor, ctas: int,
                     tiles: int, stream=None) -> None:
    """Enqueue the random-row gather probe (include/sa.h): `ctas` CTAs copy
    `tiles` 32 KB tiles each of the first part_bytes of the rows of `table`
    (a contiguous CUDA uint8 tensor of whole rows) that idx picks."""
    if table.dtype != torch.uint8 or not table.is_cuda or not table.is_contiguous():
        raise ValueError("table must be a contiguous CUDA uint8 tensor")
    if idx.dtype != torch.int32 or not idx.is_cuda or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous CUDA int32 tensor")
    if row_bytes <= 0 or table.numel() % row_bytes != 0 or part_bytes <= 0:
        raise ValueError("table must hold whole rows of row_bytes bytes")
    if idx.numel() != ctas * tiles * (32768 // part_bytes):
        raise ValueError("idx must hold ctas * tiles * (32768 // part_bytes) rows")
    _check("sa_probe_row_gather", load().sa_probe_row_gather(
        _dptr(table), table.numel() // row_bytes, row_bytes, part_bytes, _dptr(idx), ctas, tiles,
        _stream_ptr(stream)))


def workspace_for(B, S, H, D, K, num_splits=0, device=None) -> torch.Tensor | None:
    n = sa_sparse_attn_workspace_size(B, S, H, D, K, num_splits)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def sparse_attn(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor, topk_idxs: torch.Tensor,
                softmax_scale: float, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                num_splits: int = 0, stream=None, topk_length: torch.Tensor | None = None) -> torch.Tensor:
    """o = sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale) on the GPU.

    q bf16 [B,S,H,D], kv bf16 [B,T,D], attn_sink fp32 [H], topk_idxs int32
    [B,S,K] (-1 = invalid), all contiguous on one CUDA device.  topk_length:
    optional int32 [B,S]; slot j counts only below clamp(topk_length, 0, K)."""
    for name, t, dt in (("q", q, torch.bfloat16), ("kv", kv, torch.bfloat16),
                        ("attn_sink", attn_sink, torch.float32), ("topk_idxs", topk_idxs, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    B, S, H, D = q.shape
    T = kv.shape[1]
    K = topk_idxs.shape[-1]
    if kv.shape != (B, T, D) or topk_idxs.shape != (B, S, K) or attn_sink.shape != (H,):
        raise ValueError("shape mismatch among q, kv, attn_sink, topk_idxs")
    if out is None:
        out = torch.empty_like(q)
    need = sa_sparse_attn_workspace_size(B, S, H, D, K, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if topk_length is not None:
        if topk_length.dtype != torch.int32 or not topk_length.is_cuda or not topk_length.is_contiguous() \
                or topk_length.numel() != B * S:
            raise ValueError("topk_length must be a contiguous CUDA int32 tensor with B*S elements")
        rc = sa_sparse_attn_fwd_topk_length(_dptr(q), _dptr(kv), _dptr(attn_sink), _dptr(topk_idxs),
                                            _dptr(topk_length), float(softmax_scale), _dptr(out), B, S, H, D, T, K,
                                            int(num_splits), _dptr(workspace), ws_bytes, _stream_ptr(stream))
        _check("sa_sparse_attn_fwd_topk_length", rc)
        return out
    rc = sa_sparse_attn_fwd_splits(_dptr(q), _dptr(kv), _dptr(attn_sink), _dptr(topk_idxs), float(softmax_scale),
                                   _dptr(out), B, S, H, D, T, K, int(num_splits), _dptr(workspace), ws_bytes,
                                   _stream_ptr(stream))
    _check("sa_sparse_attn_fwd_splits", rc)
    return out


def sa_sparse_attn_fwd_extra(q, kv, attn_sink, topk_idxs, topk_length, extra_kv, extra_topk_idxs,
                             extra_topk_length, softmax_scale, o, B, S, H, D, T, K, T2, K2, num_splits, workspace,
                             workspace_bytes, stream):
    return int(load().sa_sparse_attn_fwd_extra(q, kv, attn_sink, topk_idxs, topk_length, extra_kv, extra_topk_idxs,
                                               extra_topk_length, softmax_scale, o, B, S, H, D, T, K, T2, K2,
                                               num_splits, workspace, workspace_bytes, stream))


def sa_sparse_attn_fwd_fp8_extra(q, kv_fp8, attn_sink, topk_idxs, topk_length, extra_kv_fp8, extra_topk_idxs,
                                 extra_topk_length, softmax_scale, o, B, S, H, T, K, T2, K2, num_splits, workspace,
                                 workspace_bytes, stream):
    return int(load().sa_sparse_attn_fwd_fp8_extra(q, kv_fp8, attn_sink, topk_idxs, topk_length, extra_kv_fp8,
                                                   extra_topk_idxs, extra_topk_length, softmax_scale, o, B, S, H, T,
                                                   K, T2, K2, num_splits, workspace, workspace_bytes, stream))


def sparse_attn_extra(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor, topk_idxs: torch.Tensor,
                      extra_kv: torch.Tensor, extra_topk_idxs: torch.Tensor, softmax_scale: float,
                      topk_length: torch.Tensor | None = None, extra_topk_length: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, num_splits: int = 0,
                      stream=None) -> torch.Tensor:
    """sparse_attn over two kv sources: each token's K main slots (kv,
    topk_idxs) and its K2 extra slots (extra_kv [B,T2,D] or, for FP8 caches,
    uint8 [B,T2,584] like kv; extra_topk_idxs [B,S,K2]) in one softmax."""
    fp8 = kv.dtype == torch.uint8
    B, S, H, D = q.shape
    T, T2 = kv.shape[1], extra_kv.shape[1]
    K, K2 = topk_idxs.shape[-1], extra_topk_idxs.shape[-1]
    for name, t in (("q", q), ("kv", kv), ("attn_sink", attn_sink), ("topk_idxs", topk_idxs),
                    ("extra_kv", extra_kv), ("extra_topk_idxs", extra_topk_idxs), ("topk_length", topk_length),
                    ("extra_topk_length", extra_topk_length)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if extra_kv.dtype != kv.dtype or topk_idxs.dtype != torch.int32 or extra_topk_idxs.dtype != torch.int32:
        raise ValueError("kv and extra_kv share a dtype; the index lists are int32")
    if out is None:
        out = torch.empty_like(q)
    need = sa_sparse_attn_workspace_size(B, S, H, D, K + K2, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if fp8:
        rc = sa_sparse_attn_fwd_fp8_extra(_dptr(q), _dptr(kv), _dptr(attn_sink), _dptr(topk_idxs), _dptr(topk_length),
                                          _dptr(extra_kv), _dptr(extra_topk_idxs), _dptr(extra_topk_length),
                                          float(softmax_scale), _dptr(out), B, S, H, T, K, T2, K2, int(num_splits),
                                          _dptr(workspace), ws_bytes, _stream_ptr(stream))
        _check("sa_sparse_attn_fwd_fp8_extra", rc)
    else:
        rc = sa_sparse_attn_fwd_extra(_dptr(q), _dptr(kv), _dptr(attn_sink), _dptr(topk_idxs), _dptr(topk_length),
                                      _dptr(extra_kv), _dptr(extra_topk_idxs), _dptr(extra_topk_length),
                                      float(softmax_scale), _dptr(out), B, S, H, D, T, K, T2, K2, int(num_splits),
                                      _dptr(workspace), ws_bytes, _stream_ptr(stream))
        _check("sa_sparse_attn_fwd_extra", rc)
    return out


def topk_mask_shape(batch: int, max_query_len: int, max_key_len: int,
                    reserve_key_starts_word: bool = False) -> tuple[int, int, int]:
    return sa_topk_mask_shape(batch, max_query_len, max_key_len, reserve_key_starts_word)


def build_topk_mask(topk: torch.Tensor, cu_q_lens: torch.Tensor, max_q_len: int, max_key_len: int,
                    key_starts: torch.Tensor | None = None, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """uint32 mask [B, rows, words] (stored as int32 storage when ``out`` is
    int32, as the pages' test allocates it).  Words the build does not write
    keep the contents of ``out``."""
    B = cu_q_lens.numel() - 1
    shape = topk_mask_shape(B, max_q_len, max_key_len, key_starts is not None)
    if out is None:
        out = torch.zeros(shape, dtype=torch.int32, device=topk.device)
    if tuple(out.shape) != shape or out.element_size() != 4 or not out.is_contiguous():
        raise ValueError(f"mask buffer must be a contiguous 32-bit tensor of shape {shape}")
    if topk.dtype != torch.int32 or cu_q_lens.dtype != torch.int32:
        raise ValueError("topk and cu_q_lens must be int32")
    tk = topk if topk.dim() == 2 else topk.reshape(-1, topk.shape[-1] if topk.dim() else 1)
    rc = sa_build_topk_mask(_dptr(tk), tk.shape[0], _dptr(cu_q_lens), B, max_q_len, max_key_len, tk.shape[1],
                            _dptr(key_starts), _dptr(out), shape, _stream_ptr(stream))
    _check("sa_build_topk_mask", rc)
    return out


def masked_dense_attn(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor, mask: torch.Tensor,
                      softmax_scale: float, key_start_word: bool = False, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, num_splits: int = 0, stream=None) -> torch.Tensor:
    """Attention of q bf16 [B,S,H,D] over the keys of kv bf16 [B,T,D] that the
    bit-packed mask (32-bit words [B, rows >= S, words], as build_topk_mask
    returns it) admits, with the per-head sink.  key_start_word: test bit
    t + mask[b, 0, words-1] for key t (a context chunk at that offset)."""
    for name, t, dt in (("q", q, torch.bfloat16), ("kv", kv, torch.bfloat16), ("attn_sink", attn_sink, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if mask.element_size() != 4 or mask.dim() != 3 or not mask.is_cuda or not mask.is_contiguous():
        raise ValueError("mask must be a contiguous CUDA 32-bit tensor [B, rows, words]")
    B, S, H, D = q.shape
    T = kv.shape[1]
    if kv.shape != (B, T, D) or attn_sink.shape != (H,) or mask.shape[0] != B:
        raise ValueError("shape mismatch among q, kv, attn_sink, mask")
    if out is None:
        out = torch.empty_like(q)
    need = sa_masked_dense_attn_workspace_size(B, S, H, D, T, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = sa_masked_dense_attn_fwd(_dptr(q), _dptr(kv), _dptr(attn_sink), _dptr(mask), mask.shape[1], mask.shape[2],
                                  int(bool(key_start_word)), float(softmax_scale), _dptr(out), B, S, H, D, T,
                                  int(num_splits), _dptr(workspace), ws_bytes, _stream_ptr(stream))
    _check("sa_masked_dense_attn_fwd", rc)
    return out


FP8_ROW_BYTES = 584


def sparse_attn_fp8(q: torch.Tensor, kv_fp8: torch.Tensor, attn_sink: torch.Tensor, topk_idxs: torch.Tensor,
                    softmax_scale: float, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    num_splits: int = 0, stream=None, topk_length: torch.Tensor | None = None) -> torch.Tensor:
    """sparse_attn over an FP8 kv cache: q bf16 [B,S,H,512], kv_fp8 uint8
    [B,T,584] (448 E4M3 codes, 64 bf16 RoPE dims, 8 E8M0 tile-scale bytes per
    row), attn_sink fp32 [H], topk_idxs int32 [B,S,K]; o bf16 [B,S,H,512]."""
    for name, t, dt in (("q", q, torch.bfloat16), ("kv_fp8", kv_fp8, torch.uint8),
                        ("attn_sink", attn_sink, torch.float32), ("topk_idxs", topk_idxs, torch.int32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    B, S, H, D = q.shape
    T = kv_fp8.shape[1]
    K = topk_idxs.shape[-1]
    if D != 512 or kv_fp8.shape != (B, T, FP8_ROW_BYTES) or topk_idxs.shape != (B, S, K) or attn_sink.shape != (H,):
        raise ValueError("shape mismatch among q, kv_fp8, attn_sink, topk_idxs")
    if topk_length is not None and (topk_length.dtype != torch.int32 or not topk_length.is_cuda
                                    or not topk_length.is_contiguous() or topk_length.numel() != B * S):
        raise ValueError("topk_length must be a contiguous CUDA int32 tensor with B*S elements")
    if out is None:
        out = torch.empty_like(q)
    need = sa_sparse_attn_workspace_size(B, S, H, 512, K, num_splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = sa_sparse_attn_fwd_fp8(_dptr(q), _dptr(kv_fp8), _dptr(attn_sink), _dptr(topk_idxs), _dptr(topk_length),
                                float(softmax_scale), _dptr(out), B, S, H, T, K, int(num_splits), _dptr(workspace),
                                ws_bytes, _stream_ptr(stream))
    _check("sa_sparse_attn_fwd_fp8", rc)
    return out


def build_topk_mask_window(topk: torch.Tensor, cu_q_lens: torch.Tensor, q0: int, q_rows: int, max_key_len: int,
                           key_starts: torch.Tensor | None = None, key_ends: torch.Tensor | None = None,
                           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Mask window [B, rows, words]: row i is query q0 + i of each request;
    only the words below each request's live key end are written."""
    B = cu_q_lens.numel() - 1
    shape = topk_mask_shape(B, q_rows, max_key_len, key_starts is not None)
    if out is None:
        out = torch.zeros(shape, dtype=torch.int32, device=topk.device)
    if tuple(out.shape) != shape or out.element_size() != 4 or not out.is_contiguous():
        raise ValueError(f"mask buffer must be a contiguous 32-bit tensor of shape {shape}")
    tk = topk if topk.dim() == 2 else topk.reshape(-1, topk.shape[-1] if topk.dim() else 1)
    rc = sa_build_topk_mask_window(_dptr(tk), tk.shape[0], _dptr(cu_q_lens), B, q0, q_rows, max_key_len, tk.shape[1],
                                   _dptr(key_starts), _dptr(key_ends), _dptr(out), shape, _stream_ptr(stream))
    _check("sa_build_topk_mask_window", rc)
    return out


def topk_masked_attn(q: torch.Tensor, kv: torch.Tensor, attn_sink: torch.Tensor, topk: torch.Tensor,
                     cu_q_lens: torch.Tensor, softmax_scale: float, max_key_len: int,
                     key_starts: torch.Tensor | None = None, key_ends: torch.Tensor | None = None,
                     cap_bytes: int = 0, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Attention of q bf16 [B, max_q_len, H, D] over the keys its top-k rows
    select, through the bit-packed mask built and consumed in windows of
    query rows that fit cap_bytes (0: 64 MiB).  Rows past a request's query
    count are left unspecified."""
    B, Q, H, D = q.shape
    T = kv.shape[1]
    tk = topk if topk.dim() == 2 else topk.reshape(-1, topk.shape[-1])
    reserve = key_starts is not None
    qc = sa_topk_mask_chunk_rows(B, Q, max_key_len, reserve, cap_bytes)
    if qc < 1:
        raise ValueError("no window of query rows fits the mask cap")
    shape = topk_mask_shape(B, qc, max_key_len, reserve)
    mbuf = torch.empty(shape, dtype=torch.int32, device=q.device)
    nws = sa_topk_masked_attn_workspace_size(B, Q, H, D, T, max_key_len, reserve, cap_bytes)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    rc = sa_topk_masked_attn_fwd(_dptr(q), _dptr(kv), _dptr(attn_sink), _dptr(tk), tk.shape[0], _dptr(cu_q_lens),
                                 _dptr(key_starts), _dptr(key_ends), float(softmax_scale), _dptr(out), B, Q, H, D, T,
                                 max_key_len, tk.shape[1], int(cap_bytes), _dptr(mbuf), mbuf.numel() * 4, _dptr(ws),
                                 nws, _stream_ptr(stream))
    _check("sa_topk_masked_attn_fwd", rc)
    return out
