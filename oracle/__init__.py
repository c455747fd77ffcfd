"""CPU oracle for top-k sparse attention and the bit-packed top-k mask.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``deepseek_top_sparse_gb300``) never imports it, and the two
share no code: the arithmetic lives in ``oracle.c`` (plain C, float64), this
module only compiles it with gcc and marshals numpy arrays through ctypes.

What each routine follows (page title and section):

* ``sparse_attn`` -- "DeepSeek V4 源码剖析, 第5章", §5.2 pseudocode (per query
  token and head: gather the indexed kv rows, logits = scale * q.k, -inf on
  invalid slots, append the per-head sink logit, softmax, weighted sum of the
  gathered rows without the sink) and §5.5 (the sink only enters the
  denominator; sink = +inf zeroes all real weights, -inf means no sink).
* ``masked_dense_attn`` -- the consumer semantics of the bit mask from the
  vLLM PR 48770 page (``dense_mask_mod`` / ``offset_dense_mask_mod``): key k
  is admitted iff bit k&31 of word k>>5 of its query row is set.
* ``sparse_attn_fp8`` / ``decode_kv_fp8`` -- the same attention over an FP8
  kv cache in the V4 (FlashMLA "MODEL1") row format of "DeepSeek V4 源码剖析,
  第5章" §5.3 and §5.6: 448 nope dims as E4M3 codes with one E8M0 scale per
  64-dim tile, 64 RoPE dims in bf16, 584 bytes a row (byte order: reading R22
  in oracle.c).  Each gathered row is decoded to exact values first.
* ``topk_mask_shape`` / ``build_topk_mask`` -- vLLM PR 52217 page
  (``_topk_mask_shape``, ``_build_topk_mask`` and the two alignment tests) and
  the PR 48770 page (bit order, reserved key_start word).

Pins against the pages and closed forms live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_sparse_attn.argtypes = [p, p, p, p, ctypes.c_double] + [i64] * 6 + [p, ctypes.c_int]
            lib.oracle_sparse_attn_tokens.argtypes = (
                [p, p, p, p, ctypes.c_double] + [i64] * 6 + [p, i64, p, ctypes.c_int])
            lib.oracle_sparse_attn_tokens_len.argtypes = (
                [p, p, p, p, p, ctypes.c_double] + [i64] * 6 + [p, i64, p, ctypes.c_int])
            lib.oracle_sparse_attn_fp8_tokens.argtypes = (
                [p, p, p, p, p, ctypes.c_double] + [i64] * 5 + [p, i64, p, ctypes.c_int])
            lib.oracle_sparse_attn_extra_tokens.argtypes = (
                [p, p, p, p, p, p, p, p, ctypes.c_double] + [i64] * 8 + [p, i64, p, ctypes.c_int])
            lib.oracle_sparse_attn_extra_tokens.restype = ctypes.c_int
            lib.oracle_sparse_attn_fp8_extra_tokens.argtypes = (
                [p, p, p, p, p, p, p, p, ctypes.c_double] + [i64] * 7 + [p, i64, p, ctypes.c_int])
            lib.oracle_sparse_attn_fp8_extra_tokens.restype = ctypes.c_int
            lib.oracle_decode_kv_fp8.argtypes = [p, i64, p]
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_to_double.restype = ctypes.c_double
            lib.oracle_masked_dense_attn.argtypes = [p, p, p, p, i64, i64, p, p, ctypes.c_double] + [i64] * 5 + [p]
            lib.oracle_build_topk_mask_window.argtypes = [p, i64, p, i64, i64, i64, i64, i64, p, p, p, p]
            lib.oracle_build_topk_mask_window.restype = ctypes.c_int
            lib.oracle_topk_mask_shape.argtypes = [i64, i64, i64, ctypes.c_int, p]
            lib.oracle_build_topk_mask.argtypes = [p, i64, p, i64, i64, i64, i64, p, p, p]
            for f in (lib.oracle_sparse_attn, lib.oracle_sparse_attn_tokens, lib.oracle_sparse_attn_tokens_len,
                      lib.oracle_masked_dense_attn, lib.oracle_sparse_attn_fp8_tokens, lib.oracle_decode_kv_fp8,
                      lib.oracle_topk_mask_shape, lib.oracle_build_topk_mask):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bit patterns."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # local: numpy-only callers need no torch

    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _np(x, dtype):
    if not hasattr(x, "detach"):          # numpy arrays, lists, tuples
        return np.ascontiguousarray(np.asarray(x), dtype=dtype)
    return np.ascontiguousarray(x.detach().cpu().numpy(), dtype=dtype)


def sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale: float, tokens=None, nthreads: int = 0,
                topk_length=None, extra_kv=None, extra_idxs=None, extra_length=None):
    """float64 o[B,S,H,D] (or o[len(tokens),H,D] for flat token ids b*S+s).
    topk_length: optional int32 [B,S]; slot j of token (b,s) counts only if
    j < clamp(topk_length[b,s], 0, K).  extra_kv [B,T2,D] bf16 with
    extra_idxs int32 [B,S,K2] (and optional extra_length [B,S]): a second kv
    source whose slots join each token's softmax after its K main slots."""
    qb, kvb = _bf16_bits(q), _bf16_bits(kv)
    sink = _np(attn_sink, np.float32)
    idx = _np(topk_idxs, np.int32)
    B, S, H, D = qb.shape
    T = kvb.shape[1]
    K = idx.shape[-1]
    assert kvb.shape == (B, T, D) and idx.shape == (B, S, K) and sink.shape == (H,)
    lens = None
    if topk_length is not None:
        lens = _np(topk_length, np.int32).reshape(B, S)
    tok = np.arange(B * S, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    o = np.zeros((tok.shape[0], H, D), dtype=np.float64)
    if extra_kv is None:
        rc = _load().oracle_sparse_attn_tokens_len(_ptr(qb), _ptr(kvb), _ptr(sink), _ptr(idx), _ptr(lens),
                                                  float(softmax_scale), B, S, H, D, T, K, _ptr(tok), tok.shape[0],
                                                  _ptr(o), int(nthreads))
    else:
        kv2 = _bf16_bits(extra_kv)
        idx2 = _np(extra_idxs, np.int32)
        T2, K2 = kv2.shape[1], idx2.shape[-1]
        assert kv2.shape == (B, T2, D) and idx2.shape == (B, S, K2)
        lens2 = None if extra_length is None else _np(extra_length, np.int32).reshape(B, S)
        rc = _load().oracle_sparse_attn_extra_tokens(_ptr(qb), _ptr(kvb), _ptr(sink), _ptr(idx), _ptr(lens),
                                                    _ptr(kv2), _ptr(idx2), _ptr(lens2), float(softmax_scale), B, S,
                                                    H, D, T, K, T2, K2, _ptr(tok), tok.shape[0], _ptr(o),
                                                    int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_sparse_attn rejected its arguments (rc={rc})")
    return o.reshape(B, S, H, D) if tokens is None else o


FP8_ROW_BYTES = 584   # one kv row of the FP8 cache (R22)


def _u8(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint8
        return np.ascontiguousarray(x)
    import torch

    assert x.dtype == torch.uint8
    return np.ascontiguousarray(x.detach().cpu().contiguous().numpy())


def e4m3_to_float(code: int) -> float:
    return float(_load().oracle_e4m3_to_double(int(code)))


def e8m0_to_float(byte: int) -> float:
    return float(_load().oracle_e8m0_to_double(int(byte)))


def decode_kv_fp8(kv8) -> np.ndarray:
    """float64 [..., 512] exact values of FP8 kv rows uint8 [..., 584]."""
    a = _u8(kv8)
    assert a.shape[-1] == FP8_ROW_BYTES
    rows = int(np.prod(a.shape[:-1]))
    out = np.zeros((rows, 512), dtype=np.float64)
    rc = _load().oracle_decode_kv_fp8(_ptr(a), rows, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_decode_kv_fp8 rejected its arguments")
    return out.reshape(*a.shape[:-1], 512)


def sparse_attn_fp8(q, kv8, attn_sink, topk_idxs, softmax_scale: float, tokens=None, nthreads: int = 0,
                    topk_length=None, extra_kv8=None, extra_idxs=None, extra_length=None):
    """sparse_attn over an FP8 kv cache uint8 [B,T,584]; q bf16 [B,S,H,512];
    optionally an extra FP8 source extra_kv8 [B,T2,584] with extra_idxs
    [B,S,K2] (and extra_length [B,S])."""
    qb, kb = _bf16_bits(q), _u8(kv8)
    sink = _np(attn_sink, np.float32)
    idx = _np(topk_idxs, np.int32)
    B, S, H, D = qb.shape
    T = kb.shape[1]
    K = idx.shape[-1]
    assert D == 512 and kb.shape == (B, T, FP8_ROW_BYTES) and idx.shape == (B, S, K) and sink.shape == (H,)
    lens = None if topk_length is None else _np(topk_length, np.int32).reshape(B, S)
    tok = np.arange(B * S, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    o = np.zeros((tok.shape[0], H, D), dtype=np.float64)
    if extra_kv8 is None:
        rc = _load().oracle_sparse_attn_fp8_tokens(_ptr(qb), _ptr(kb), _ptr(sink), _ptr(idx), _ptr(lens),
                                                   float(softmax_scale), B, S, H, T, K, _ptr(tok), tok.shape[0],
                                                   _ptr(o), int(nthreads))
    else:
        kb2 = _u8(extra_kv8)
        idx2 = _np(extra_idxs, np.int32)
        T2, K2 = kb2.shape[1], idx2.shape[-1]
        assert kb2.shape == (B, T2, FP8_ROW_BYTES) and idx2.shape == (B, S, K2)
        lens2 = None if extra_length is None else _np(extra_length, np.int32).reshape(B, S)
        rc = _load().oracle_sparse_attn_fp8_extra_tokens(_ptr(qb), _ptr(kb), _ptr(sink), _ptr(idx), _ptr(lens),
                                                        _ptr(kb2), _ptr(idx2), _ptr(lens2), float(softmax_scale), B,
                                                        S, H, T, K, T2, K2, _ptr(tok), tok.shape[0], _ptr(o),
                                                        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_sparse_attn_fp8 rejected its arguments (rc={rc})")
    return o.reshape(B, S, H, D) if tokens is None else o


def masked_dense_attn(q, kv, attn_sink, mask, softmax_scale: float, key_offset=None, key_ends=None):
    """float64 o[B,S,H,D]: dense attention over the keys the bit mask admits
    (key_ends: per-request live end in mask positions, or None)."""
    qb, kvb = _bf16_bits(q), _bf16_bits(kv)
    sink = _np(attn_sink, np.float32)
    m = _np(mask, np.int64).astype(np.uint32) if not isinstance(mask, np.ndarray) or mask.dtype != np.uint32 \
        else np.ascontiguousarray(mask)
    B, S, H, D = qb.shape
    T = kvb.shape[1]
    assert m.shape[0] == B and m.shape[1] >= S
    off = None if key_offset is None else np.ascontiguousarray(key_offset, dtype=np.int64)
    ends = None if key_ends is None else np.ascontiguousarray(_np(key_ends, np.int64))
    o = np.zeros((B, S, H, D), dtype=np.float64)
    rc = _load().oracle_masked_dense_attn(_ptr(qb), _ptr(kvb), _ptr(sink), _ptr(m), m.shape[1], m.shape[2],
                                          _ptr(off), _ptr(ends), float(softmax_scale), B, S, H, D, T, _ptr(o))
    if rc != 0:
        raise ValueError(f"oracle_masked_dense_attn rejected its arguments (rc={rc})")
    return o


def topk_mask_shape(batch: int, max_query_len: int, max_key_len: int,
                    reserve_key_starts_word: bool = False) -> tuple[int, int, int]:
    out = np.zeros(3, dtype=np.int64)
    rc = _load().oracle_topk_mask_shape(batch, max_query_len, max_key_len, int(bool(reserve_key_starts_word)),
                                        _ptr(out))
    if rc != 0:
        raise ValueError("oracle_topk_mask_shape: negative size")
    return int(out[0]), int(out[1]), int(out[2])


def build_topk_mask(topk, cu_q_lens, batch: int, max_q_len: int, max_key_len: int,
                    key_starts=None, out: np.ndarray | None = None) -> np.ndarray:
    """uint32 mask [B, padded_Q, W].  ``out`` (uint32, the right shape) keeps
    whatever it holds outside the words the build writes."""
    tk = _np(topk, np.int32)
    if tk.ndim == 1:
        tk = tk.reshape(-1, 1)
    cu = _np(cu_q_lens, np.int32)
    assert cu.shape == (batch + 1,)
    ks = None if key_starts is None else _np(key_starts, np.int32)
    shape = topk_mask_shape(batch, max_q_len, max_key_len, ks is not None)
    if out is None:
        out = np.zeros(shape, dtype=np.uint32)
    assert out.dtype == np.uint32 and out.ndim == 3 and out.flags.c_contiguous
    shp = np.asarray(out.shape, dtype=np.int64)  # the C routine rejects a wrong shape
    rc = _load().oracle_build_topk_mask(_ptr(tk), tk.shape[0], _ptr(cu), batch, max_q_len, max_key_len,
                                        tk.shape[1], _ptr(ks), _ptr(out), _ptr(shp))
    if rc != 0:
        raise ValueError(f"oracle_build_topk_mask rejected its arguments (rc={rc})")
    return out


def build_topk_mask_window(topk, cu_q_lens, batch: int, q0: int, q_rows: int, max_key_len: int, key_starts=None,
                           key_ends=None, out: np.ndarray | None = None) -> np.ndarray:
    """uint32 mask [B, padded(q_rows), W] whose row i is query q0 + i of each
    request; only words below each request's live end (key_ends, or
    max_key_len) are written."""
    tk = _np(topk, np.int32)
    if tk.ndim == 1:
        tk = tk.reshape(-1, 1)
    cu = _np(cu_q_lens, np.int32)
    assert cu.shape == (batch + 1,)
    ks = None if key_starts is None else _np(key_starts, np.int32)
    ke = None if key_ends is None else _np(key_ends, np.int32)
    shape = topk_mask_shape(batch, q_rows, max_key_len, ks is not None)
    if out is None:
        out = np.zeros(shape, dtype=np.uint32)
    assert out.dtype == np.uint32 and out.ndim == 3 and out.flags.c_contiguous
    shp = np.asarray(out.shape, dtype=np.int64)
    rc = _load().oracle_build_topk_mask_window(_ptr(tk), tk.shape[0], _ptr(cu), batch, q0, q_rows, max_key_len,
                                               tk.shape[1], _ptr(ks), _ptr(ke), _ptr(out), _ptr(shp))
    if rc != 0:
        raise ValueError(f"oracle_build_topk_mask_window rejected its arguments (rc={rc})")
    return out
