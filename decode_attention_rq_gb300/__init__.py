"""Python binding of librq (ResidualQuant KV cache + decode attention on GB300).

Argument marshalling only: every function calls the C entry point of the same
name in librq.so (declared in include/rq.h).  Tensors are passed by device
pointer; streams by handle.  There is no fallback: if the library is missing
this module raises on import.  Build it with
`python decode_attention_rq_gb300/build.py` (nvcc, sm_103a).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "RQ_OK", "RQ_MODE_SHARED", "RQ_MODE_CHAINED", "RQ_MODE_NORM_RATIO", "RQ_MODE_HADAMARD", "RqError", "rq_config",
    "lib", "LIB_PATH",
    "rq_cache_bytes", "rq_cache_create", "rq_cache_destroy", "rq_append",
    "rq_decode_workspace_bytes", "rq_decode_attention", "rq_bf16_workspace_bytes",
    "rq_decode_attention_bf16", "rq_status_string", "EXPORTED_SYMBOLS",
    "rq_decode_attention_noalloc", "RQ_NOALLOC_WORKSPACE_BYTES", "rq_decode_attention_append",
    "rq_cache_paged_bytes", "rq_cache_create_paged",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librq.so")

RQ_OK = 0
RQ_MODE_SHARED = 0
RQ_MODE_CHAINED = 1
RQ_MODE_NORM_RATIO = 2   # flag: norm-ratio coefficient instead of least squares
RQ_MODE_HADAMARD = 4     # flag: R = H_d / sqrt(d) as a fast Walsh-Hadamard transform (d = 128); R_dev may be None
_STATUS_NAMES = {0: "RQ_OK", 1: "RQ_ERR_INVALID_ARG", 2: "RQ_ERR_ALIGNMENT", 3: "RQ_ERR_CAPACITY",
                 4: "RQ_ERR_WORKSPACE", 5: "RQ_ERR_CUDA", 6: "RQ_ERR_UNSUPPORTED", 7: "RQ_ERR_TIMEOUT"}

EXPORTED_SYMBOLS = (
    "rq_cache_bytes", "rq_cache_create", "rq_cache_destroy", "rq_append",
    "rq_decode_workspace_bytes", "rq_decode_attention", "rq_bf16_workspace_bytes",
    "rq_decode_attention_bf16", "rq_status_string", "rq_decode_attention_noalloc",
    "rq_decode_attention_append", "rq_cache_paged_bytes", "rq_cache_create_paged",
)

# size of the workspace built into the library for rq_decode_attention_noalloc (rq.h)
RQ_NOALLOC_WORKSPACE_BYTES = 2 * 1024 * 1024


class RqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_STATUS_NAMES.get(status, status)} ({rq_status_string(status)})")


class rq_config(ctypes.Structure):
    """rq.h's rq_config; num_query_heads (last, default 0) > num_heads selects grouped-query attention."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "loops_per_group", "num_groups", "num_heads", "head_dim", "group_size",
        "max_batch", "max_seq_len", "mode", "num_query_heads")]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python decode_attention_rq_gb300/build.py`")
lib = ctypes.CDLL(LIB_PATH)

_p, _i32, _sz, _f = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
_cfgp = ctypes.POINTER(rq_config)
lib.rq_cache_bytes.argtypes = [_cfgp]
lib.rq_cache_bytes.restype = _sz
lib.rq_cache_create.argtypes = [_cfgp, _p, _sz, _p, ctypes.POINTER(_p)]
lib.rq_cache_create.restype = ctypes.c_int
lib.rq_cache_paged_bytes.argtypes = [_cfgp, _i32]
lib.rq_cache_paged_bytes.restype = _sz
lib.rq_cache_create_paged.argtypes = [_cfgp, _i32, _p, _sz, _p, _i32, _p, ctypes.POINTER(_p)]
lib.rq_cache_create_paged.restype = ctypes.c_int
lib.rq_cache_destroy.argtypes = [_p]
lib.rq_cache_destroy.restype = ctypes.c_int
lib.rq_append.argtypes = [_p, _i32, _i32, _i32, _p, _p, _i32, _p, _p]
lib.rq_append.restype = ctypes.c_int
lib.rq_decode_workspace_bytes.argtypes = [_cfgp, _i32]
lib.rq_decode_workspace_bytes.restype = _sz
lib.rq_decode_attention.argtypes = [_p, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f, _p, _p, _sz, _p]
lib.rq_decode_attention.restype = ctypes.c_int
lib.rq_decode_attention_noalloc.argtypes = [_p, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _f, _p, _p, _p]
lib.rq_decode_attention_noalloc.restype = ctypes.c_int
lib.rq_decode_attention_append.argtypes = [_p, _i32, _i32, _i32, _p, _p, _p, _f, _p, _p, _sz, _p]
lib.rq_decode_attention_append.restype = ctypes.c_int
lib.rq_bf16_workspace_bytes.argtypes = [_i32, _i32, _i32]
lib.rq_bf16_workspace_bytes.restype = _sz
lib.rq_decode_attention_bf16.argtypes = [_p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _f, _p, _p, _sz, _p]
lib.rq_decode_attention_bf16.restype = ctypes.c_int
lib.rq_status_string.argtypes = [ctypes.c_int]
lib.rq_status_string.restype = ctypes.c_char_p


def _ptr(x):
    """Device/host address of a tensor (data_ptr) or an int; None -> NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, st):
    if st != RQ_OK:
        raise RqError(fn, st)


def rq_status_string(status: int) -> str:
    return lib.rq_status_string(status).decode()


def rq_cache_bytes(cfg: rq_config) -> int:
    return lib.rq_cache_bytes(ctypes.byref(cfg))


def rq_cache_create(cfg: rq_config, dev_buf, nbytes: int, R_dev) -> int:
    """Returns the opaque handle (int)."""
    h = _p()
    _check("rq_cache_create", lib.rq_cache_create(ctypes.byref(cfg), _ptr(dev_buf), nbytes, _ptr(R_dev),
                                                  ctypes.byref(h)))
    return h.value


def rq_cache_paged_bytes(cfg: rq_config, num_pages: int) -> int:
    return lib.rq_cache_paged_bytes(ctypes.byref(cfg), num_pages)


def rq_cache_create_paged(cfg: rq_config, num_pages: int, pool, nbytes: int, block_table, max_tiles_per_row: int,
                          R_dev) -> int:
    """Paged layout: tile t of row b lives in page block_table[b, t] of each
    (layer, group)'s pool.  Returns the opaque handle (int)."""
    h = _p()
    _check("rq_cache_create_paged", lib.rq_cache_create_paged(
        ctypes.byref(cfg), num_pages, _ptr(pool), nbytes, _ptr(block_table), max_tiles_per_row, _ptr(R_dev),
        ctypes.byref(h)))
    return h.value


def rq_cache_destroy(handle: int) -> None:
    _check("rq_cache_destroy", lib.rq_cache_destroy(handle))


def rq_append(handle, layer, group, batch, kv, seq_lens, n_tokens, status=None, stream=None):
    _check("rq_append", lib.rq_append(handle, layer, group, batch, _ptr(kv), _ptr(seq_lens), n_tokens,
                                      _ptr(status), _stream(stream)))


def rq_decode_workspace_bytes(cfg: rq_config, batch: int) -> int:
    return lib.rq_decode_workspace_bytes(ctypes.byref(cfg), batch)


def rq_decode_attention(handle, layer, group, loop, batch, q, k_cur, v_cur, seq_lens, softmax_scale,
                        out, workspace, workspace_bytes, stream=None):
    _check("rq_decode_attention", lib.rq_decode_attention(
        handle, layer, group, loop, batch, _ptr(q), _ptr(k_cur), _ptr(v_cur), _ptr(seq_lens),
        softmax_scale, _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def rq_decode_attention_append(handle, layer, group, batch, q, kv_cur, seq_lens, softmax_scale, out, workspace,
                               workspace_bytes, stream=None):
    """Anchor-loop attention call that also appends the current token of every
    loop (kv_cur: [P, 2, batch, H, d] bf16) at position seq_lens[b]."""
    _check("rq_decode_attention_append", lib.rq_decode_attention_append(
        handle, layer, group, batch, _ptr(q), _ptr(kv_cur), _ptr(seq_lens), softmax_scale, _ptr(out),
        _ptr(workspace), workspace_bytes, _stream(stream)))


def rq_decode_attention_noalloc(handle, layer, group, loop, batch, q, k_cur, v_cur, seq_lens, softmax_scale,
                                out, status=None, stream=None):
    """rq_decode_attention without a caller workspace, for callers that cannot
    allocate device memory: the scratch lives in a fixed array inside the library
    (RQ_NOALLOC_WORKSPACE_BYTES).  Calls that overlap on the GPU race on it."""
    _check("rq_decode_attention_noalloc", lib.rq_decode_attention_noalloc(
        handle, layer, group, loop, batch, _ptr(q), _ptr(k_cur), _ptr(v_cur), _ptr(seq_lens),
        softmax_scale, _ptr(out), _ptr(status), _stream(stream)))


def rq_bf16_workspace_bytes(batch: int, num_heads: int, head_dim: int) -> int:
    return lib.rq_bf16_workspace_bytes(batch, num_heads, head_dim)


def rq_decode_attention_bf16(k_cache, v_cache, k_cur, v_cur, q, seq_lens, batch, num_heads, head_dim,
                             max_seq, softmax_scale, out, workspace, workspace_bytes, stream=None):
    _check("rq_decode_attention_bf16", lib.rq_decode_attention_bf16(
        _ptr(k_cache), _ptr(v_cache), _ptr(k_cur), _ptr(v_cur), _ptr(q), _ptr(seq_lens), batch,
        num_heads, head_dim, max_seq, softmax_scale, _ptr(out), _ptr(workspace), workspace_bytes,
        _stream(stream)))
