"""Paged-KV attention for GB300 (sm_103a): thin Python binding of the C ABI.

The compute is entirely in ``_build/libpaged_attn.so`` (hand-written CUDA,
see ``include/paged_attn.h``).  This module only marshals torch tensors into
pointers and sizes; it never computes attention itself, and every call raises
if the library is missing or returns an error.

    out = paged_attn_mixed(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens)

Tensors: q ``[total_q, Hq, d]`` (bf16/f16/f32), caches
``[num_pages, page_size, Hkv, d]`` (same dtype, or uint8 / float8_e5m2 for
fp8 E5M2 with ``k_scale``/``v_scale``), ``block_table`` int32
``[B, max_pages]``, ``cu_seqlens_q`` int32 ``[B + 1]``, ``seq_lens`` int32
``[B]`` (each row's total KV length, its new tokens included), all on the
same CUDA device.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = ["paged_attn_prefill", "paged_attn_decode", "paged_attn_mixed",
           "paged_attn_decode_static", "STATIC_SCRATCH_BYTES", "workspace_size",
           "make_workspace", "read_errors", "load", "PagedAttnError", "library_path",
           "PA_SPLITS_BY_LENGTH", "PA_PREFILL_PARTS_AUTO", "PA_VERIFY_TOKENWISE",
           "PA_MERGE_AUTO", "PA_MERGE_SEPARATE", "PA_MERGE_SAME_LAUNCH",
           "PA_F32", "PA_F16", "PA_BF16", "PA_E5M2"]

PA_F32, PA_F16, PA_BF16, PA_E5M2 = 0, 1, 2, 3
STATIC_SCRATCH_BYTES = 16 << 20  # PA_STATIC_SCRATCH_BYTES of include/paged_attn.h
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small",
           4: "CUDA error", 5: "no sm_103 device"}
DEVERR = {1: "bad block-table entry", 4: "decode row q_len > max_decode_q"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpaged_attn.so")
_lock = threading.Lock()
_lib = None


class PagedAttnError(RuntimeError):
    pass


class Params(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("max_decode_q", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("verify_mode", ctypes.c_int32),
                ("prefill_kv_parts", ctypes.c_int32), ("merge_mode", ctypes.c_int32)]

PA_VERIFY_PACKED, PA_VERIFY_TOKENWISE = 0, 1
PA_PREFILL_PARTS_AUTO = -1
PA_SPLITS_BY_LENGTH = -1
PA_MERGE_AUTO, PA_MERGE_SEPARATE, PA_MERGE_SAME_LAUNCH = 0, 1, 2


class Batch(ctypes.Structure):
    _fields_ = [("num_rows", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_pages_per_row", ctypes.c_int32),
                ("cu_seqlens_q", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("cu_seqlens_q_host", ctypes.c_void_p),
                ("seq_lens_host", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str):
    """A copy of the C library at `path` with its function signatures
    declared (the package itself uses load(); tests also load test builds)."""
    lib = ctypes.CDLL(path)
    P, B = ctypes.POINTER(Params), ctypes.POINTER(Batch)
    for name in ("paged_attn_prefill", "paged_attn_decode", "paged_attn_mixed"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, B, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.paged_attn_decode_static.restype = ctypes.c_int
    lib.paged_attn_decode_static.argtypes = [P, B, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p]
    lib.paged_attn_workspace_size.restype = ctypes.c_size_t
    lib.paged_attn_workspace_size.argtypes = [P, ctypes.c_int32, ctypes.c_int32]
    lib.paged_attn_read_errors.restype = ctypes.c_int
    lib.paged_attn_read_errors.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.POINTER(ctypes.c_uint32)]
    lib.paged_attn_status_string.restype = ctypes.c_char_p
    lib.paged_attn_status_string.argtypes = [ctypes.c_int]
    lib.paged_attn_version.restype = ctypes.c_int32
    return lib


def load():
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise PagedAttnError(
                    f"paged attention CUDA library missing at {_LIB_PATH}; "
                    "build it with paged_kv_attention_prefill_gb300.build.build()")
            _lib = load_library(_LIB_PATH)
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype in (torch.uint8, getattr(torch, "float8_e5m2", None)):
        return PA_E5M2
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_params(q, k_cache, *, softmax_scale=0.0, k_scale=1.0, v_scale=1.0, max_decode_q=0,
                num_splits=0, verify_mode=PA_VERIFY_PACKED, prefill_kv_parts=0,
                merge_mode=PA_MERGE_AUTO) -> Params:
    return Params(int(q.shape[1]), int(k_cache.shape[2]), int(q.shape[2]),
                  int(k_cache.shape[1]), _dtype_code(q), _dtype_code(k_cache),
                  float(softmax_scale or 0.0), float(k_scale), float(v_scale),
                  int(max_decode_q), int(num_splits), int(verify_mode), int(prefill_kv_parts),
                  int(merge_mode))


def workspace_size(params: Params, num_rows: int, total_q: int) -> int:
    n = load().paged_attn_workspace_size(ctypes.byref(params), int(num_rows), int(total_q))
    if n == 0:
        raise PagedAttnError("invalid parameters for workspace_size")
    return int(n)


def make_workspace(params: Params, num_rows: int, total_q: int, device) -> torch.Tensor:
    """A zero-filled workspace (the header's error word must start at zero)."""
    return torch.zeros(workspace_size(params, num_rows, total_q), dtype=torch.uint8,
                       device=device)


def _check_status(rc: int, what: str):
    if rc != 0:
        msg = load().paged_attn_status_string(rc).decode()
        raise PagedAttnError(f"{what} failed: {msg} (status {rc})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _call(name, q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, *, out=None,
          workspace=None, softmax_scale=0.0, k_scale=1.0, v_scale=1.0, max_decode_q=0,
          num_splits=0, verify_mode=PA_VERIFY_PACKED, prefill_kv_parts=0,
          merge_mode=PA_MERGE_AUTO, cu_seqlens_q_host=None, seq_lens_host=None, stream=None):
    for t in (q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens):
        if not t.is_cuda:
            raise PagedAttnError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise PagedAttnError("all tensors must be contiguous")
    if block_table.dtype != torch.int32 or cu_seqlens_q.dtype != torch.int32 or \
            seq_lens.dtype != torch.int32:
        raise PagedAttnError("block_table, cu_seqlens_q and seq_lens must be int32")
    prm = make_params(q, k_cache, softmax_scale=softmax_scale, k_scale=k_scale,
                      v_scale=v_scale, max_decode_q=max_decode_q, num_splits=num_splits,
                      verify_mode=verify_mode, prefill_kv_parts=prefill_kv_parts,
                      merge_mode=merge_mode)
    B = int(seq_lens.shape[0])
    total_q = int(q.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = make_workspace(prm, B, total_q, q.device)
    hcu = hl = None
    if cu_seqlens_q_host is not None and seq_lens_host is not None:
        hcu = torch.as_tensor(cu_seqlens_q_host, dtype=torch.int32).contiguous()
        hl = torch.as_tensor(seq_lens_host, dtype=torch.int32).contiguous()
    bat = Batch(B, total_q, int(k_cache.shape[0]), int(block_table.shape[1]) if B else 0,
                _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(block_table), _ptr(hcu), _ptr(hl))
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        rc = getattr(load(), name)(ctypes.byref(prm), ctypes.byref(bat), _ptr(q), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), sp)
    _check_status(rc, name)
    return out


def paged_attn_prefill(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, **kw):
    """Varlen causal paged prefill of every row (see include/paged_attn.h)."""
    return _call("paged_attn_prefill", q, k_cache, v_cache, block_table, cu_seqlens_q,
                 seq_lens, **kw)


def paged_attn_decode(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, **kw):
    """Split-KV paged decode of every row (q_len <= max_decode_q)."""
    return _call("paged_attn_decode", q, k_cache, v_cache, block_table, cu_seqlens_q,
                 seq_lens, **kw)


def paged_attn_mixed(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, **kw):
    """Mixed batch: short rows to split-KV decode, the rest to prefill."""
    return _call("paged_attn_mixed", q, k_cache, v_cache, block_table, cu_seqlens_q,
                 seq_lens, **kw)


def paged_attn_decode_static(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, *,
                             out=None, softmax_scale=0.0, k_scale=1.0, v_scale=1.0,
                             max_decode_q=0, verify_mode=PA_VERIFY_PACKED,
                             merge_mode=PA_MERGE_AUTO, cu_seqlens_q_host=None,
                             seq_lens_host=None, stream=None):
    """Split-KV decode without a workspace: for callers that cannot allocate
    device memory.  The library's fixed device array (STATIC_SCRATCH_BYTES,
    shared by every call) holds the scratch; larger batches are refused.
    Calls that overlap on the GPU race -- serialize them."""
    for t in (q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens):
        if not t.is_cuda or not t.is_contiguous():
            raise PagedAttnError("all tensors must be contiguous CUDA tensors")
    prm = make_params(q, k_cache, softmax_scale=softmax_scale, k_scale=k_scale,
                      v_scale=v_scale, max_decode_q=max_decode_q, verify_mode=verify_mode,
                      merge_mode=merge_mode)
    B = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    hcu = hl = None
    if cu_seqlens_q_host is not None and seq_lens_host is not None:
        hcu = torch.as_tensor(cu_seqlens_q_host, dtype=torch.int32).contiguous()
        hl = torch.as_tensor(seq_lens_host, dtype=torch.int32).contiguous()
    bat = Batch(B, int(q.shape[0]), int(k_cache.shape[0]), int(block_table.shape[1]) if B else 0,
                _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(block_table), _ptr(hcu), _ptr(hl))
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        rc = load().paged_attn_decode_static(ctypes.byref(prm), ctypes.byref(bat), _ptr(q),
                                             _ptr(k_cache), _ptr(v_cache), _ptr(out), sp)
    _check_status(rc, "paged_attn_decode_static")
    return out


def read_errors(workspace: torch.Tensor, stream=None) -> int:
    """Sticky device-side error flags of a workspace (then cleared)."""
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    v = ctypes.c_uint32(0)
    with torch.cuda.device(workspace.device):
        rc = load().paged_attn_read_errors(_ptr(workspace), stream.cuda_stream, ctypes.byref(v))
    _check_status(rc, "paged_attn_read_errors")
    return int(v.value)
