"""Paged-KV attention oracle (fp64, CPU) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never calls it, and this package never imports the product.

The arithmetic lives in ``paged_attention_oracle.c`` (plain C, double
precision, OpenMP over (token, head)); this module compiles it with gcc and
marshals numpy buffers into it.  What it computes is the plain definition of
attention over a paged KV cache for a packed varlen batch, as described on the
vllm-rlt PR #128 page ("Purpose", prefill bullets: cu_seqlens_q, one block
table per sequence, bottom-right causal alignment, GQA; "Test Plan" item 3:
zero output for empty rows) and the 1Cat-vLLM PR #616 page (fp8_e5m2 KV cache,
page sizes that are multiples of 16, comparison with a dense exact reference).

Parity status: pinned by the CPU tests in ``tests/test_oracle.py`` against an
independent dense brute force, closed forms, the number formats' definitions
and the invariants the pages state.  The pages print no worked example with
concrete input values, so no absolute value from the pages pins the attention
output itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attention_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "e5m2": 3}
_RAW_NP = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "e5m2": np.uint8}

_lock = threading.Lock()
_libs: dict = {}


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_rows", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages_per_row", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
    ]


def compile_source(src: str, out: str) -> str:
    """gcc -O2 (with OpenMP where the compiler has it) into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", tmp, src, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (idempotent: skipped while the library is newer than
    its source)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


SOURCE = _SRC


def _load(path: str | None = None):
    """The compiled oracle (or, for the tests' mutation checks, another build
    of the same source at ``path``)."""
    with _lock:
        key = path or _LIB_PATH
        if key not in _libs:
            lib = ctypes.CDLL(path or build())
            lib.oracle_paged_attention.restype = ctypes.c_int
            lib.oracle_paged_attention.argtypes = [
                ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_decode.argtypes = [ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_void_p]
            lib.oracle_num_threads.restype = ctypes.c_int
            _libs[key] = lib
    return _libs[key]


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _raw(a, dtype: str) -> np.ndarray:
    """Contiguous numpy view of raw storage for the given format name."""
    a = np.ascontiguousarray(a)
    want = _RAW_NP[dtype]
    if a.dtype != want:
        if a.dtype.itemsize != np.dtype(want).itemsize:
            raise TypeError(f"{dtype} storage must have {np.dtype(want).itemsize}-byte items")
        a = a.view(want)
    return a


def decode(raw, dtype: str, *, lib: str | None = None) -> np.ndarray:
    """Exact decode of raw storage (f32/f16/bf16/e5m2) to float64."""
    r = _raw(raw, dtype).reshape(-1)
    out = np.empty(r.size, dtype=np.float64)
    rc = _load(lib).oracle_decode(DTYPE_CODES[dtype], r.ctypes.data, r.size, out.ctypes.data)
    if rc:
        raise ValueError("bad dtype")
    return out.reshape(np.shape(raw))


def paged_attention(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, *,
                    num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                    q_dtype: str, kv_dtype: str, softmax_scale: float | None = None,
                    k_scale: float = 1.0, v_scale: float = 1.0, tokens=None,
                    threads: int = 0, lib: str | None = None) -> np.ndarray:
    """fp64 attention over a paged KV cache.

    q        : raw storage [total_q, Hq, d]
    k_cache  : raw storage [num_pages, page_size, Hkv, d]; v_cache likewise
    block_table : int32 [num_rows, max_pages_per_row]
    cu_seqlens_q: int32 [num_rows + 1];  seq_lens: int32 [num_rows] (total KV
                  length of each row, the new query tokens included)
    tokens   : optional int64 list of global query-token indices to compute
    Returns float64 [n_tokens, Hq, d].
    """
    q = _raw(q, q_dtype)
    k_cache = _raw(k_cache, kv_dtype)
    v_cache = _raw(v_cache, kv_dtype)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    if bt.ndim != 2:
        raise ValueError("block_table must be 2-D")
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_rows = lens.shape[0]
    if cu.shape[0] != num_rows + 1 or bt.shape[0] != num_rows:
        raise ValueError("inconsistent row counts")
    num_pages = k_cache.size // (page_size * num_kv_heads * head_dim)
    for b in range(num_rows):
        qb = int(cu[b + 1] - cu[b])
        L = int(lens[b])
        if qb < 0 or L < 0 or L > bt.shape[1] * page_size:
            raise ValueError(f"row {b}: bad lengths q={qb} L={L}")
        used = (L + page_size - 1) // page_size
        if used and (bt[b, :used].min() < 0 or bt[b, :used].max() >= num_pages):
            raise ValueError(f"row {b}: block table entry out of range")
    if softmax_scale is None or softmax_scale == 0:
        softmax_scale = 1.0 / np.sqrt(head_dim)
    total_q = int(cu[-1]) if num_rows else 0
    if q.size != total_q * num_q_heads * head_dim:
        raise ValueError("q has the wrong size")
    if tokens is None:
        tok = None
        n = total_q
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int64)
        n = tok.size
    out = np.zeros((n, num_q_heads, head_dim), dtype=np.float64)
    prob = _Problem(num_rows, num_q_heads, num_kv_heads, head_dim, page_size, bt.shape[1],
                    DTYPE_CODES[q_dtype], DTYPE_CODES[kv_dtype], float(softmax_scale),
                    float(k_scale), float(v_scale))
    rc = _load(lib).oracle_paged_attention(
        ctypes.byref(prob), cu.ctypes.data, lens.ctypes.data, bt.ctypes.data,
        q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
        None if tok is None else tok.ctypes.data, n, out.ctypes.data, int(threads))
    if rc:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return out
