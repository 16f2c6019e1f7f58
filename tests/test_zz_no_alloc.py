"""paged_attn_decode_static: split-KV decode that allocates nothing.

Some callers cannot allocate device memory (a plugin inside a program that
has reserved all device memory for its own pool, or a C host that must keep
its device memory fixed after start-up), so the library offers one decode
entry point whose scratch lives in a fixed device array instead of a
caller-provided workspace.  This file checks it through the C ABI against the
regular decode call, bit for bit, on two calls in a row after a call on an
unrelated batch (the array keeps the previous call's contents, so this shows
that what must start at zero is cleared and that stale partial states never
reach a result), and checks that its sticky error flag reports a bad
block-table entry.  It is collected last so that a failure here, in a run that stops at
the first failure, comes after every other test.
"""
import ctypes
import dataclasses

import pytest
import torch

import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

def _batch_structs(b, host=True):
    prm = pa.make_params(b.q, b.k_cache, softmax_scale=b.softmax_scale, k_scale=b.k_scale,
                         v_scale=b.v_scale)
    cu_h = b.cu_seqlens_q.cpu().contiguous()
    lens_h = b.seq_lens.cpu().contiguous()
    bat = pa.Batch(b.num_rows, b.total_q, b.num_pages, int(b.block_table.shape[1]),
                   b.cu_seqlens_q.data_ptr(), b.seq_lens.data_ptr(), b.block_table.data_ptr(),
                   cu_h.data_ptr() if host else None, lens_h.data_ptr() if host else None)
    return prm, bat, (cu_h, lens_h)


def _static_call(lib, b, out, host=True):
    prm, bat, keep = _batch_structs(b, host)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.paged_attn_decode_static(ctypes.byref(prm), ctypes.byref(bat), b.q.data_ptr(),
                                      b.k_cache.data_ptr(), b.v_cache.data_ptr(),
                                      out.data_ptr(), stream)
    torch.cuda.synchronize()
    del keep
    return rc


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    torch.cuda.init()
    return pa.load()


def _read_static_errors(lib):
    """Reads and clears the sticky error word of the static call's array."""
    v = ctypes.c_uint32(0)
    rc = lib.paged_attn_read_errors(None, torch.cuda.current_stream().cuda_stream,
                                    ctypes.byref(v))
    assert rc == 0
    return int(v.value)


@pytest.mark.parametrize("q_dtype,kv_dtype,d", [("bf16", None, 128), ("f16", "e5m2", 256)])
def test_static_decode_matches_regular_decode_twice(lib, q_dtype, kv_dtype, d):
    kw = dict(head_dim=d, page_size=16, q_dtype=q_dtype, kv_dtype=kv_dtype,
              k_scale=0.5 if kv_dtype else 1.0, v_scale=2.0 if kv_dtype else 1.0, device="cuda")
    # an unrelated batch first (other lengths and head counts), so that the
    # array holds partial states and work counts that have nothing to do with
    # the batch under test when the two calls below run
    other = workloads.make_batch([3, 1, 2, 1], [5000, 17, 900, 64], num_q_heads=16,
                                 num_kv_heads=4, seed=30, **kw)
    assert _static_call(lib, other, torch.empty_like(other.q)) == 0
    b = workloads.make_batch([1, 4, 1, 5, 1, 1], [1, 700, 2049, 64, 0, 9000], num_q_heads=8,
                             num_kv_heads=2, seed=31, **kw)
    need = pa.workspace_size(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q)
    assert need <= pa.STATIC_SCRATCH_BYTES
    ref = pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                               b.seq_lens, softmax_scale=b.softmax_scale, k_scale=b.k_scale,
                               v_scale=b.v_scale)
    torch.cuda.synchronize()
    # the same kernels on the same arithmetic: bit for bit, with and without
    # the host mirrors
    for call in range(2):
        out = torch.full_like(b.q, float("nan"))
        assert _static_call(lib, b, out, host=(call == 0)) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}"
    assert _read_static_errors(lib) == 0


def test_static_decode_reports_a_bad_block_table_entry(lib):
    # without host mirrors only the kernels see the bad entry: they must not
    # read through it and must raise the sticky flag in the array's header
    b = workloads.make_batch([1, 1], [40, 60], num_q_heads=8, num_kv_heads=2, head_dim=128,
                             page_size=16, q_dtype="bf16", seed=33, device="cuda")
    bt = b.block_table.clone()
    bt[1, 2] = 10 ** 6
    bad = dataclasses.replace(b, block_table=bt)
    _read_static_errors(lib)  # start clean
    assert _static_call(lib, bad, torch.empty_like(b.q), host=False) == 0
    assert _read_static_errors(lib) & 0x1
    assert _read_static_errors(lib) == 0   # cleared by the read
    # and the array then serves a good call as before
    out = torch.empty_like(b.q)
    assert _static_call(lib, b, out) == 0
    ref = pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                               b.seq_lens)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert _read_static_errors(lib) == 0


def test_static_decode_refuses_batches_beyond_its_array(lib):
    # 96 rows x 32 heads x 16 splits x (128 + 2) x 4 B of partial state: 25.6 MB > 16 MiB
    b = workloads.make_batch([1] * 96, [32] * 96, num_q_heads=32, num_kv_heads=8,
                             head_dim=128, page_size=16, q_dtype="bf16", seed=32,
                             device="cuda")
    need = pa.workspace_size(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q)
    assert need > pa.STATIC_SCRATCH_BYTES
    out = torch.zeros_like(b.q)
    assert _static_call(lib, b, out) == 3  # PA_ERR_WORKSPACE_TOO_SMALL, nothing launched
    assert bool((out == 0).all())
