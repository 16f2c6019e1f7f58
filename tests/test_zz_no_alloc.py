"""paged_attn_decode_static: split-KV decode that allocates nothing.

Some callers cannot allocate device memory (a plugin inside a program that
has reserved all device memory for its own pool, or a C host that must keep
its device memory fixed after start-up), so the library offers one decode
entry point whose scratch lives in a fixed device array instead of a
caller-provided workspace.  This file checks it through the C ABI against the
regular decode call, on two calls in a row (the array keeps the previous
call's contents, so the second call shows that what must start at zero is
cleared).  It is collected last so that a failure here, in a run that stops at
the first failure, comes after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2, "e5m2": 2e-2}


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


@pytest.mark.parametrize("q_dtype,kv_dtype,d", [("bf16", None, 128), ("f16", "e5m2", 256)])
def test_static_decode_matches_regular_decode_twice(lib, q_dtype, kv_dtype, d):
    q_lens = [1, 4, 1, 5, 1, 1]
    kv_lens = [1, 700, 2049, 64, 0, 9000]
    b = workloads.make_batch(q_lens, kv_lens, num_q_heads=8, num_kv_heads=2, head_dim=d,
                             page_size=16, q_dtype=q_dtype, kv_dtype=kv_dtype, seed=31,
                             k_scale=0.5 if kv_dtype else 1.0, v_scale=2.0 if kv_dtype else 1.0,
                             device="cuda")
    need = pa.workspace_size(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q)
    assert need <= pa.STATIC_SCRATCH_BYTES
    ref = pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                               b.seq_lens, softmax_scale=b.softmax_scale, k_scale=b.k_scale,
                               v_scale=b.v_scale)
    torch.cuda.synchronize()
    tol = TOL[kv_dtype or q_dtype]
    for call in range(2):
        out = torch.full_like(b.q, float("nan"))
        assert _static_call(lib, b, out, host=(call == 0)) == 0
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        assert float(np.abs(got - ref.float().cpu().numpy()).max()) <= tol


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
