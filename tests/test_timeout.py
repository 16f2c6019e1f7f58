"""The bounded-wait timeout path, made to run on purpose.

Every wait in the tcgen05 and TMA kernels gives up after a clock limit,
raises PA_DEVERR_TIMEOUT in the workspace header, lets the copies and MMAs
its CTA already started land (drains keep the full limit), frees TMEM and
exits, so a lost arrival ends a kernel with an error flag instead of a hang.
This file builds a second copy of the library in which a wait polls without
suspending and gives up at its first unsuccessful poll (the shipped library
gives up after about two seconds), so waits run out at once, at whatever
point of the pipeline they happen to be.  It
checks, through that copy's C ABI, that each kind of call returns, that the
calls' kernels finish, and that the flag is reported; then that the regular
library, in the same process, still computes the same batches correctly on
fresh workspaces.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

TIMEOUT_FLAG = 0x8


@pytest.fixture(scope="module")
def libs():
    pa_build.build()
    oracle.build()
    path = pa_build.build(variant="timeout", extra_flags=["-DPA_WAIT_LIMIT_CYCLES=0ll",
                                                          "-DPA_WAIT_CHECK_EVERY=1u",
                                                          "-DPA_WAIT_POLL_ONLY"])
    torch.cuda.init()
    return pa.load(), pa.load_library(path)


def call(lib, name, b, ws, **kw):
    prm = pa.make_params(b.q, b.k_cache, softmax_scale=b.softmax_scale, k_scale=b.k_scale,
                         v_scale=b.v_scale, **kw)
    cu_h, lens_h = b.cu_seqlens_q.cpu().contiguous(), b.seq_lens.cpu().contiguous()
    bat = pa.Batch(b.num_rows, b.total_q, b.num_pages, int(b.block_table.shape[1]),
                   b.cu_seqlens_q.data_ptr(), b.seq_lens.data_ptr(), b.block_table.data_ptr(),
                   cu_h.data_ptr(), lens_h.data_ptr())
    out = torch.zeros_like(b.q)
    rc = getattr(lib, name)(ctypes.byref(prm), ctypes.byref(bat), b.q.data_ptr(),
                            b.k_cache.data_ptr(), b.v_cache.data_ptr(), out.data_ptr(),
                            ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()  # the kernels have finished
    return rc, out


def flags(lib, ws):
    v = ctypes.c_uint32(0)
    assert lib.paged_attn_read_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream,
                                      ctypes.byref(v)) == 0
    return int(v.value)


def make(q_lens, kv_lens, d, dtype="bf16", kv_dtype=None, hq=8, hkv=2, seed=50, P=16, **kw):
    return workloads.make_batch(q_lens, kv_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                page_size=P, q_dtype=dtype, kv_dtype=kv_dtype, seed=seed,
                                device="cuda", **kw)


# (entry, batch, params): the two-tile prefill (16-bit and fp8 caches), the
# one-tile d = 256 prefill (16-bit and fp8), the TMA decode, the long-row
# decode splits on the tile kernel, and the large-page instances
CASES = {
    "prefill_d128": ("paged_attn_prefill", lambda: make([300, 200], [3000, 2500], 128), {}),
    "prefill_d128_fp8": ("paged_attn_prefill",
                         lambda: make([300], [3000], 128, "f16", "e5m2", k_scale=0.5, v_scale=2.0),
                         {}),
    "prefill_d256": ("paged_attn_prefill", lambda: make([200], [3000], 256, "f16", hq=12), {}),
    "prefill_d256_fp8": ("paged_attn_prefill",
                         lambda: make([200], [3000], 256, "f16", "e5m2", hq=12, k_scale=0.5,
                                      v_scale=2.0), {}),
    "decode_d128": ("paged_attn_decode", lambda: make([1] * 6 + [4], [5000] * 6 + [900], 128),
                    {}),
    "decode_long_d256": ("paged_attn_decode", lambda: make([1, 4], [40000, 34000], 256, "f16",
                                                          hq=12),
                         {"num_splits": pa.PA_SPLITS_BY_LENGTH}),
    # the large-page instances (a key tile in one page copied in one box per
    # chunk)
    "prefill_d128_pages256": ("paged_attn_prefill", lambda: make([300, 200], [3000, 2500], 128,
                                                                 P=256), {}),
    "prefill_d256_pages784": ("paged_attn_prefill", lambda: make([200], [3000], 256, "f16",
                                                                 hq=12, P=784), {}),
    "prefill_d256_fp8_pages784": ("paged_attn_prefill",
                                  lambda: make([200], [3000], 256, "f16", "e5m2", hq=12,
                                               k_scale=0.5, v_scale=2.0, P=784), {}),
    "decode_long_d256_pages784": ("paged_attn_decode",
                                  lambda: make([1, 4], [40000, 34000], 256, "f16", hq=12, P=784),
                                  {"num_splits": pa.PA_SPLITS_BY_LENGTH}),
}


@pytest.mark.parametrize("case", list(CASES))
def test_waits_that_run_out_end_the_call_with_the_timeout_flag(libs, case):
    reg, tlib = libs
    name, mk, kw = CASES[case]
    b = mk()
    prm = pa.make_params(b.q, b.k_cache, **kw)
    # the timeout build: the call returns, its kernels end, the flag is set.
    # The L2 is flushed first, so the first copies come from DRAM and arrive
    # well after the first poll of their barrier.
    ws = torch.zeros(pa.workspace_size(prm, b.num_rows, b.total_q), dtype=torch.uint8,
                     device="cuda")
    torch.empty(256 << 20, dtype=torch.uint8, device="cuda").fill_(1)
    torch.cuda.synchronize()
    rc, _ = call(tlib, name, b, ws, **kw)
    assert rc == 0
    assert flags(tlib, ws) & TIMEOUT_FLAG
    # twice more on the same workspace: work counters left by the aborted
    # call do not stop the next one from finishing
    for _ in range(2):
        rc, _ = call(tlib, name, b, ws, **kw)
        assert rc == 0
    flags(tlib, ws)
    # the regular library on a fresh workspace: correct results, no flags
    ws2 = torch.zeros_like(ws)
    rc, out = call(reg, name, b, ws2, **kw)
    assert rc == 0
    assert flags(reg, ws2) == 0
    toks = sorted({0, b.total_q // 2, b.total_q - 1})
    ref = oracle.paged_attention(tokens=toks, **b.oracle_args())
    tol = 2e-2 if b.kv_dtype == "e5m2" else 1e-2
    err = float(np.abs(out[toks].float().cpu().numpy() - ref).max())
    assert err <= tol
