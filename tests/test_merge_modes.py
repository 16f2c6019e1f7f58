"""The split-KV merge in the decode launch itself (merge_mode =
PA_MERGE_SAME_LAUNCH) against the separate merge kernel (PA_MERGE_SEPARATE),
through the C ABI: the same bits on every decode case -- every head dim and
cache type of the decode kernel, verify rows packed and one token at a time,
the decode batch with the longest-split-first work order, the five-row
decode-only workload, the 256-row split-KV workload (whose grid fills the
GPU) and the long-context fp8 workload -- and the default choice
(PA_MERGE_AUTO) equals both (vllm-rlt PR #128, Test Result: the same-launch
merge is bitwise identical to the two-kernel path).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

SEP, SAME, AUTO = pa.PA_MERGE_SEPARATE, pa.PA_MERGE_SAME_LAUNCH, pa.PA_MERGE_AUTO


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()
    oracle.build()
    torch.cuda.init()


def run(b, mode, host=True, static=False, **kw):
    extra = {}
    if host:
        extra = dict(cu_seqlens_q_host=b.cu_seqlens_q.cpu(), seq_lens_host=b.seq_lens.cpu())
    fn = pa.paged_attn_decode_static if static else pa.paged_attn_decode
    out = fn(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens,
             softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale,
             merge_mode=mode, **extra, **kw)
    torch.cuda.synchronize()
    return out


def same_bits(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def check(b, **kw):
    sep = run(b, SEP, **kw)
    assert same_bits(run(b, SAME, **kw), sep)
    assert same_bits(run(b, AUTO, **kw), sep)
    assert same_bits(run(b, SAME, host=False, **kw), sep)
    return sep


DECODE_LENS = [0, 1, 31, 32, 33, 511, 512, 513, 4097, 10000]


@pytest.mark.parametrize("dtype,kv,d", [("bf16", None, 64), ("bf16", None, 128),
                                        ("f16", None, 256), ("f16", "e5m2", 128),
                                        ("bf16", "e5m2", 256)])
def test_same_launch_merge_bitwise_small(dtype, kv, d):
    ql = [1, 1, 1, 1, 4, 5, 1, 16, 4, 1]
    b = workloads.make_batch(ql, DECODE_LENS, num_q_heads=8, num_kv_heads=2, head_dim=d,
                             page_size=16, q_dtype=dtype, kv_dtype=kv, seed=3 * d,
                             k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0)
    g = b.to("cuda")
    out = check(g)
    ref = oracle.paged_attention(**b.oracle_args())
    tol = 2e-2 if kv else 1e-2
    assert float(np.abs(out.float().cpu().numpy() - ref).max()) <= tol
    # one token at a time, and the entry without a workspace
    check(g, verify_mode=pa.PA_VERIFY_TOKENWISE)
    assert same_bits(run(g, SAME, static=True), out)


def test_same_launch_merge_bitwise_work_order():
    # 40 rows: the decode rows are handed out longest split first
    gen = torch.Generator().manual_seed(77)
    kl = torch.randint(0, 3000, (40,), generator=gen).tolist()
    kl[:4] = [0, 1, 2999, 64]
    ql = [1 + (i % 3 == 0) for i in range(40)]
    b = workloads.make_batch(ql, kl, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                             q_dtype="f16", seed=31, device="cuda")
    check(b)


@pytest.mark.parametrize("n", [1, 4, 5])
def test_same_launch_merge_bitwise_workloads(n):
    b = workloads.make_workload(n, device="cuda", data_device="cuda")
    check(b)
