"""Prefill work items cut into key-range parts (prefill_kv_parts), against
the fp64 oracle.

A work item whose rows see more than 16384 keys runs as several CTAs over
equal runs of whole 128-key units, merged by log-sum-exp in fixed order
(1Cat-vLLM PR #1279, commit 5).  Checked here: every cut path against the
oracle (tokens sampled along long rows, all tokens of short ones), the cut
result against the uncut one, the invariants that still hold bitwise (page
size, physical-page order, a row alone vs in a batch, repeated calls, with
and without host mirrors, mixed vs prefill), and that paths which do not cut
(fp32, fp8 caches at d = 64 / 256) give the uncut bits.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-5, "e5m2": 2e-2}
ENTRY = {"prefill": pa.paged_attn_prefill, "mixed": pa.paged_attn_mixed}

# row 0: 3 parts (40000 keys); row 1: 2 parts (16500); row 2: not cut;
# row 3: empty; row 4: a short row whose queries are all its keys
Q_LENS = [300, 65, 100, 0, 20]
KV_LENS = [40000, 16500, 5000, 0, 20]


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()
    oracle.build()
    torch.cuda.init()


def batch(q_lens=Q_LENS, kv_lens=KV_LENS, *, d=128, dtype="bf16", kv=None, P=16, seed=31,
          hq=8, hkv=2, **kw):
    cpu = workloads.make_batch(q_lens, kv_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                               page_size=P, q_dtype=dtype, kv_dtype=kv, seed=seed,
                               k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0, **kw)
    return cpu, cpu.to("cuda")


def run(entry, b, parts, host=True, num_splits=0):
    extra = {}
    if host:
        extra = dict(cu_seqlens_q_host=b.cu_seqlens_q.cpu(), seq_lens_host=b.seq_lens.cpu())
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache, prefill_kv_parts=parts,
                                          num_splits=num_splits), b.num_rows, b.total_q, "cuda")
    out = ENTRY[entry](b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens,
                       softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale,
                       prefill_kv_parts=parts, num_splits=num_splits, workspace=ws, **extra)
    torch.cuda.synchronize()
    assert pa.read_errors(ws) == 0
    return out


def sampled(q_lens, every=13, edge=6):
    toks, base = [], 0
    for q in q_lens:
        idx = set(range(min(edge, q))) | set(range(max(0, q - edge), q)) | set(range(0, q, every))
        toks += [base + i for i in sorted(idx)]
        base += q
    return toks


def err(out, ref):
    o = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all()
    return float(np.abs(o - ref).max())


def bitwise(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("dtype,kv,d", [("bf16", None, 128), ("f16", None, 128),
                                        ("bf16", None, 64), ("f16", None, 256),
                                        ("bf16", None, 256), ("f16", "e5m2", 128),
                                        ("bf16", "e5m2", 128), ("f16", "e5m2", 256),
                                        ("bf16", "e5m2", 256)])
def test_cut_items_match_oracle(dtype, kv, d):
    cpu, gpu = batch(d=d, dtype=dtype, kv=kv, seed=31 + d)
    tol = TOL["e5m2" if kv else dtype]
    cut = run("prefill", gpu, parts=4)
    whole = run("prefill", gpu, parts=0)
    toks = sampled(Q_LENS)
    ref = oracle.paged_attention(tokens=toks, **cpu.oracle_args())
    assert err(cut[toks], ref) <= tol
    assert err(whole[toks], ref) <= tol
    # the cut and uncut results differ by rounding only
    assert float((cut.float() - whole.float()).abs().max()) <= tol
    assert not bitwise(cut, whole)
    # the empty row's tokens do not exist; the short uncut rows are untouched
    assert bitwise(cut[365:465], whole[365:465]) and bitwise(cut[465:], whole[465:])


@pytest.mark.parametrize("dtype,kv,d", [("f32", None, 128), ("f16", "e5m2", 64),
                                        ("bf16", "e5m2", 64)])
def test_paths_that_do_not_cut_ignore_the_field(dtype, kv, d):
    ql, kl = [40, 3], [17000, 17000]
    cpu, gpu = batch(ql, kl, d=d, dtype=dtype, kv=kv, seed=41)
    assert bitwise(run("prefill", gpu, parts=8), run("prefill", gpu, parts=0))


def test_cap_on_parts_and_long_row():
    # 60000 keys would make 4 parts; K = 2 caps it (two parts of ~30000)
    ql, kl = [129, 40], [60000, 33000]
    cpu, gpu = batch(ql, kl, seed=43)
    toks = sampled(ql, every=11)
    ref = oracle.paged_attention(tokens=toks, **cpu.oracle_args())
    for k in (2, 3, 16):
        assert err(run("prefill", gpu, parts=k)[toks], ref) <= TOL["bf16"]


def test_invariants_bitwise_with_parts():
    base = run("prefill", batch(P=16)[1], parts=4)
    for P in (48, 784):
        assert bitwise(run("prefill", batch(P=P)[1], parts=4), base)
    assert bitwise(run("prefill", batch(P=16, perm_seed=9)[1], parts=4), base)
    cpu, gpu = batch(P=16)
    assert bitwise(run("prefill", gpu, parts=4, host=False), base)
    assert bitwise(run("prefill", gpu, parts=4), base)
    cu = cpu.cu_seqlens_q.tolist()
    for r in (0, 1, 4):
        alone = run("prefill", workloads.sub_batch(cpu, [r]).to("cuda"), parts=4)
        assert bitwise(alone, base[cu[r]:cu[r + 1]])


def test_mixed_with_parts_and_decode_rows():
    # decode rows next to cut prefill rows: the decode rows are untouched by
    # the field, the prefill rows equal the prefill call's, bitwise
    ql, kl = [300, 1, 4, 65, 5], [40000, 20000, 30000, 16500, 100]
    cpu, gpu = batch(ql, kl, seed=47)
    mixed = run("mixed", gpu, parts=8)
    plain = run("mixed", gpu, parts=0)
    assert bitwise(mixed[300:305], plain[300:305])
    assert bitwise(mixed[305:305 + 65 + 5][-5:], plain[305:305 + 65 + 5][-5:])
    pre = run("prefill", workloads.sub_batch(cpu, [0, 3]).to("cuda"), parts=8)
    assert bitwise(mixed[:300], pre[:300])
    assert bitwise(mixed[305:370], pre[300:])
    toks = sampled(ql, every=29)
    ref = oracle.paged_attention(tokens=toks, **cpu.oracle_args())
    assert err(mixed[toks], ref) <= TOL["bf16"]


def test_mixed_workload_with_parts():
    # the mixed serving batch (a 2048-token chunk after 150,000 keys, three
    # rows at 240,000 keys with q = 1, 4, 5; d = 256, fp16): pages of 784 and
    # 896 give the same bits with parts, sampled tokens match the oracle
    outs = {}
    for P in (784, 896):
        gpu = workloads.make_workload(3, device="cuda", data_device="cuda", page_size=P)
        outs[P] = run("mixed", gpu, parts=8)
        if P == 784:
            cpu0 = workloads.sub_batch(gpu, [0])
            toks = [0, 1, 700, 1500, 2047]
            ref = oracle.paged_attention(tokens=toks, **cpu0.oracle_args())
            assert err(outs[P][toks], ref) <= TOL["f16"]
        del gpu
        torch.cuda.empty_cache()
    assert bitwise(outs[896], outs[784])


def _run_auto(entry, b, host=True):
    return run(entry, b, parts=pa.PA_PREFILL_PARTS_AUTO, host=host)


def test_auto_part_count_on_the_long_chunk():
    # the 2048-token chunk after 150,000 keys (d = 256, 384 equal CTAs = 2.5
    # waves on 152 SMs): the count chosen per call cuts it in 3 (the fewest
    # finish-time CTA waves), which equals the explicit 3-part cut here
    gpu = workloads.make_workload(3, device="cuda", data_device="cuda", page_size=784)
    row = workloads.sub_batch(gpu, [0], device="cuda")
    auto = _run_auto("prefill", row)
    assert bitwise(auto, run("prefill", row, parts=3))
    assert not bitwise(auto, run("prefill", row, parts=0))
    toks = [0, 1, 1000, 2047]
    ref = oracle.paged_attention(tokens=toks, **workloads.sub_batch(gpu, [0]).oracle_args())
    assert err(auto[toks], ref) <= TOL["f16"]
    # with decode rows beside it (the mixed call) or without host mirrors,
    # nothing is cut
    assert bitwise(_run_auto("mixed", gpu), run("mixed", gpu, parts=0))
    assert bitwise(_run_auto("prefill", row, host=False), run("prefill", row, parts=0))
    # unless the decode rows' long splits are short tile-kernel items
    # (PA_SPLITS_BY_LENGTH): then the chunk is cut in 3 there too
    by_len = pa.PA_SPLITS_BY_LENGTH
    mixed = run("mixed", gpu, parts=pa.PA_PREFILL_PARTS_AUTO, num_splits=by_len)
    assert bitwise(mixed, run("mixed", gpu, parts=3, num_splits=by_len))
    assert bitwise(mixed[:2048], auto)
    del gpu, row
    torch.cuda.empty_cache()


def test_auto_part_count_leaves_many_waves_alone():
    # the varlen prefill batch runs 960 CTAs (6.3 waves): not cut
    gpu = workloads.make_workload(2, device="cuda", data_device="cuda")
    assert bitwise(_run_auto("prefill", gpu), run("prefill", gpu, parts=0))
    del gpu
    torch.cuda.empty_cache()
