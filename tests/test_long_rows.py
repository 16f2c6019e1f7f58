"""GPU parity of the length-only split count for long decode rows
(num_splits = PA_SPLITS_BY_LENGTH), through the C ABI, against the fp64
oracle.

A decode row of at most 32768 keys keeps the 16-part partition (bitwise the
same result as the default); a longer row is cut into parts of 2048 keys
(whole 128-key tiles).  At d = 256 with a 16-bit cache the parts run on the
tcgen05 tile kernel, one 128-row tile holding all of the row's GQA-packed
query rows; with an fp8 cache or another head dim they run on the decode
kernel.  The count depends on the row's length alone, so the invariances the
pages require still hold bitwise: page size, physical page order, a row alone
vs in a batch, the mixed call vs the decode call, with and without host
mirrors.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2}
BY_LEN = pa.PA_SPLITS_BY_LENGTH
ENTRY = {"decode": pa.paged_attn_decode, "mixed": pa.paged_attn_mixed,
         "prefill": pa.paged_attn_prefill}


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()
    oracle.build()
    torch.cuda.init()


def run(entry, b, host=True, **kw):
    extra = {}
    if host:
        extra = dict(cu_seqlens_q_host=b.cu_seqlens_q.cpu(), seq_lens_host=b.seq_lens.cpu())
    out = ENTRY[entry](b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens,
                       softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale,
                       **extra, **kw)
    torch.cuda.synchronize()
    return out


def max_err(out, ref):
    o = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all(), "non-finite output"
    return float(np.abs(o - ref).max())


def same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def batch(q_lens, kv_lens, dtype="f16", P=16, hq=12, hkv=2, seed=0, d=256, **kw):
    return workloads.make_batch(q_lens, kv_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                page_size=P, q_dtype=dtype, seed=seed, device="cuda",
                                data_device="cuda", **kw)


# long rows (q = 1 decode and q = 4/5 verify rows, one ending mid-tile) next
# to short ones, one of exactly 32768 keys (the last length with 16 parts)
Q_LENS = [1, 4, 5, 1, 2, 1]
KV_LENS = [40000, 70001, 33000, 500, 32768, 32769]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_long_rows_match_oracle(dtype):
    b = batch(Q_LENS, KV_LENS, dtype=dtype, seed=41)
    out = run("decode", b, num_splits=BY_LEN)
    ref = oracle.paged_attention(**b.oracle_args())
    assert max_err(out, ref) <= TOL[dtype]
    # rows of at most 32768 keys: bitwise the default partition's result
    dflt = run("decode", b)
    cu = np.cumsum([0] + Q_LENS)
    for r, L in enumerate(KV_LENS):
        s = slice(cu[r], cu[r + 1])
        if L <= 32768:
            assert same_bits(out[s], dflt[s]), r
    assert max_err(dflt, ref) <= TOL[dtype]


def test_long_rows_invariances_bitwise():
    b = batch(Q_LENS, KV_LENS, seed=42)
    ref = run("decode", b, num_splits=BY_LEN)
    # no host mirrors (device-built work list, persistent grid)
    assert same_bits(run("decode", b, host=False, num_splits=BY_LEN), ref)
    # the mixed call (routing on the device), with and without mirrors
    assert same_bits(run("mixed", b, num_splits=BY_LEN), ref)
    assert same_bits(run("mixed", b, host=False, num_splits=BY_LEN), ref)
    # page size and physical page order
    for P, perm in ((784, None), (816, 7), (896, 11)):
        o = run("decode", batch(Q_LENS, KV_LENS, P=P, seed=42, perm_seed=perm), num_splits=BY_LEN)
        assert same_bits(o, ref), P
    # each row alone
    cu = np.cumsum([0] + Q_LENS)
    for r in range(len(Q_LENS)):
        alone = run("decode", workloads.sub_batch(b, [r], device="cuda"), num_splits=BY_LEN)
        assert same_bits(alone, ref[cu[r]:cu[r + 1]]), r
    # repeated calls on one workspace
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache, num_splits=BY_LEN), b.num_rows,
                           b.total_q, "cuda")
    for _ in range(3):
        assert same_bits(run("decode", b, num_splits=BY_LEN, workspace=ws), ref)
    assert pa.read_errors(ws) == 0


def test_long_rows_in_a_mixed_batch_with_a_prefill_row():
    # a prefill row next to long decode rows: the decode rows' bits are the
    # decode call's, the prefill row's the prefill call's
    q_lens, kv_lens = [300, 1, 5], [5000, 50000, 45000]
    b = batch(q_lens, kv_lens, seed=43)
    out = run("mixed", b, num_splits=BY_LEN)
    dec = run("decode", workloads.sub_batch(b, [1, 2], device="cuda"), num_splits=BY_LEN)
    pre = run("prefill", workloads.sub_batch(b, [0], device="cuda"))
    assert same_bits(out[300:], dec)
    assert same_bits(out[:300], pre)
    ref = oracle.paged_attention(tokens=list(range(290, 306)), **b.oracle_args())
    assert max_err(out[290:306], ref) <= TOL["f16"]


def test_long_rows_running_maximum_grows_along_the_row():
    # keys ramped along the row (and every query aligned with the ramp's
    # direction) so that every row's running maximum passes its exponent
    # reference by more than 2^8 inside the parts: the lazy O rescale of the
    # long-row kernel, and the merge of parts whose maxima differ widely
    q_lens, kv_lens = [1, 4], [36000, 41000]
    b = batch(q_lens, kv_lens, seed=44)
    P = b.page_size
    k = b.k_cache.view(-1, b.num_kv_heads, 256)
    for r, L in enumerate(kv_lens):
        j = torch.arange(L, device="cuda")
        phys = b.block_table[r, (j // P).long()].long() * P + (j % P)
        ramp = (j.float() / L * 64.0).view(-1, 1, 1)
        k[phys] = (k[phys].float() * 0.25 + ramp * 0.5).to(k.dtype)
    b.q.copy_((b.q.float() * 0.3 + 0.5).to(b.q.dtype))
    out = run("decode", b, num_splits=BY_LEN)
    ref = oracle.paged_attention(**b.oracle_args())
    assert max_err(out, ref) <= TOL["f16"]


def test_workload3_decode_rows_by_length():
    # the mixed workload's three resident rows (240000 keys, q = 1/4/5, 24/4
    # heads), whole, at page 784 and 896
    outs = {}
    for P in (784, 896):
        full = workloads.make_workload(3, device="cuda", data_device="cuda", page_size=P)
        b = workloads.sub_batch(full, [1, 2, 3], device="cuda")
        del full
        torch.cuda.empty_cache()
        outs[P] = run("decode", b, num_splits=BY_LEN)
        if P == 784:
            ref = oracle.paged_attention(**b.oracle_args())
            assert max_err(outs[P], ref) <= TOL["f16"]
            assert same_bits(run("decode", b, host=False, num_splits=BY_LEN), outs[P])
        del b
        torch.cuda.empty_cache()
    assert same_bits(outs[896], outs[784])


# the decode kernel's cases: an fp8 cache (d = 256 and 128) and 16-bit caches
# at d = 64 and 128
DEC_CASES = {
    "e5m2_d256": dict(dtype="f16", d=256, kv_dtype="e5m2", k_scale=0.5, v_scale=2.0),
    "e5m2_d128": dict(dtype="bf16", d=128, kv_dtype="e5m2", k_scale=0.37, v_scale=1.7),
    "bf16_d128": dict(dtype="bf16", d=128, hq=8),
    "f16_d64": dict(dtype="f16", d=64, hq=8),
}


@pytest.mark.parametrize("case", list(DEC_CASES))
def test_long_rows_on_the_decode_kernel(case):
    kw = dict(DEC_CASES[case])
    tol = 2e-2 if kw.get("kv_dtype") else 1e-2
    b = batch(Q_LENS, KV_LENS, seed=45, **kw)
    out = run("decode", b, num_splits=BY_LEN)
    ref = oracle.paged_attention(**b.oracle_args())
    assert max_err(out, ref) <= tol
    # rows of at most 32768 keys: bitwise the default partition's result
    dflt = run("decode", b)
    cu = np.cumsum([0] + Q_LENS)
    for r, L in enumerate(KV_LENS):
        if L <= 32768:
            assert same_bits(out[cu[r]:cu[r + 1]], dflt[cu[r]:cu[r + 1]]), r
    # without host mirrors (128 split indices per row), the mixed call
    assert same_bits(run("decode", b, host=False, num_splits=BY_LEN), out)
    assert same_bits(run("mixed", b, num_splits=BY_LEN), out)
    assert same_bits(run("mixed", b, host=False, num_splits=BY_LEN), out)
    # page size and page order, and each long row alone
    o = run("decode", batch(Q_LENS, KV_LENS, P=800, seed=45, perm_seed=5, **kw),
            num_splits=BY_LEN)
    assert same_bits(o, out)
    for r in (1, 5):
        alone = run("decode", workloads.sub_batch(b, [r], device="cuda"), num_splits=BY_LEN)
        assert same_bits(alone, out[cu[r]:cu[r + 1]]), r


def test_workload5_by_length_sampled():
    # the long-context fp8 workload (64 rows of 128000-240000 keys) whole,
    # sampled tokens against the oracle, and bitwise without host mirrors
    b = workloads.make_workload(5, device="cuda", data_device="cuda")
    out = run("decode", b, num_splits=BY_LEN)
    toks = [0, 1, b.total_q // 2, b.total_q - 1]
    ref = oracle.paged_attention(tokens=toks, **b.oracle_args())
    assert max_err(out[toks], ref) <= 2e-2
    assert same_bits(run("decode", b, host=False, num_splits=BY_LEN), out)
    del b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", ["tile_f16_d256", "decode_e5m2_d128"])
def test_rows_past_the_part_cap(case):
    # rows over 262144 keys: at most 128 parts, so the parts grow past 2048
    # keys (whole 128-key tiles); sampled tokens against the oracle, bitwise
    # without host mirrors and row alone vs in the batch
    if case == "tile_f16_d256":
        kw = dict(dtype="f16", d=256, hq=8, hkv=2)
        tol = TOL["f16"]
    else:
        kw = dict(dtype="bf16", d=128, hq=8, hkv=2, kv_dtype="e5m2", k_scale=0.37, v_scale=1.7)
        tol = 2e-2
    q_lens, kv_lens = [1, 4, 1], [300000, 270001, 5000]
    b = batch(q_lens, kv_lens, seed=47, **kw)
    out = run("decode", b, num_splits=BY_LEN)
    toks = [0, 1, 4, 5]
    ref = oracle.paged_attention(tokens=toks, **b.oracle_args())
    assert max_err(out[toks], ref) <= tol
    assert same_bits(run("decode", b, host=False, num_splits=BY_LEN), out)
    alone = run("decode", workloads.sub_batch(b, [1], device="cuda"), num_splits=BY_LEN)
    assert same_bits(alone, out[1:5])
    del b
    torch.cuda.empty_cache()
