"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Tolerances (max-abs error against the oracle): 1e-2 for bf16/fp16 inputs,
2e-2 for an fp8 E5M2 KV cache, 1e-5 for fp32.  Invariants the pages state are
checked bitwise: page size, physical-page order, a row alone vs in a batch,
the mixed call vs the single-path calls, repeated calls; empty rows give
exact zeros and poisoned (even NaN) cache slots outside the rows never leak.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f16": 1e-2, "f32": 1e-5, "e5m2": 2e-2}
ENTRY = {"prefill": pa.paged_attn_prefill, "decode": pa.paged_attn_decode,
         "mixed": pa.paged_attn_mixed}


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()
    oracle.build()
    torch.cuda.init()


def tol_of(b):
    return TOL["e5m2"] if b.kv_dtype == "e5m2" else TOL[b.q_dtype]


def run(entry, b, host=True, **kw):
    """Runs one entry point on batch b (already on the GPU)."""
    extra = {}
    if host:
        extra = dict(cu_seqlens_q_host=b.cu_seqlens_q.cpu(), seq_lens_host=b.seq_lens.cpu())
    out = ENTRY[entry](b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens,
                       softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale,
                       **extra, **kw)
    torch.cuda.synchronize()
    return out


def ref_of(b, tokens=None):
    return oracle.paged_attention(tokens=tokens, **b.oracle_args())


def max_err(out, ref):
    o = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o).all(), "non-finite output"
    return float(np.abs(o - ref).max()) if o.size else 0.0


def small(q_lens, kv_lens, *, hq=8, hkv=2, d=128, P=16, dtype="bf16", kv_dtype=None, seed=0,
          **kw):
    b = workloads.make_batch(q_lens, kv_lens, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                             page_size=P, q_dtype=dtype, kv_dtype=kv_dtype, seed=seed, **kw)
    return b, b.to("cuda")


def assert_bitwise(a, b):
    assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                       b.view(torch.uint8) if b.dtype != torch.uint8 else b)


# --------------------------------------------------------------------------
# small ragged cases, every path, every dtype / head dim
# --------------------------------------------------------------------------

PREFILL_LENS = ([65, 130, 1, 7, 200, 64], [65, 500, 1, 40, 1000, 64])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 1), (4, 4)])
def test_prefill_small(dtype, d, hq, hkv):
    cpu, gpu = small(*PREFILL_LENS, hq=hq, hkv=hkv, d=d, P=32, dtype=dtype, seed=d + hq)
    out = run("prefill", gpu)
    assert max_err(out, ref_of(cpu)) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_prefill_fp8_cache(dtype, d):
    # E5M2 K/V with per-tensor scales on the prefill path: ragged rows (a
    # partial last page slot, q > L, several 128-key tiles), page-size
    # invariance bitwise, NaN poison in unused slots never reaching the output
    ql, kl = [65, 300, 3, 129, 40], [65, 1500, 1, 700, 33]
    outs = {}
    for P in (16, 48):
        cpu, gpu = small(ql, kl, hq=8, hkv=2, d=d, P=P, dtype=dtype, kv_dtype="e5m2",
                         seed=5 + d, k_scale=0.37, v_scale=1.7,
                         poison="nan" if P == 48 else "finite")
        outs[P] = run("prefill", gpu)
        if P == 16:
            assert max_err(outs[P], ref_of(cpu)) <= TOL["e5m2"]
    assert_bitwise(outs[48], outs[16])


@pytest.mark.parametrize("dtype,kv,d", [("bf16", None, 64), ("bf16", None, 128),
                                        ("f16", "e5m2", 128), ("f16", None, 256),
                                        ("bf16", None, 256), ("f16", "e5m2", 256)])
def test_prefill_whole_tile_copies(dtype, kv, d):
    # pages that can hold a whole 128-key tile: a tile (or V half) whose keys
    # lie in one page is copied with one box per 128-byte chunk instead of one
    # per 16-token slot.  Pages of 128 tokens (every full tile inside a page),
    # 144 (tiles across page boundaries) and 784, shuffled page order, rows
    # ending mid-slot, NaN in the unused slots: bitwise the result with
    # 16-token pages, which is within tolerance of the oracle
    ql, kl = [65, 300, 3, 129, 600], [65, 1500, 1, 700, 2000]
    kw = dict(hq=8, hkv=2, d=d, dtype=dtype, kv_dtype=kv, seed=60 + d,
              k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0)
    cpu, gpu = small(ql, kl, P=16, **kw)
    base = run("prefill", gpu)
    assert max_err(base, ref_of(cpu)) <= TOL[kv or dtype]
    for P in (128, 144, 784):
        for perm in (None, 3):
            _, g = small(ql, kl, P=P, perm_seed=perm, poison="nan", **kw)
            assert_bitwise(run("prefill", g), base)


@pytest.mark.parametrize("dtype,kv,d", [("bf16", None, 128), ("f16", "e5m2", 128),
                                        ("f16", None, 256), ("f16", "e5m2", 256)])
def test_whole_tile_copies_with_key_range_parts(dtype, kv, d):
    # key-range parts (whole 128-key units) start their copies mid-row: with
    # pages of 256 and 784 tokens the parts' tiles take the whole-tile boxes
    # where they lie in one page; bitwise the 16-token-page result, itself
    # within tolerance of the oracle; and a mixed call (decode rows beside the
    # cut prefill rows) bitwise its single-path calls
    ql, kl = [700, 1, 4, 300], [9000, 3000, 2500, 6000]
    kw = dict(hq=8, hkv=2, d=d, dtype=dtype, kv_dtype=kv, seed=90 + d,
              k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0)
    cpu, gpu = small(ql, kl, P=16, **kw)
    base = run("mixed", gpu, prefill_kv_parts=3)
    toks = [0, 350, 699, 700, 701, 705, 1004]
    assert max_err(base[toks], ref_of(cpu, toks)) <= TOL[kv or dtype]
    for P in (256, 784):
        _, g = small(ql, kl, P=P, perm_seed=9, **kw)
        assert_bitwise(run("mixed", g, prefill_kv_parts=3), base)
    pre = run("prefill", workloads.sub_batch(cpu, [0, 3]).to("cuda"), prefill_kv_parts=3)
    assert_bitwise(base[:700], pre[:700])
    assert_bitwise(base[705:], pre[700:])


DECODE_LENS = [0, 1, 31, 32, 33, 511, 512, 513, 4097, 10000]


@pytest.mark.parametrize("dtype,kv", [("bf16", None), ("f16", None), ("f32", None),
                                      ("f16", "e5m2"), ("bf16", "e5m2")])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_small(dtype, kv, d):
    ql = [1, 1, 1, 1, 4, 5, 1, 16, 4, 1]      # row 0: L = 0, an empty row
    cpu, gpu = small(ql, DECODE_LENS, hq=8, hkv=2, d=d, P=16, dtype=dtype, kv_dtype=kv,
                     seed=3 * d, k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0)
    out = run("decode", gpu)
    tol = TOL["e5m2"] if kv else TOL[dtype]
    assert max_err(out, ref_of(cpu)) <= tol


@pytest.mark.parametrize("entry", ["decode", "mixed"])
@pytest.mark.parametrize("kv", [None, "e5m2"])
def test_decode_many_rows_work_order(entry, kv):
    # enough rows that the decode work is handed out longest-split-first:
    # every row, whatever its place in that order, matches the oracle, and
    # equals the same row computed alone
    g = torch.Generator().manual_seed(77)
    n = 40
    kl = torch.randint(0, 3000, (n,), generator=g).tolist()
    kl[:4] = [0, 1, 2999, 64]
    ql = [1 + (i % 3 == 0) for i in range(n)]
    if entry == "mixed":
        ql[5], kl[5] = 40, 700      # a prefill row among the decode rows
    cpu, gpu = small(ql, kl, hq=8, hkv=2, d=128, P=16, dtype="f16", kv_dtype=kv, seed=31)
    out = run(entry, gpu)
    assert max_err(out, ref_of(cpu)) <= tol_of(cpu)
    cu = cpu.cu_seqlens_q.tolist()
    for r in (2, 17, 39):
        alone = run(entry, workloads.sub_batch(cpu, [r]).to("cuda"))
        assert_bitwise(out[cu[r]:cu[r + 1]], alone)


def _serial_rows(b, rows):
    """Each token i of each listed row as a q = 1 row of its own over the first
    L - q + 1 + i keys of the same pages (what decoding the tokens one at a
    time computes)."""
    cu = b.cu_seqlens_q.cpu().tolist()
    L = b.seq_lens.cpu().tolist()
    bt = b.block_table
    toks, lens, tabs = [], [], []
    for r in rows:
        q = cu[r + 1] - cu[r]
        for i in range(q):
            toks.append(cu[r] + i)
            lens.append(max(0, L[r] - q + 1 + i))
            tabs.append(bt[r])
    dev = b.q.device
    return dict(q=b.q[toks].contiguous(), block_table=torch.stack(tabs).contiguous(),
                cu_seqlens_q=torch.arange(len(toks) + 1, dtype=torch.int32, device=dev),
                seq_lens=torch.tensor(lens, dtype=torch.int32, device=dev)), toks


@pytest.mark.parametrize("dtype,kv", [("bf16", None), ("f16", "e5m2")])
def test_verify_rows_tokenwise_equal_serial_decode(dtype, kv):
    # q > 1 decode rows in one-token mode: every token bitwise equal to a q = 1
    # decode of its own prefix, through the decode and the mixed entries
    ql = [1, 4, 5, 16, 3, 2]
    kl = [300, 700, 129, 2049, 2, 5000]          # row 4: q > L, its first token sees nothing
    cpu, gpu = small(ql, kl, hq=8, hkv=2, d=128, P=16, dtype=dtype, kv_dtype=kv, seed=41,
                     k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0)
    tw = run("decode", gpu, verify_mode=pa.PA_VERIFY_TOKENWISE)
    assert max_err(tw, ref_of(cpu)) <= tol_of(cpu)
    ser, toks = _serial_rows(gpu, range(len(ql)))
    serial = pa.paged_attn_decode(ser["q"], gpu.k_cache, gpu.v_cache, ser["block_table"],
                                  ser["cu_seqlens_q"], ser["seq_lens"],
                                  softmax_scale=gpu.softmax_scale, k_scale=gpu.k_scale,
                                  v_scale=gpu.v_scale)
    torch.cuda.synchronize()
    assert_bitwise(tw[toks], serial)
    # the same rows next to a prefill row in a mixed call
    ql2, kl2 = ql + [100], kl + [900]
    cpu2, gpu2 = small(ql2, kl2, hq=8, hkv=2, d=128, P=16, dtype=dtype, kv_dtype=kv, seed=41,
                       k_scale=0.37 if kv else 1.0, v_scale=1.7 if kv else 1.0)
    mixed = run("mixed", gpu2, verify_mode=pa.PA_VERIFY_TOKENWISE)
    dec_alone = run("decode", workloads.sub_batch(cpu2, range(len(ql))).to("cuda"),
                    verify_mode=pa.PA_VERIFY_TOKENWISE)
    assert_bitwise(mixed[:sum(ql)], dec_alone)
    assert max_err(mixed, ref_of(cpu2)) <= tol_of(cpu2)


@pytest.mark.parametrize("dtype,kv", [("bf16", None), ("f16", "e5m2"), ("f32", None)])
def test_mixed_small_and_routing_bitwise(dtype, kv):
    ql = [300, 1, 4, 0, 17, 16, 2]
    kl = [900, 700, 90, 0, 17, 2000, 2]
    cpu, gpu = small(ql, kl, hq=12, hkv=2, d=128, P=48, dtype=dtype, kv_dtype=kv, seed=9)
    out = run("mixed", gpu)
    assert max_err(out, ref_of(cpu)) <= tol_of(cpu)
    # rows routed to decode equal the decode call's rows; the others the prefill call's
    cu = cpu.cu_seqlens_q.tolist()
    dec_rows = [r for r, q in enumerate(ql) if 1 <= q <= 16]
    pre_rows = [r for r, q in enumerate(ql) if q > 16]
    for rows, entry in ((dec_rows, "decode"), (pre_rows, "prefill")):
        sub_cpu = workloads.sub_batch(cpu, rows)
        sub_out = run(entry, sub_cpu.to("cuda"))
        got = torch.cat([out[cu[r]:cu[r + 1]] for r in rows])
        assert_bitwise(got, sub_out)


def test_mixed_without_host_mirrors_matches():
    ql, kl = [100, 1, 3, 0], [400, 300, 50, 0]
    cpu, gpu = small(ql, kl, seed=11)
    a = run("mixed", gpu, host=True)
    b = run("mixed", gpu, host=False)
    assert_bitwise(a, b)
    cpu2, gpu2 = small([1, 3, 2], [40, 50, 1000], seed=12)
    assert_bitwise(run("decode", gpu2, host=True), run("decode", gpu2, host=False))
    a = run("prefill", gpu, host=True)
    b = run("prefill", gpu, host=False)
    assert_bitwise(a, b)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("entry", ["prefill", "mixed", "decode"])
def test_page_size_and_permutation_invariance_bitwise(entry):
    if entry == "decode":
        ql, kl = [1, 4, 1, 5], [1, 700, 2049, 64]
    else:
        ql, kl = [70, 1, 129, 5], [70, 700, 2049, 64]
    base = run(entry, small(ql, kl, P=16, seed=21)[1])
    for P in (32, 64, 784, 816, 896):
        assert_bitwise(run(entry, small(ql, kl, P=P, seed=21)[1]), base)
    assert_bitwise(run(entry, small(ql, kl, P=16, seed=21, perm_seed=5)[1]), base)


@pytest.mark.parametrize("entry", ["prefill", "mixed", "decode"])
def test_row_alone_equals_row_in_batch(entry):
    if entry == "decode":
        ql, kl = [1, 4, 1, 5, 1], [1, 700, 2049, 64, 9000]
    else:
        ql, kl = [70, 1, 129, 5, 300], [70, 700, 2049, 64, 9000]
    cpu, gpu = small(ql, kl, seed=22)
    full = run(entry, gpu)
    cu = cpu.cu_seqlens_q.tolist()
    for r in range(len(ql)):
        alone = run(entry, workloads.sub_batch(cpu, [r]).to("cuda"))
        assert_bitwise(alone, full[cu[r]:cu[r + 1]])


def test_empty_rows_zero_and_nan_poison_does_not_leak():
    ql, kl = [1, 0, 1, 70, 1, 3], [0, 0, 33, 100, 17, 2]   # rows 0 and 5: tokens with no key
    for entry in ("mixed", "prefill"):
        cpu, gpu = small(ql, kl, seed=23, poison="nan")
        out = run(entry, gpu)
        assert torch.isfinite(out.float()).all()
        assert (out[0] == 0).all()          # row 0 has L = 0
        assert max_err(out, ref_of(cpu)) <= TOL["bf16"]
    cpu, gpu = small([1, 1, 1], [0, 17, 0], seed=24, poison="nan", dtype="f16", kv_dtype="e5m2")
    out = run("decode", gpu)
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert max_err(out, ref_of(cpu)) <= TOL["e5m2"]


def test_repeated_calls_bitwise_and_no_device_errors():
    cpu, gpu = small([100, 1, 4], [1000, 3000, 40], seed=25)
    ws = pa.make_workspace(pa.make_params(gpu.q, gpu.k_cache), 3, gpu.total_q, "cuda")
    a = run("mixed", gpu, workspace=ws)
    b = run("mixed", gpu, workspace=ws)
    assert_bitwise(a, b)
    assert pa.read_errors(ws) == 0


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (256, "bf16"), (256, "f16")])
def test_many_key_tiles_repeated_runs_match_oracle(d, dtype):
    # long rows over many key tiles and several query tiles per row, run
    # repeatedly: every run within tolerance and bitwise equal to the first
    # (guards the ordering of P stores against the P V products in flight,
    # whose violation showed up only intermittently and only on such rows)
    ql, kl = [200, 300, 129], [1000, 3000, 5000]
    cpu, gpu = small(ql, kl, d=d, dtype=dtype, P=16, seed=27)
    ref = ref_of(cpu)
    first = run("prefill", gpu)
    assert max_err(first, ref) <= TOL[dtype]
    for _ in range(5):
        assert_bitwise(run("prefill", gpu), first)


def _ramp_keys(b, growth):
    """Scales key t of every row by (1 + growth * t / L): the logits, and with
    them each row's running maximum, keep growing along the row.  V is
    scaled by 1/4 (exactly): the softmax gets nearly one-hot, so outputs
    approach single V entries, and bf16 rounds values above 4 by up to 2^-6,
    more than the tolerance."""
    b.v_cache.mul_(0.25)
    P = b.k_cache.shape[1]
    for r, L in enumerate(b.kv_lens):
        t = torch.arange(L)
        pages = b.block_table[r, t // P].long()
        f = (1.0 + growth * t.double() / max(L, 1)).to(torch.float32)
        rows = b.k_cache[pages, t % P].float() * f[:, None, None]
        b.k_cache[pages, t % P] = rows.to(b.k_cache.dtype)
    return b


@pytest.mark.parametrize("d,dtype,parts", [(64, "bf16", 0), (128, "bf16", 0), (128, "f16", 2),
                                           (256, "f16", 0), (256, "bf16", 3)])
def test_running_maximum_growing_along_rows_rescales_o(d, dtype, parts):
    # keys scaled up along each row, so every query's running maximum passes
    # its exponent reference by more than 2^8 again and again over the key
    # tiles: the lazy O rescale runs mid-row on the prefill kernels (and its
    # ordering against the P V product in flight), in cut parts, and in the
    # decode rows of the mixed call
    ql, kl = [200, 1, 300, 4], [3000, 4000, 5000, 2500]
    cpu = workloads.make_batch(ql, kl, num_q_heads=8, num_kv_heads=2, head_dim=d, page_size=16,
                               q_dtype=dtype, seed=31)
    cpu = _ramp_keys(cpu, 12.0)
    gpu = cpu.to("cuda")
    ref = ref_of(cpu)
    kw = dict(prefill_kv_parts=parts) if parts else {}
    first = run("mixed", gpu, **kw)
    assert max_err(first, ref) <= TOL[dtype]
    for _ in range(3):
        assert_bitwise(run("mixed", gpu, **kw), first)


def test_device_flags_bad_block_table_entry_without_fault():
    # the host mirrors are withheld so only the kernels can see the bad entry;
    # the kernels must not dereference it and must raise the sticky flag
    cpu, gpu = small([1, 20], [40, 60], seed=26)
    bt = gpu.block_table.clone()
    bt[0, 1] = 10 ** 6           # out of range
    bt[1, 0] = -7                # negative
    ws = pa.make_workspace(pa.make_params(gpu.q, gpu.k_cache), 2, gpu.total_q, "cuda")
    for entry in ("mixed", "prefill"):
        ENTRY[entry](gpu.q, gpu.k_cache, gpu.v_cache, bt, gpu.cu_seqlens_q, gpu.seq_lens,
                     workspace=ws)
        torch.cuda.synchronize()
        assert pa.read_errors(ws) & 0x1
    assert pa.read_errors(ws) == 0   # cleared by the read


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

def test_workload1_decode_only():
    cpu = workloads.make_workload(1)
    gpu = cpu.to("cuda")
    out = run("decode", gpu)
    assert max_err(out, ref_of(cpu)) <= TOL["bf16"]
    assert_bitwise(run("mixed", gpu), out)


def _sample_tokens(cpu_q_lens, every=17, edge=32):
    toks, base = [], 0
    for q in cpu_q_lens:
        idx = set(range(min(edge, q))) | set(range(max(0, q - edge), q)) | set(range(0, q, every))
        toks += [base + i for i in sorted(idx)]
        base += q
    return toks


def test_workload2_varlen_prefill_full_size():
    outs = {}
    for P in (16, 32, 64):
        gpu = workloads.make_workload(2, device="cuda", data_device="cuda", page_size=P)
        outs[P] = run("mixed", gpu)
        if P == 16:
            direct = run("prefill", gpu)
            assert_bitwise(direct, outs[16])
            ql = gpu.q_lens
            toks = _sample_tokens(ql, every=97, edge=8)
            cpu = gpu.to("cpu")
            ref = ref_of(cpu, tokens=toks)
            assert max_err(outs[16][toks], ref) <= TOL["bf16"]
        del gpu
        torch.cuda.empty_cache()
    assert_bitwise(outs[32], outs[16])
    assert_bitwise(outs[64], outs[16])


def test_workload3_mixed_pages_784_816_896():
    outs = {}
    for P in (784, 816, 896):
        gpu = workloads.make_workload(3, device="cuda", data_device="cuda", page_size=P)
        outs[P] = run("mixed", gpu)
        if P == 784:
            # decode rows in full, the chunk's rows sampled
            cpu_rows = workloads.sub_batch(gpu, [1, 2, 3])
            out_rows = outs[P][2048:]
            assert max_err(out_rows, ref_of(cpu_rows)) <= TOL["f16"]
            cpu0 = workloads.sub_batch(gpu, [0])
            toks = [0, 1, 2, 500, 1023, 1500, 2046, 2047]
            assert max_err(outs[P][toks], ref_of(cpu0, tokens=toks)) <= TOL["f16"]
        del gpu
        torch.cuda.empty_cache()
    assert_bitwise(outs[816], outs[784])
    assert_bitwise(outs[896], outs[784])


def test_workload4_split_kv_decode_batch_invariance():
    gpu = workloads.make_workload(4, device="cuda", data_device="cuda")
    out = run("decode", gpu)
    assert_bitwise(run("mixed", gpu), out)
    lens = gpu.kv_lens
    rows = list(range(6)) + list(range(6, 256, 23))
    cpu = workloads.sub_batch(gpu, rows)
    ref = ref_of(cpu)
    assert max_err(out[rows], ref) <= TOL["bf16"]
    # every row alone equals the row in the batch, bitwise
    for r in range(256):
        alone = run("decode", workloads.sub_batch(gpu, [r], device="cuda"))
        assert_bitwise(alone, out[r:r + 1])
    assert all((out[r] == 0).all() for r in range(256) if lens[r] == 0)


@pytest.mark.parametrize("scales", [(0.5, 2.0), (0.37, 1.7)])
def test_workload5_long_context_fp8(scales):
    gpu = workloads.make_workload(5, device="cuda", data_device="cuda", k_scale=scales[0],
                                  v_scale=scales[1])
    out = run("decode", gpu)
    assert_bitwise(run("mixed", gpu), out)
    ql = gpu.q_lens
    cu = np.cumsum([0] + ql)
    rows = [0, 1, 17, 40, 63]
    cpu = workloads.sub_batch(gpu, rows)
    ref = ref_of(cpu)
    got = torch.cat([out[cu[r]:cu[r + 1]] for r in rows])
    assert max_err(got, ref) <= TOL["e5m2"]
