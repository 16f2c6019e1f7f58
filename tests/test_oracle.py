"""Pins for the fp64 oracle, on the CPU.

The oracle is checked against things other than itself:

* the number formats' definitions (golden code points) and library decoders
  (numpy float16, torch bfloat16 / float8_e5m2) over every code;
* an independent dense brute force written here with numpy: K/V copied out of
  the block table into dense arrays, an explicit mask matrix, a softmax over
  each masked row -- on tiny problems, exhaustively over q <= L;
* closed forms (one key, all-equal logits, a dominant key, two keys by hand);
* the invariants the pages state (page size, physical-page permutation, empty
  rows, a row alone vs in a batch, a q-token row vs q single-token rows);
* the pages' own figures where they pin a formula we use (FLOP convention,
  decode workspace size);
* mutation checks: plausible mistakes planted into a copy of the oracle's C
  source must each fail at least one of the pins above.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_prefill_gb300 import metrics, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# independent helpers (no oracle code)
# --------------------------------------------------------------------------

def to_f64(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Library decode of storage to float64 (independent of the oracle's C)."""
    t = t.detach().cpu()
    if dtype == "e5m2":
        return t.view(torch.float8_e5m2).to(torch.float32).double().numpy()
    if dtype == "f16":
        return t.numpy().astype(np.float64)
    if dtype == "bf16":
        return t.to(torch.float32).double().numpy()
    return t.double().numpy()


def brute_force(batch: workloads.Batch) -> np.ndarray:
    """Dense softmax attention with an explicit mask matrix."""
    P = batch.page_size
    g = batch.num_q_heads // batch.num_kv_heads
    s = batch.softmax_scale or 1.0 / math.sqrt(batch.head_dim)
    q = to_f64(batch.q, batch.q_dtype)
    kc = to_f64(batch.k_cache, batch.kv_dtype) * batch.k_scale
    vc = to_f64(batch.v_cache, batch.kv_dtype) * batch.v_scale
    bt = batch.block_table.numpy()
    cu = batch.cu_seqlens_q.numpy()
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(batch.num_rows):
        qb, L = int(cu[b + 1] - cu[b]), int(batch.seq_lens[b])
        if qb == 0:
            continue
        # dense K/V of the row: [L, Hkv, d]
        K = np.stack([kc[bt[b, j // P], j % P] for j in range(L)]) if L else None
        V = np.stack([vc[bt[b, j // P], j % P] for j in range(L)]) if L else None
        mask = np.zeros((qb, L), dtype=bool)
        for i in range(qb):
            mask[i, : max(0, L - qb + i + 1)] = True
        for h in range(batch.num_q_heads):
            if L == 0:
                continue
            Q = q[cu[b]:cu[b + 1], h]                       # [qb, d]
            S = s * Q @ K[:, h // g].T                       # [qb, L]
            S = np.where(mask, S, -np.inf)
            for i in range(qb):
                if not mask[i].any():
                    continue
                w = np.exp(S[i] - S[i].max())
                out[cu[b] + i, h] = (w[:, None] * V[:, h // g]).sum(0) / w.sum()
    return out


def run_oracle(batch, lib=None, **kw):
    args = batch.oracle_args()
    args.update(kw)
    return oracle.paged_attention(lib=lib, **args)


def tiny(q_lens, kv_lens, *, hq=4, hkv=2, d=8, P=16, dtype="bf16", kv_dtype=None, seed=0,
         **kw):
    return workloads.make_batch(q_lens, kv_lens, num_q_heads=hq, num_kv_heads=hkv,
                                head_dim=d, page_size=P, q_dtype=dtype, kv_dtype=kv_dtype,
                                seed=seed, **kw)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def _golden_e5m2():
    rows = []
    with open(os.path.join(GOLDEN, "e5m2_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


def check_formats(lib=None):
    for code, val in _golden_e5m2():
        got = oracle.decode(np.array([code], np.uint8), "e5m2", lib=lib)[0]
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)
    codes8 = np.arange(256, dtype=np.uint8)
    ref8 = torch.from_numpy(codes8).view(torch.float8_e5m2).to(torch.float32).double().numpy()
    got8 = oracle.decode(codes8, "e5m2", lib=lib)
    np.testing.assert_array_equal(np.isnan(got8), np.isnan(ref8))
    ok = ~np.isnan(ref8)
    np.testing.assert_array_equal(got8[ok], ref8[ok])
    codes16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref16 = codes16.view(np.float16).astype(np.float64)
    got16 = oracle.decode(codes16, "f16", lib=lib)
    np.testing.assert_array_equal(np.isnan(got16), np.isnan(ref16))
    ok = ~np.isnan(ref16)
    np.testing.assert_array_equal(got16[ok], ref16[ok])
    refb = torch.from_numpy(codes16.view(np.int16)).view(torch.bfloat16).float().double().numpy()
    gotb = oracle.decode(codes16, "bf16", lib=lib)
    np.testing.assert_array_equal(np.isnan(gotb), np.isnan(refb))
    ok = ~np.isnan(refb)
    np.testing.assert_array_equal(gotb[ok], refb[ok])
    f = np.array([1.5, -0.0, 3.4028235e38, 1e-45], dtype=np.float32)
    np.testing.assert_array_equal(oracle.decode(f, "f32", lib=lib), f.astype(np.float64))


def test_formats():
    check_formats()


# --------------------------------------------------------------------------
# brute force on tiny inputs
# --------------------------------------------------------------------------

BRUTE_CASES = [
    # (q_lens, kv_lens, hq, hkv, d, P, dtype, kv_dtype, k_scale, v_scale)
    ([1, 3, 2], [1, 17, 40], 4, 2, 8, 16, "bf16", None, 1.0, 1.0),
    ([5, 1], [33, 16], 2, 2, 4, 32, "f16", None, 1.0, 1.0),
    ([4, 7], [4, 39], 6, 2, 8, 16, "f32", None, 1.0, 1.0),
    ([3, 2, 1], [20, 2, 31], 4, 1, 8, 16, "f16", "e5m2", 0.5, 2.0),
    ([2], [35], 4, 2, 4, 32, "bf16", "e5m2", 0.37, 1.7),
]


def check_brute_force(lib=None):
    for n, (ql, kl, hq, hkv, d, P, dt, kvt, ks, vs) in enumerate(BRUTE_CASES):
        b = tiny(ql, kl, hq=hq, hkv=hkv, d=d, P=P, dtype=dt, kv_dtype=kvt, seed=100 + n,
                 k_scale=ks, v_scale=vs)
        np.testing.assert_allclose(run_oracle(b, lib), brute_force(b), rtol=0, atol=1e-12)
    # exhaustive over q <= L for one row length, two page sizes
    for P in (16, 32):
        L = 37
        for q in range(0, L + 1):
            b = tiny([q], [L], hq=2, hkv=1, d=4, P=P, dtype="f32", seed=7)
            np.testing.assert_allclose(run_oracle(b, lib), brute_force(b), rtol=0, atol=1e-12)


def test_brute_force():
    check_brute_force()


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def check_closed_forms(lib=None):
    # one key: the output is that key's value, exactly
    b = tiny([1], [1], hq=2, hkv=1, d=8, dtype="f32", seed=3)
    out = run_oracle(b, lib)
    v0 = b.v_cache[b.block_table[0, 0], 0, 0].double().numpy()
    np.testing.assert_array_equal(out[0, 0], v0)
    np.testing.assert_array_equal(out[0, 1], v0)

    # zero queries: every visible key has logit 0 -> mean of the visible values
    b = tiny([3], [10], hq=2, hkv=2, d=4, dtype="f32", seed=4)
    b.q.zero_()
    out = run_oracle(b, lib)
    V = np.stack([b.v_cache[b.block_table[0, j // 16], j % 16].double().numpy()
                  for j in range(10)])
    for i in range(3):
        np.testing.assert_allclose(out[i], V[: 10 - 3 + i + 1].mean(0), rtol=0, atol=1e-14)

    # a dominant key: k_j = lambda * q for one j, lambda large -> out -> v_j
    b = tiny([1], [5], hq=1, hkv=1, d=4, dtype="f32", seed=5)
    qv = torch.tensor([1.0, -2.0, 0.5, 3.0])
    b.q[0, 0] = qv
    P0 = int(b.block_table[0, 0])
    b.k_cache[P0, :5, 0] = 0.0
    b.k_cache[P0, 2, 0] = 50.0 * qv
    out = run_oracle(b, lib)
    np.testing.assert_allclose(out[0, 0], b.v_cache[P0, 2, 0].double().numpy(), atol=1e-12)

    # two keys by hand: logits x0, x1 -> (e^x0 v0 + e^x1 v1) / (e^x0 + e^x1)
    b = tiny([1], [2], hq=1, hkv=1, d=2, dtype="f32", seed=6, softmax_scale=0.5)
    b.q[0, 0] = torch.tensor([1.0, 2.0])
    P0 = int(b.block_table[0, 0])
    b.k_cache[P0, 0, 0] = torch.tensor([3.0, -1.0])    # q.k = 1   -> x0 = 0.5
    b.k_cache[P0, 1, 0] = torch.tensor([0.0, 1.5])     # q.k = 3   -> x1 = 1.5
    b.v_cache[P0, 0, 0] = torch.tensor([2.0, 0.0])
    b.v_cache[P0, 1, 0] = torch.tensor([0.0, 4.0])
    w0, w1 = math.exp(0.5), math.exp(1.5)
    want = np.array([2.0 * w0, 4.0 * w1]) / (w0 + w1)
    np.testing.assert_allclose(run_oracle(b, lib)[0, 0], want, rtol=1e-15, atol=0)

    # GQA: g = 2 equals g = 1 with each KV head replicated for its query heads
    b = tiny([3, 1], [9, 20], hq=4, hkv=2, d=4, dtype="f32", seed=8)
    rep = workloads.Batch(**{**b.__dict__})
    rep.k_cache = b.k_cache.repeat_interleave(2, dim=2)
    rep.v_cache = b.v_cache.repeat_interleave(2, dim=2)
    rep.num_kv_heads = 4
    np.testing.assert_array_equal(run_oracle(b, lib), run_oracle(rep, lib))


def test_closed_forms():
    check_closed_forms()


# --------------------------------------------------------------------------
# invariants the pages state
# --------------------------------------------------------------------------

def check_invariants(lib=None):
    ql, kl = [3, 1, 0, 4], [50, 1, 0, 70]
    ref = run_oracle(tiny(ql, kl, P=16, seed=11), lib)
    # page size (1Cat-vLLM PR #616: any multiple of 16, bit-identical)
    for P in (32, 48, 64, 784):
        np.testing.assert_array_equal(run_oracle(tiny(ql, kl, P=P, seed=11), lib), ref)
    # physical-page permutation (vllm-rlt PR #128 test plan: out-of-order pages)
    np.testing.assert_array_equal(run_oracle(tiny(ql, kl, P=16, seed=11, perm_seed=99), lib), ref)
    # empty row (L = 0, q = 0) and its neighbours; zero output for empty rows
    b = tiny([1, 0, 1], [5, 0, 0], seed=12)
    out = run_oracle(b, lib)
    assert np.all(out[1] == 0.0)           # the q=1, L=0 row (token index 1)
    # more new tokens than keys: the leading tokens see no key -> zero output
    b = tiny([3], [1], hq=2, hkv=1, d=4, dtype="f32", seed=15)
    out = run_oracle(b, lib)
    assert np.all(out[:2] == 0.0)
    np.testing.assert_array_equal(out[2, 0], b.v_cache[b.block_table[0, 0], 0, 0].double().numpy())
    # a row alone equals the same row in a batch, bitwise
    full = run_oracle(tiny(ql, kl, seed=11), lib)
    cu = np.cumsum([0] + ql)
    for r in range(len(ql)):
        alone = workloads.sub_batch(tiny(ql, kl, seed=11), [r])
        np.testing.assert_array_equal(run_oracle(alone, lib), full[cu[r]:cu[r + 1]])
    # a q-token row equals q single-token rows of lengths L - q + 1 + i
    b = tiny([5], [30], seed=13)
    out = run_oracle(b, lib)
    bt = b.block_table.repeat(5, 1)
    exp = workloads.Batch(**{**b.__dict__})
    exp.block_table = bt
    exp.cu_seqlens_q = torch.arange(6, dtype=torch.int32)
    exp.seq_lens = torch.tensor([30 - 5 + 1 + i for i in range(5)], dtype=torch.int32)
    np.testing.assert_array_equal(run_oracle(exp, lib), out)
    # scales: k_scale c is the same as softmax_scale c; v_scale is linear
    b1 = tiny([2], [20], dtype="f16", kv_dtype="e5m2", seed=14, k_scale=0.25)
    b2 = tiny([2], [20], dtype="f16", kv_dtype="e5m2", seed=14, k_scale=0.25)
    b2.k_scale = 1.0
    b2.softmax_scale = 0.25 / math.sqrt(b2.head_dim)
    np.testing.assert_allclose(run_oracle(b1, lib), run_oracle(b2, lib), rtol=1e-13, atol=1e-15)
    b3 = tiny([2], [20], dtype="f16", kv_dtype="e5m2", seed=14, k_scale=0.25)
    b3.v_scale = 4.0
    np.testing.assert_allclose(run_oracle(b3, lib), 4.0 * run_oracle(b1, lib), rtol=1e-14,
                               atol=1e-15)


def test_invariants():
    check_invariants()


def test_sampled_tokens_match_full():
    b = tiny([6, 2, 9], [30, 2, 60], hq=4, hkv=1, seed=21)
    full = run_oracle(b)
    toks = [16, 0, 5, 8, 7]
    np.testing.assert_array_equal(run_oracle(b, tokens=toks), full[toks])


def test_rejects_malformed():
    b = tiny([2], [20], seed=22)
    args = b.oracle_args()
    args["seq_lens"] = np.array([10 ** 6], np.int32)
    with pytest.raises(ValueError):
        oracle.paged_attention(**args)


# --------------------------------------------------------------------------
# the pages' figures that pin our formulas
# --------------------------------------------------------------------------

def test_flop_convention_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "flop_convention.json")))
    F = metrics.prefill_flops([g["q_len"]], [g["cached"] + g["q_len"]], g["num_q_heads"],
                              g["head_dim"])
    for c in g["cases"]:
        tf = F / (c["ms"] * 1e-3) / 1e12
        assert abs(tf - c["tflops_printed"]) <= c["tol"], (tf, c)
    # and the formula itself against brute counting on a small case
    ql, kl = [3, 5, 0, 2], [3, 9, 4, 1]
    pairs = sum(max(0, L - q + i + 1) for q, L in zip(ql, kl) for i in range(q))
    assert metrics.visible_pairs(ql, kl) == pairs


def test_decode_workspace_figure():
    g = json.load(open(os.path.join(GOLDEN, "decode_workspace.json")))
    per_row = g["num_q_heads"] * g["num_splits"] * (g["head_dim"] + 2) * 4
    assert per_row == g["bytes_per_row"]
    assert round(per_row / 1024) == g["kib_per_row_printed"]


# --------------------------------------------------------------------------
# mutation checks: each planted mistake must fail a pin
# --------------------------------------------------------------------------

MUTANTS = {
    "causal_off_by_one": ("const int64_t last = L - qb + i;", "const int64_t last = L - qb + i - 1;"),
    "gqa_mapping": ("const int kh = h / g;", "const int kh = h % p->num_kv_heads;"),
    "page_index": ("j / P]", "j / 16]"),
    "slot_index": ("(page * P + j % P)", "(page * P + j % 16)"),
    "dropped_k_scale": ("* p->k_scale)", ")"),
    "dropped_v_scale": ("* p->v_scale)", ")"),
    "dropped_softmax_scale": ("p->softmax_scale * acc", "acc"),
    "e5m2_bias": ("ldexp(4.0 + (double)f, e - 17)", "ldexp(4.0 + (double)f, e - 16)"),
    "f16_subnormal": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "empty_row_nonzero": ("if (L <= 0 || last < 0) return;", "if (L <= 0) return;"),
}

PINS = [check_formats, check_brute_force, check_closed_forms, check_invariants]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    a, b = MUTANTS[name]
    assert a in src, f"mutation anchor for {name} not found"
    mutated = tmp_path / f"mut_{name}.c"
    mutated.write_text(src.replace(a, b))
    lib = oracle.compile_source(str(mutated), str(tmp_path / f"libmut_{name}.so"))
    caught = False
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught = True
            break
    assert caught, f"planted mistake {name} passed every pin"
