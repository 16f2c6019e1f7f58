"""Algorithmic work of a paged attention call, for throughput figures.

FLOPs (prefill): 4 * d * Hq per visible (query, key) pair -- one multiply-add
for the logit and one for the value product, per element of d -- summed over
the pairs the bottom-right causal mask leaves visible; masked pairs are not
counted.  This is the convention that reproduces the Turing prefill page's
printed throughput (1Cat-vLLM PR #1279, "Kernel microbenchmarks": a
2048-token chunk after 150k context, 12 query heads, head dim 256, 165.8 ms
"about 23 TFLOPS" and 61.5 ms "61 TFLOPS").

Bytes (decode): every K and V element of a row's KV length read once (each
row's keys are shared by all of its query tokens and heads of a group), plus
the queries read, the output written and the block-table entries read.
Partial-state traffic of the split-KV path is overhead and not counted.
"""
from __future__ import annotations

from typing import Sequence

ELT_BYTES = {"bf16": 2, "f16": 2, "f32": 4, "e5m2": 1}


def visible_pairs(q_lens: Sequence[int], kv_lens: Sequence[int]) -> int:
    """sum_b sum_{i<q_b} (L_b - q_b + i + 1), clipped at zero."""
    tot = 0
    for q, L in zip(q_lens, kv_lens):
        q, L = int(q), int(L)
        if q <= 0 or L <= 0:
            continue
        first = L - q + 1            # keys visible to query 0
        lo = max(first, 1)
        hi = L                       # keys visible to the last query
        if hi < lo:
            continue
        n = hi - lo + 1              # queries with at least one visible key
        tot += (lo + hi) * n // 2
    return tot


def prefill_flops(q_lens, kv_lens, num_q_heads: int, head_dim: int) -> int:
    return 4 * head_dim * num_q_heads * visible_pairs(q_lens, kv_lens)


def decode_bytes(q_lens, kv_lens, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 q_dtype: str, kv_dtype: str, page_size: int) -> int:
    kv = sum(int(L) for L in kv_lens) * num_kv_heads * head_dim * 2 * ELT_BYTES[kv_dtype]
    tq = sum(int(q) for q in q_lens)
    qo = 2 * tq * num_q_heads * head_dim * ELT_BYTES[q_dtype]
    bt = sum((int(L) + page_size - 1) // page_size for L in kv_lens) * 4
    return kv + qo + bt
