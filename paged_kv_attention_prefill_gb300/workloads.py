"""Seeded synthetic inputs for paged-KV attention.

This module only draws numbers and lays them out: it holds none of the
attention arithmetic, so both the CUDA library's tests and the oracle may use
it.  Recipe (the same for every workload):

* lengths first, from ``torch.Generator().manual_seed(seed)`` on the CPU;
* logical K/V per row ``[L_b, Hkv, d]`` and Q ``[total_q, Hq, d]`` drawn as
  N(0, 1) in fp32 (on ``data_device`` with its own generator seeded by
  ``seed + 1``), then rounded to the storage type (RNE); fp8 E5M2 stores
  ``e5m2(clamp(x / scale, +-57344))``;
* a physical page pool of ``sum_b ceil(L_b / P)`` pages plus about 10 % spare,
  handed out to the rows in a random permutation (``torch.randperm``); unused
  block-table entries are -1;
* the slots of the pool that hold no key of any row (the tail of each row's
  last page, and the spare pages) are poisoned: a large finite value of
  alternating sign (+-3e4 for 16-bit types, +-57344 for fp8, +-1e30 for fp32)
  or NaN for the ``poison="nan"`` variant.

Because the logical data does not depend on the page size or the permutation,
the same seed with another page size or permutation seed gives the same
attention problem laid out differently -- which is what the page-size and
page-permutation invariance checks need.

The five named workloads follow the attention shapes of the pages (a decode
batch with mixed short lengths, a varlen prefill batch, a chunked prefill next
to long resident decode/verify rows with pages of 784/816/896 tokens, a large
split-KV decode batch, and a long-context fp8 decode batch).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32,
                "e5m2": torch.uint8}
POISON_FINITE = {"bf16": 3.0e4, "f16": 3.0e4, "f32": 1.0e30, "e5m2": 57344.0}


@dataclasses.dataclass
class Batch:
    """One paged attention problem.  Tensors live on ``device``."""
    q: torch.Tensor              # [total_q, Hq, d]
    k_cache: torch.Tensor        # [num_pages, P, Hkv, d] (uint8 for e5m2)
    v_cache: torch.Tensor
    block_table: torch.Tensor    # int32 [B, max_pages_per_row]
    cu_seqlens_q: torch.Tensor   # int32 [B + 1]
    seq_lens: torch.Tensor       # int32 [B]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    q_dtype: str
    kv_dtype: str
    k_scale: float = 1.0
    v_scale: float = 1.0
    softmax_scale: float = 0.0
    name: str = ""

    @property
    def num_rows(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def q_lens(self) -> list:
        cu = self.cu_seqlens_q.cpu().tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    @property
    def kv_lens(self) -> list:
        return self.seq_lens.cpu().tolist()

    def to(self, device) -> "Batch":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
             for k, v in dataclasses.asdict(self).items()}
        return Batch(**f)

    def oracle_args(self) -> dict:
        """Host numpy buffers and sizes, in the oracle's keyword form."""
        def raw(t):
            t = t.detach().cpu().contiguous()
            if t.dtype in (torch.bfloat16, torch.float16):
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        return dict(q=raw(self.q), k_cache=raw(self.k_cache), v_cache=raw(self.v_cache),
                    block_table=self.block_table.cpu().numpy(),
                    cu_seqlens_q=self.cu_seqlens_q.cpu().numpy(),
                    seq_lens=self.seq_lens.cpu().numpy(), num_q_heads=self.num_q_heads,
                    num_kv_heads=self.num_kv_heads, head_dim=self.head_dim,
                    page_size=self.page_size, q_dtype=self.q_dtype,
                    kv_dtype=self.kv_dtype, softmax_scale=self.softmax_scale or None,
                    k_scale=self.k_scale, v_scale=self.v_scale)


def _to_storage(x: torch.Tensor, dtype: str, scale: float) -> torch.Tensor:
    if dtype == "e5m2":
        y = (x / scale).clamp(-57344.0, 57344.0).to(torch.float8_e5m2)
        return y.view(torch.uint8)
    return x.to(TORCH_DTYPES[dtype])


def _poison_value(dtype: str, poison: str, n: int, device) -> torch.Tensor:
    """Poison values for n slots' worth of elements, in storage form."""
    if poison == "nan":
        if dtype == "e5m2":
            return torch.full((n,), 0x7F, dtype=torch.uint8, device=device)  # E5M2 NaN
        return torch.full((n,), float("nan"), dtype=TORCH_DTYPES[dtype], device=device)
    v = POISON_FINITE[dtype]
    sign = torch.ones(n, device=device)
    sign[1::2] = -1.0
    x = sign * v
    if dtype == "e5m2":
        return x.to(torch.float8_e5m2).view(torch.uint8)
    return x.to(TORCH_DTYPES[dtype])


def make_batch(q_lens: Sequence[int], kv_lens: Sequence[int], *, num_q_heads: int,
               num_kv_heads: int, head_dim: int, page_size: int, q_dtype: str = "bf16",
               kv_dtype: Optional[str] = None, seed: int = 0, perm_seed: Optional[int] = None,
               device="cpu", data_device=None, k_scale: float = 1.0, v_scale: float = 1.0,
               softmax_scale: float = 0.0, poison: str = "finite", spare_frac: float = 0.1,
               name: str = "") -> Batch:
    """Builds one seeded problem.  ``kv_lens[b]`` is the row's total KV length
    (its new query tokens included); ``q_lens[b] <= kv_lens[b]``."""
    kv_dtype = kv_dtype or q_dtype
    B = len(kv_lens)
    assert len(q_lens) == B
    P = int(page_size)
    data_device = torch.device(data_device if data_device is not None else device)
    gen_data = torch.Generator(device=data_device).manual_seed(seed + 1)
    gen_perm = torch.Generator().manual_seed(seed + 2 if perm_seed is None else perm_seed)

    pages_per_row = [(int(L) + P - 1) // P for L in kv_lens]
    used = sum(pages_per_row)
    num_pages = used + int(math.ceil(spare_frac * used)) + 1
    perm = torch.randperm(num_pages, generator=gen_perm).to(torch.int32)
    maxp = max(1, max(pages_per_row) if B else 1)
    bt = torch.full((B, maxp), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_row):
        bt[b, :n] = perm[off:off + n]
        off += n

    Hkv, d = num_kv_heads, head_dim
    sd = TORCH_DTYPES[kv_dtype]
    k_cache = torch.empty((num_pages, P, Hkv, d), dtype=sd, device=data_device)
    v_cache = torch.empty_like(k_cache)
    # poison everything first; the rows' keys overwrite their own slots below
    slot_elems = Hkv * d
    for cache in (k_cache, v_cache):
        flat = cache.view(num_pages * P, slot_elems)
        pv = _poison_value(kv_dtype, poison, num_pages * P, data_device)
        flat.copy_(pv.view(-1, 1).expand(-1, slot_elems))

    bt_dev = bt.to(data_device)
    for b in range(B):
        L = int(kv_lens[b])
        if L == 0:
            continue
        for cache, sc in ((k_cache, k_scale), (v_cache, v_scale)):
            x = torch.randn((L, Hkv, d), generator=gen_data, device=data_device,
                            dtype=torch.float32)
            xs = _to_storage(x, kv_dtype, sc)
            del x
            j = torch.arange(L, device=data_device)
            phys = bt_dev[b, (j // P).long()].long() * P + (j % P)
            cache.view(num_pages * P, Hkv, d).index_copy_(0, phys, xs)
            del xs

    total_q = int(sum(int(x) for x in q_lens))
    qx = torch.randn((total_q, num_q_heads, d), generator=gen_data, device=data_device,
                     dtype=torch.float32)
    q = qx.to(TORCH_DTYPES[q_dtype])
    del qx
    cu = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        cu[1:] = torch.cumsum(torch.tensor([int(x) for x in q_lens], dtype=torch.int64), 0).to(torch.int32)
    lens = torch.tensor([int(x) for x in kv_lens], dtype=torch.int32)
    dev = torch.device(device)
    return Batch(q=q.to(dev), k_cache=k_cache.to(dev), v_cache=v_cache.to(dev),
                 block_table=bt.to(dev), cu_seqlens_q=cu.to(dev), seq_lens=lens.to(dev),
                 num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                 page_size=P, q_dtype=q_dtype, kv_dtype=kv_dtype, k_scale=k_scale,
                 v_scale=v_scale, softmax_scale=softmax_scale, name=name)


# --------------------------------------------------------------------------
# The five named workloads.
# --------------------------------------------------------------------------

WORKLOADS = {
    1: "decode-only: 4 rows q=1, L={1,31,33,513}, 8/2 heads, d=128, page 16, bf16",
    2: "varlen causal prefill: 8 rows q~U[65,2048], ctx~U[0,16384], 32/8 heads, d=128, "
       "pages 16/32/64, bf16",
    3: "mixed: 2048-token chunk after 150000 cached + 3 rows at 240000 with q=1/4/5, "
       "24/4 heads, d=256, fp16, pages 784/816/896",
    4: "split-KV decode: 256 rows q=1, L~U[0,32768] incl. 0/1/31/32/33/4097, 32/8 heads, "
       "d=128, page 16, bf16",
    5: "long-context decode: 64 rows q=1|4, L~U[128000,240000], 16/4 heads, d=256, fp16 Q, "
       "fp8_e5m2 KV (k_scale 0.5, v_scale 2.0), page 16",
}


def workload_lengths(n: int, seed: Optional[int] = None):
    """(q_lens, kv_lens) of workload n, drawn from its seed (20260 + n)."""
    g = torch.Generator().manual_seed(20260 + n if seed is None else seed)
    if n == 1:
        return [1, 1, 1, 1], [1, 31, 33, 513]
    if n == 2:
        q = torch.randint(65, 2049, (8,), generator=g).tolist()
        ctx = torch.randint(0, 16385, (8,), generator=g).tolist()
        return q, [a + b for a, b in zip(q, ctx)]
    if n == 3:
        return [2048, 1, 4, 5], [150000 + 2048, 240000, 240000, 240000]
    if n == 4:
        L = torch.randint(0, 32769, (256,), generator=g).tolist()
        L[:6] = [0, 1, 31, 32, 33, 4097]
        return [1] * 256, L
    if n == 5:
        q = (torch.rand(64, generator=g) < 0.5).long().mul(3).add(1).tolist()
        L = torch.randint(128000, 240001, (64,), generator=g).tolist()
        return q, L
    raise ValueError(n)


def workload_shape(n: int) -> dict:
    return {
        1: dict(num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, q_dtype="bf16"),
        2: dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, q_dtype="bf16"),
        3: dict(num_q_heads=24, num_kv_heads=4, head_dim=256, page_size=784, q_dtype="f16"),
        4: dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, q_dtype="bf16"),
        5: dict(num_q_heads=16, num_kv_heads=4, head_dim=256, page_size=16, q_dtype="f16",
                kv_dtype="e5m2", k_scale=0.5, v_scale=2.0),
    }[n]


def make_workload(n: int, *, device="cpu", data_device=None, page_size: Optional[int] = None,
                  perm_seed: Optional[int] = None, poison: str = "finite",
                  rows: Optional[Sequence[int]] = None, **over) -> Batch:
    """Workload n.  ``rows`` keeps only the listed rows' lengths (the same
    shapes and distributions; the data drawn for them differs from the whole
    workload's), so a small case of the same kernels never holds the rest."""
    q_lens, kv_lens = workload_lengths(n)
    if rows is not None:
        q_lens = [q_lens[int(r)] for r in rows]
        kv_lens = [kv_lens[int(r)] for r in rows]
    shape = workload_shape(n)
    if page_size is not None:
        shape["page_size"] = page_size
    shape.update(over)
    return make_batch(q_lens, kv_lens, seed=20260 + n, perm_seed=perm_seed, device=device,
                      data_device=data_device, poison=poison, name=f"workload{n}", **shape)


def sub_batch(batch: Batch, rows: Sequence[int], device="cpu") -> Batch:
    """The listed rows of a batch as a compact problem of their own (same page
    size, pages renumbered densely in row order).  The attention result of
    each kept row does not depend on where its pages sit, so this lets the
    oracle check a few rows of a batch too large to copy whole."""
    rows = [int(r) for r in rows]
    P = batch.page_size
    cu = batch.cu_seqlens_q.cpu()
    lens = batch.seq_lens.cpu()
    bt = batch.block_table.cpu()
    q_parts, k_pages, v_pages, new_lens, new_q = [], [], [], [], []
    for r in rows:
        L = int(lens[r])
        n = (L + P - 1) // P
        phys = bt[r, :n].long().to(batch.k_cache.device)
        k_pages.append(batch.k_cache.index_select(0, phys).to(device))
        v_pages.append(batch.v_cache.index_select(0, phys).to(device))
        q_parts.append(batch.q[int(cu[r]):int(cu[r + 1])].to(device))
        new_lens.append(L)
        new_q.append(int(cu[r + 1] - cu[r]))
    maxp = max([1] + [(L + P - 1) // P for L in new_lens])
    nbt = torch.full((len(rows), maxp), -1, dtype=torch.int32)
    off = 0
    for i, L in enumerate(new_lens):
        n = (L + P - 1) // P
        nbt[i, :n] = torch.arange(off, off + n, dtype=torch.int32)
        off += n
    empty = batch.k_cache[:0].to(device)
    kc = torch.cat(k_pages) if k_pages else empty
    vc = torch.cat(v_pages) if v_pages else empty
    if kc.shape[0] == 0:
        kc = torch.zeros((1,) + tuple(batch.k_cache.shape[1:]), dtype=batch.k_cache.dtype,
                         device=device)
        vc = kc.clone()
    ncu = torch.zeros(len(rows) + 1, dtype=torch.int32)
    ncu[1:] = torch.cumsum(torch.tensor(new_q, dtype=torch.int64), 0).to(torch.int32)
    return Batch(q=torch.cat(q_parts) if q_parts else batch.q[:0].to(device), k_cache=kc,
                 v_cache=vc, block_table=nbt.to(device), cu_seqlens_q=ncu.to(device),
                 seq_lens=torch.tensor(new_lens, dtype=torch.int32, device=device),
                 num_q_heads=batch.num_q_heads, num_kv_heads=batch.num_kv_heads,
                 head_dim=batch.head_dim, page_size=P, q_dtype=batch.q_dtype,
                 kv_dtype=batch.kv_dtype, k_scale=batch.k_scale, v_scale=batch.v_scale,
                 softmax_scale=batch.softmax_scale, name=batch.name + "[rows]")
