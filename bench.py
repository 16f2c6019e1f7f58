#!/usr/bin/env python
"""Benchmark of the paged attention hot path on GB300.

One step = one paged_attn_mixed call (row routing, then the prefill kernel;
rows short enough for the decode path would also run split-KV decode + merge)
over the varlen causal prefill workload: 8 rows, new query lengths uniform in
[65, 2048], prior cached context uniform in [0, 16384], 32 query / 8 KV heads,
head dim 128, pages of 16 tokens, bf16, shuffled block table (seed 20262).
The headline value is prefill TFLOP/s by the visible-pair FLOP convention.
The decode half of the metric (KV GB/s) is measured on the split-KV decode
batch (256 rows, L up to 32768) and the long-context fp8 decode batch, and
reported under "parts" with the mixed batch and the small decode batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own copy of the workload on its own GPU
(rows are independent: weak scaling, no data-path collective).  The
reference arm (--impl reference) times the fp64 CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import datetime as _dt
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_attention_prefill_gb300 import dist as padist  # noqa: E402
from paged_kv_attention_prefill_gb300 import metrics, workloads  # noqa: E402

METRIC = "prefill TFLOPS & decode KV GB/s (fraction of GB300 roofline), 1 GPU"
HEADLINE_WORKLOAD = 2
L2_BYTES = 129 * 1024 * 1024


# DRAM bytes (read + write) per launch of the prefill kernel on this workload,
# from one ncu capture of the headline step (dram__bytes_read.sum +
# dram__bytes_write.sum of one prefill_tc2_kernel launch, page 16).  Reported
# only while the kernel's sources hash to the ones that were profiled.
PROFILED_PREFILL_TRAFFIC = {
    "sources": {
        "paged_kv_attention_prefill_gb300/csrc/pa_prefill_tc2.cu": "a5b45c33948c01dfe93911f7a6286ed1a0308b74000aad8c1c5e87f4881de834",
        "paged_kv_attention_prefill_gb300/csrc/pa_sm100.cuh": "7d06c7946e0693914ca226a6d0f71e3825078c65055e4edd196bfeb33a533b84",
        "paged_kv_attention_prefill_gb300/csrc/pa_internal.cuh": "a83b5cf1cddace0bea41b9a50005ac4c9176cdee12d0c0315dbf0d09448b1988",
    },
    "bytes_per_launch": 1185263872 + 53544960,
}


def profiled_traffic():
    import hashlib
    for rel, digest in PROFILED_PREFILL_TRAFFIC["sources"].items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        except OSError:
            return None
    return PROFILED_PREFILL_TRAFFIC["bytes_per_launch"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.sel = str(device_index)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.6)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) < 9:
                    continue
                try:
                    ts = _dt.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                rows.append((ts, [x.strip() for x in r[1:]]))
        os.unlink(self.path)
        inside = [x for t, x in rows if self.t0 is not None and self.t0 <= t <= self.t1 + 0.05]
        note = "inside timed region"
        if not inside:
            inside = [x for _, x in rows]
            note = "timed region shorter than the sampling interval: all samples of the run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(x[0]) for x in inside if x[0].replace(".", "").isdigit()]
        mx = [float(x[1]) for x in inside if x[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for x in inside for i in range(4) if x[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def launches_per_call(q_lens, max_dq=16, mixed=True):
    """Kernels one call launches: the plan (mixed and prefill calls), then for
    decode rows the work-order sort (16 or more rows in the call), the decode
    kernel and the merge, then the prefill kernel."""
    n_rows = len(q_lens)
    dec = any(1 <= q <= max_dq for q in q_lens) if mixed else n_rows > 0
    pre = mixed and any(q > max_dq for q in q_lens)
    n = 1 if mixed else 0
    if dec:
        n += 2 + (1 if n_rows >= 16 else 0)
    return n + (1 if pre else 0)


def headline_config(b, world):
    """The headline workload's description, the same for both arms."""
    names = ("q", "k_cache", "v_cache", "block_table", "cu_seqlens_q", "seq_lens")
    in_bytes = sum(getattr(b, k).numel() * getattr(b, k).element_size() for k in names)
    return {"workload": workloads.WORKLOADS[HEADLINE_WORKLOAD], "rows": b.num_rows,
            "q_lens": b.q_lens, "kv_lens": b.kv_lens, "page_size": b.page_size,
            "flops_per_step": metrics.prefill_flops(b.q_lens, b.kv_lens, b.num_q_heads,
                                                    b.head_dim),
            "l2": f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB > 129 MiB), no flush",
            "parallelism": f"replicas x{world} (rows independent)"}


def call_args(b):
    return dict(cu_seqlens_q_host=b.cu_seqlens_q.cpu(), seq_lens_host=b.seq_lens.cpu(),
                softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale)


def time_calls(fn, steps, warmup, stream, sampler=None):
    """Times exactly `steps` calls with CUDA events on the launching stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    padist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark("t0")
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    padist.barrier()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def graph_ms(fn, steps, warmup, stream):
    """Times `steps` replays of a CUDA graph holding one call of fn (the call
    runs once outside the capture first, for its one-time set-up)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    ms = time_calls(g.replay, steps, warmup, stream)
    del g
    return ms


def part_decode(n, steps, warmup, stream, pk, by_length=False):
    import paged_kv_attention_prefill_gb300 as pa
    b = workloads.make_workload(n, device="cuda", data_device="cuda")
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache, num_splits=pa.PA_SPLITS_BY_LENGTH),
                           b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    kw = call_args(b)

    def call(ns):
        def fn():
            pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                                 b.seq_lens, out=out, workspace=ws, num_splits=ns, **kw)
        return fn
    fn = call(0)
    ms = time_calls(fn, steps, warmup, stream)
    ms_graph = graph_ms(fn, steps, warmup, stream)
    byt = metrics.decode_bytes(b.q_lens, b.kv_lens, num_q_heads=b.num_q_heads,
                               num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                               q_dtype=b.q_dtype, kv_dtype=b.kv_dtype, page_size=b.page_size)
    gbs = byt / (ms * 1e-3) / 1e9
    res = {"workload": workloads.WORKLOADS[n], "ms": round(ms, 4), "kv_bytes": byt,
           "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm"], 4),
           "graph_replay_GB/s": round(byt / (ms_graph * 1e-3) / 1e9, 1),
           "launches_per_call": launches_per_call(b.q_lens, mixed=False)}
    if by_length:
        # the same batch with the length-only split count (2048-key parts)
        ms_bl = time_calls(call(pa.PA_SPLITS_BY_LENGTH), steps, warmup, stream)
        gbs_bl = byt / (ms_bl * 1e-3) / 1e9
        res["by_length_splits"] = {"ms": round(ms_bl, 4), "GB/s": round(gbs_bl, 1),
                                   "frac_of_hbm": round(gbs_bl / pk["hbm"], 4)}
    del b, ws, out
    torch.cuda.empty_cache()
    return res


def part_mixed3(steps, warmup, stream, pk):
    import paged_kv_attention_prefill_gb300 as pa
    b = workloads.make_workload(3, device="cuda", data_device="cuda")
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    kw = call_args(b)

    def fn():
        pa.paged_attn_mixed(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, out=out, workspace=ws, **kw)
    ms = time_calls(fn, steps, warmup, stream)
    ql, kl = b.q_lens, b.kv_lens
    F = metrics.prefill_flops(ql[:1], kl[:1], b.num_q_heads, b.head_dim)
    byt = metrics.decode_bytes(ql[1:], kl[1:], num_q_heads=b.num_q_heads,
                               num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                               q_dtype=b.q_dtype, kv_dtype=b.kv_dtype, page_size=b.page_size)
    res = {"workload": workloads.WORKLOADS[3], "ms": round(ms, 4), "prefill_flops": F,
           "decode_bytes": byt, "whole_call_TFLOP/s_of_prefill": round(F / (ms * 1e-3) / 1e12, 1),
           "launches_per_call": launches_per_call(ql)}
    lws = pa.make_workspace(pa.make_params(b.q, b.k_cache, num_splits=pa.PA_SPLITS_BY_LENGTH),
                            b.num_rows, b.total_q, "cuda")

    def lfn():
        pa.paged_attn_mixed(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, out=out, workspace=lws,
                            num_splits=pa.PA_SPLITS_BY_LENGTH, **kw)
    lms = time_calls(lfn, steps, warmup, stream)
    res["whole_call_by_length"] = {"ms": round(lms, 4),
                                   "TFLOP/s_of_prefill": round(F / (lms * 1e-3) / 1e12, 1)}
    del lws
    # and with the prefill row cut into key-range parts, the count chosen per
    # call (the chunk's row is cut in 3)
    aws = pa.make_workspace(pa.make_params(b.q, b.k_cache, num_splits=pa.PA_SPLITS_BY_LENGTH,
                                           prefill_kv_parts=pa.PA_PREFILL_PARTS_AUTO),
                            b.num_rows, b.total_q, "cuda")

    def afn():
        pa.paged_attn_mixed(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, out=out, workspace=aws,
                            num_splits=pa.PA_SPLITS_BY_LENGTH,
                            prefill_kv_parts=pa.PA_PREFILL_PARTS_AUTO, **kw)
    ams = time_calls(afn, steps, warmup, stream)
    res["whole_call_by_length_auto_parts"] = {
        "ms": round(ams, 4), "TFLOP/s_of_prefill": round(F / (ams * 1e-3) / 1e12, 1),
        "note": "num_splits = PA_SPLITS_BY_LENGTH and prefill_kv_parts = PA_PREFILL_PARTS_AUTO"}
    del aws
    # each half as a call of its own: the chunk's row through the prefill
    # entry, the three resident rows through the decode entry
    for name, rows, entry in (("prefill_row_alone", [0], pa.paged_attn_prefill),
                              ("decode_rows_alone", [1, 2, 3], pa.paged_attn_decode)):
        sb = workloads.sub_batch(b, rows, device="cuda")
        sws = pa.make_workspace(pa.make_params(sb.q, sb.k_cache), sb.num_rows, sb.total_q, "cuda")
        sout = torch.empty_like(sb.q)
        skw = call_args(sb)

        def sfn():
            entry(sb.q, sb.k_cache, sb.v_cache, sb.block_table, sb.cu_seqlens_q, sb.seq_lens,
                  out=sout, workspace=sws, **skw)
        sms = time_calls(sfn, steps, warmup, stream)
        if name.startswith("prefill"):
            tf = F / (sms * 1e-3) / 1e12
            res[name] = {"ms": round(sms, 4), "TFLOP/s": round(tf, 1),
                         "frac_of_bf16_peak": round(tf / pk["bf16"], 4)}
        else:
            gbs = byt / (sms * 1e-3) / 1e9
            res[name] = {"ms": round(sms, 4), "GB/s": round(gbs, 1),
                         "frac_of_hbm": round(gbs / pk["hbm"], 4)}
            # the same rows with the length-only split count for long rows
            # (parts of 2048 keys on the tcgen05 tile kernel)
            lws = pa.make_workspace(pa.make_params(sb.q, sb.k_cache,
                                                   num_splits=pa.PA_SPLITS_BY_LENGTH),
                                    sb.num_rows, sb.total_q, "cuda")

            def lfn():
                entry(sb.q, sb.k_cache, sb.v_cache, sb.block_table, sb.cu_seqlens_q, sb.seq_lens,
                      out=sout, workspace=lws, num_splits=pa.PA_SPLITS_BY_LENGTH, **skw)
            lms = time_calls(lfn, steps, warmup, stream)
            lgbs = byt / (lms * 1e-3) / 1e9
            res[name + "_by_length"] = {
                "ms": round(lms, 4), "GB/s": round(lgbs, 1), "frac_of_hbm": round(lgbs / pk["hbm"], 4),
                "note": "num_splits = PA_SPLITS_BY_LENGTH: rows over 32768 keys cut into parts of "
                        "2048 keys on the tcgen05 tile kernel"}
            del lws
        if name.startswith("prefill"):
            # the same row with the part count chosen per call (cut in 3 here)
            aws = pa.make_workspace(pa.make_params(sb.q, sb.k_cache,
                                                   prefill_kv_parts=pa.PA_PREFILL_PARTS_AUTO),
                                    sb.num_rows, sb.total_q, "cuda")

            def afn():
                entry(sb.q, sb.k_cache, sb.v_cache, sb.block_table, sb.cu_seqlens_q, sb.seq_lens,
                      out=sout, workspace=aws, prefill_kv_parts=pa.PA_PREFILL_PARTS_AUTO, **skw)
            ams = time_calls(afn, steps, warmup, stream)
            atf = F / (ams * 1e-3) / 1e12
            res["prefill_row_alone_auto_parts"] = {
                "ms": round(ams, 4), "TFLOP/s": round(atf, 1),
                "frac_of_bf16_peak": round(atf / pk["bf16"], 4),
                "note": "prefill_kv_parts = PA_PREFILL_PARTS_AUTO: key-range parts merged by "
                        "log-sum-exp, count chosen for the device"}
            del aws
        del sb, sws, sout
    del b, ws, out
    torch.cuda.empty_cache()
    return res


def part_prefill_fp8(steps, warmup, stream, pk):
    """The varlen prefill workload's shapes with fp16 Q and an fp8 E5M2 cache
    (per-tensor scales 0.5 / 2.0): the prefill path's fp8 dequant."""
    import paged_kv_attention_prefill_gb300 as pa
    b = workloads.make_workload(2, device="cuda", data_device="cuda", q_dtype="f16",
                                kv_dtype="e5m2", k_scale=0.5, v_scale=2.0)
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    kw = call_args(b)

    def fn():
        pa.paged_attn_prefill(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                              b.seq_lens, out=out, workspace=ws, **kw)
    ms = time_calls(fn, steps, warmup, stream)
    F = metrics.prefill_flops(b.q_lens, b.kv_lens, b.num_q_heads, b.head_dim)
    tf = F / (ms * 1e-3) / 1e12
    res = {"workload": workloads.WORKLOADS[2] + ", with fp16 Q and an fp8_e5m2 KV cache",
           "ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_of_fp16_peak": round(tf / pk["bf16"], 4)}
    del b, ws, out
    torch.cuda.empty_cache()
    return res


def part_prefill_fp8_d256(steps, warmup, stream, pk):
    """The mixed workload's 2048-token prefill row alone (d = 256) with fp16 Q
    and an fp8 E5M2 cache (per-tensor scales 0.5 / 2.0)."""
    import paged_kv_attention_prefill_gb300 as pa
    full = workloads.make_workload(3, device="cuda", data_device="cuda", kv_dtype="e5m2",
                                   k_scale=0.5, v_scale=2.0)
    b = workloads.sub_batch(full, [0], device="cuda")
    del full
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    kw = call_args(b)

    def fn():
        pa.paged_attn_prefill(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                              b.seq_lens, out=out, workspace=ws, **kw)
    ms = time_calls(fn, steps, warmup, stream)
    F = metrics.prefill_flops(b.q_lens, b.kv_lens, b.num_q_heads, b.head_dim)
    tf = F / (ms * 1e-3) / 1e12
    res = {"workload": "the mixed workload's prefill row alone (2048 tokens after 150000 cached, "
                       "24/4 heads, d=256) with fp16 Q and an fp8_e5m2 KV cache",
           "ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac_of_fp16_peak": round(tf / pk["bf16"], 4)}
    del b, ws, out
    torch.cuda.empty_cache()
    return res


def part_small1(steps, warmup, stream):
    import paged_kv_attention_prefill_gb300 as pa
    b = workloads.make_workload(1).to("cuda")
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    kw = call_args(b)

    def fn():
        pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                             b.seq_lens, out=out, workspace=ws, **kw)
    ms = time_calls(fn, steps, warmup, stream)

    def fn_static():
        pa.paged_attn_decode_static(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                                    b.seq_lens, out=out, **kw)
    ms_graph = graph_ms(fn, steps, warmup, stream)
    ms_static_graph = graph_ms(fn_static, steps, warmup, stream)
    host_us = host_us_per_call(b, ws, out)

    def fn_sep():
        pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                             b.seq_lens, out=out, workspace=ws,
                             merge_mode=pa.PA_MERGE_SEPARATE, **kw)
    ms_sep = time_calls(fn_sep, steps, warmup, stream)
    ms_sep_graph = graph_ms(fn_sep, steps, warmup, stream)
    return {"workload": workloads.WORKLOADS[1], "us_per_call": round(ms * 1e3, 2),
            "graph_replay_us_per_call": round(ms_graph * 1e3, 2),
            "merge": "in the decode launch (PA_MERGE_AUTO picks it: the grid is smaller than "
                     "the GPU)",
            "separate_merge_us_per_call": round(ms_sep * 1e3, 2),
            "separate_merge_graph_replay_us_per_call": round(ms_sep_graph * 1e3, 2),
            "static_entry_graph_replay_us_per_call": round(ms_static_graph * 1e3, 2),
            "host_us_per_call": host_us,
            "host_note": "wall time of the C ABI call itself (argument checks, tensor-map "
                         "encoding, launches), from a loop of ctypes calls with argument "
                         "structs built once, no stream sync inside the loop; median of "
                         "10 loops of 100 calls",
            "note": "launch-latency bound (0.59 MB); paged_attn_decode_static (no workspace "
                    "argument) clears its array's work counters with a memset node first"}


def host_us_per_call(b, ws, out, calls=100, loops=10):
    """Host-side cost of one paged_attn_decode call through the C ABI."""
    import ctypes
    import paged_kv_attention_prefill_gb300 as pa
    lib = pa.load()
    prm = pa.make_params(b.q, b.k_cache, softmax_scale=b.softmax_scale, k_scale=b.k_scale,
                         v_scale=b.v_scale)
    cu_h, lens_h = b.cu_seqlens_q.cpu().contiguous(), b.seq_lens.cpu().contiguous()
    bat = pa.Batch(b.num_rows, b.total_q, b.num_pages, int(b.block_table.shape[1]),
                   b.cu_seqlens_q.data_ptr(), b.seq_lens.data_ptr(), b.block_table.data_ptr(),
                   cu_h.data_ptr(), lens_h.data_ptr())
    fn = lib.paged_attn_decode
    args = (ctypes.byref(prm), ctypes.byref(bat), b.q.data_ptr(), b.k_cache.data_ptr(),
            b.v_cache.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
            torch.cuda.current_stream().cuda_stream)
    per = []
    for _ in range(loops + 1):
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(calls):
            fn(*args)
        per.append((time.perf_counter() - t) / calls * 1e6)
        torch.cuda.synchronize()
    return round(statistics.median(per[1:]), 2)


def cpu_baseline_sample(b, budget_s=12.0, one_thread=True):
    """Times the oracle on sampled query tokens of the workload; returns
    (TFLOP/s, cores, description)."""
    import oracle
    cpu = b.to("cpu")
    args = cpu.oracle_args()
    ql, kl = cpu.q_lens, cpu.kv_lens
    cu = [0]
    for q in ql:
        cu.append(cu[-1] + q)
    # one token from the end of each row (the most keys), scaled up to the budget
    pool = []
    for r, q in enumerate(ql):
        for i in range(q - 1, -1, -max(1, q // 64)):
            pool.append((cu[r] + i, kl[r] - q + i + 1))
    pool.sort(key=lambda x: x[0])
    probe = pool[:: max(1, len(pool) // 8)][:8]
    t = time.perf_counter()
    oracle.paged_attention(tokens=[x[0] for x in probe], **args)
    dt = time.perf_counter() - t
    fl_probe = sum(4 * cpu.head_dim * cpu.num_q_heads * k for _, k in probe)
    rate = fl_probe / max(dt, 1e-6)
    want = rate * budget_s
    pick, acc = [], 0
    for x in pool[:: max(1, len(pool) // 4096)]:
        if acc >= want:
            break
        pick.append(x)
        acc += 4 * cpu.head_dim * cpu.num_q_heads * x[1]
    t = time.perf_counter()
    oracle.paged_attention(tokens=[x[0] for x in pick], **args)
    dt = time.perf_counter() - t
    cores = oracle.num_threads()  # before the one-thread run below changes it
    extra = {"cpu_model": cpu_model(), "nproc": os.cpu_count()}
    if one_thread:
        # one thread, on a thirty-second of the sample
        one = pick[: max(1, len(pick) // 32)]
        acc1 = sum(4 * cpu.head_dim * cpu.num_q_heads * x[1] for x in one)
        t = time.perf_counter()
        oracle.paged_attention(tokens=[x[0] for x in one], threads=1, **args)
        extra["one_thread_value"] = round(acc1 / (time.perf_counter() - t) / 1e12, 6)
    return acc / dt / 1e12, cores, \
        f"{len(pick)} query tokens x {cpu.num_q_heads} heads of the workload ({acc:.3e} FLOP, {dt:.1f} s)", \
        extra


def cpu_model():
    """The host CPU's model name (x86) or architecture and part number (Arm)."""
    import platform
    name = part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key = key.strip().lower()
                if key == "model name" and not name:
                    name = val.strip()
                elif key == "cpu part" and not part:
                    part = val.strip()
    except OSError:
        pass
    if name:
        return name
    return f"{platform.machine()} (CPU part {part})" if part else platform.machine()


def run_ours(args):
    import paged_kv_attention_prefill_gb300 as pa
    from paged_kv_attention_prefill_gb300 import build as pa_build
    rank, world, local = padist.env_rank_world()
    torch.cuda.set_device(local)
    padist.init("nccl")
    pa_build.build()
    pk = peaks()
    stream = torch.cuda.current_stream()
    b = workloads.make_workload(HEADLINE_WORKLOAD, device="cuda", data_device="cuda",
                                page_size=16)
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    kw = call_args(b)
    ql, kl = b.q_lens, b.kv_lens
    F = metrics.prefill_flops(ql, kl, b.num_q_heads, b.head_dim)

    def step():
        pa.paged_attn_mixed(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                            b.seq_lens, out=out, workspace=ws, **kw)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    ms_local = time_calls(step, args.steps, args.warmup, stream, sampler)
    clocks = sampler.stop() if sampler else None
    ms = padist.max_over_ranks(ms_local, device="cuda")
    total_flops = F * world
    value = total_flops / (ms * 1e-3) / 1e12
    achieved = F / (ms_local * 1e-3) / 1e12

    # end to end through the public API with host buffers, fed the way a
    # serving loop feeds it: step i+1's inputs are copied host -> device (two
    # copy streams, the K cache on one, everything else on the other) into a
    # second set of device buffers while step i computes, and step i's output
    # is copied back behind it.  Every step's copies are inside the timed
    # region, which runs from before the first upload to after the last
    # download.
    names = ("q", "k_cache", "v_cache", "block_table", "cu_seqlens_q", "seq_lens")
    in_bytes = sum(getattr(b, k).numel() * getattr(b, k).element_size() for k in names)
    host = {k: getattr(b, k).cpu().pin_memory() for k in names}
    dev = [{k: torch.empty_like(getattr(b, k)) for k in names} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    out_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    groups = (("k_cache",), ("v_cache", "q", "block_table", "cu_seqlens_q", "seq_lens"))

    def e2e_run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ready = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        back = [torch.cuda.Event() for _ in range(n)]
        start.record(stream)

        def upload(i):
            for c, keys, ev in zip(copy_streams, groups, ready[i]):
                c.wait_event(start)
                if i >= 2:
                    c.wait_event(done[i - 2])  # the buffer set is free again
                with torch.cuda.stream(c):
                    for k in keys:
                        dev[i % 2][k].copy_(host[k], non_blocking=True)
                ev.record(c)

        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            for ev in ready[i]:
                stream.wait_event(ev)
            if i >= 2:
                stream.wait_event(back[i - 2])  # the output buffer is free again
            d = dev[i % 2]
            pa.paged_attn_mixed(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                d["cu_seqlens_q"], d["seq_lens"], out=outs[i % 2], workspace=ws,
                                **kw)
            done[i].record(stream)
            c = copy_streams[1]
            c.wait_event(done[i])
            with torch.cuda.stream(c):
                out_host[i % 2].copy_(outs[i % 2], non_blocking=True)
            back[i].record(c)
        stream.wait_event(back[n - 1])
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / n

    e2e_steps = max(3, min(args.steps, 20))
    e2e_run(2)  # warm-up
    padist.barrier()
    ms_e2e = padist.max_over_ranks(e2e_run(e2e_steps), device="cuda")
    e2e_val = total_flops / (ms_e2e * 1e-3) / 1e12
    del host, dev, outs, out_host
    torch.cuda.empty_cache()

    res = None
    if rank == 0:
        parts = {}
        if not args.headline_only:
            ps, pw = max(5, min(args.steps, 30)), 3
            parts["decode_split_kv_256rows"] = part_decode(4, ps, pw, stream, pk)
            parts["decode_long_context_fp8"] = part_decode(5, ps, pw, stream, pk,
                                                           by_length=True)
            parts["mixed_chunk_plus_decode"] = part_mixed3(ps, pw, stream, pk)
            parts["prefill_fp8_cache"] = part_prefill_fp8(ps, pw, stream, pk)
            parts["prefill_fp8_cache_d256"] = part_prefill_fp8_d256(ps, pw, stream, pk)
            parts["decode_small_4rows"] = part_small1(max(ps, 50), 5, stream)
        cpu_val, cores, sample, cpu_extra = cpu_baseline_sample(b, budget_s=args.cpu_seconds)
        res = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, shuffled block tables, poisoned unused slots)",
            "config": headline_config(b, world), "entry": "paged_attn_mixed",
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                         "peak": pk["bf16"], "unit": "TFLOP/s",
                         "frac": round(achieved / pk["bf16"], 4), "traffic": profiled_traffic(),
                         "kernel": "prefill_tc2_kernel (whole call timed: routing kernel included)",
                         "peak_source": f"{pk['source']} bf16 burst"},
            "cpu_baseline": {"value": round(cpu_val, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample, **cpu_extra},
            "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "ms_per_step": round(ms_e2e, 3),
                    "h2d_bytes_per_step": in_bytes,
                    "d2h_bytes_per_step": out.numel() * out.element_size(),
                    "steps": e2e_steps,
                    "how": "pinned host buffers; step i+1's uploads (two copy streams) overlap "
                           "step i's compute, each step's download follows it"},
            "gpu_launches": launches_per_call(ql) * args.steps,
            "clocks": clocks,
            "parts": parts,
        }
        print(json.dumps(res), flush=True)
    padist.barrier()
    return res


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = padist.env_rank_world()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    b = workloads.make_workload(HEADLINE_WORKLOAD, page_size=16)
    # each step one bounded sample, sized so that the whole run stays within
    # about two and a half minutes whatever --steps and --warmup are
    budget = min(args.ref_seconds, max(0.3, 150.0 / (args.steps + args.warmup)))
    vals, secs, descr, cores = [], [], "", oracle.num_threads()
    for s in range(args.warmup + args.steps):
        t = time.perf_counter()
        v, cores, descr, _ = cpu_baseline_sample(b, budget_s=budget, one_thread=False)
        dt = time.perf_counter() - t
        if s >= args.warmup:
            vals.append(v)
            secs.append(dt)
    value = statistics.median(vals)
    F = metrics.prefill_flops(b.q_lens, b.kv_lens, b.num_q_heads, b.head_dim)
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(statistics.median(secs) * 1e3, 1),
           "ms_per_step_note": "measured wall time of one step: one bounded sample of the "
                               "workload's query tokens, not the whole workload",
           "ms_whole_workload_extrapolated": round(F / (value * 1e12) * 1e3, 1) if value > 0 else None,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) bf16, shuffled block tables, poisoned unused slots)",
           "config": headline_config(b, world), "entry": "oracle (fp64 C, OpenMP)",
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                            "kind": "oracle", "sample": f"per step: {descr}"},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


def run_profile(args):
    """Runs one part of the path `steps` times with no reporting: the command
    that ncu captures.  Only the profiled rows are generated on the device
    (--profile-rows keeps the first R rows of the part; decode3 is the mixed
    workload's three resident rows through the decode entry), so a capture
    holds the small case it measures and nothing else."""
    import paged_kv_attention_prefill_gb300 as pa
    from paged_kv_attention_prefill_gb300 import build as pa_build
    pa_build.build()
    n, rows = {"prefill": (2, None), "mixed3": (3, None), "mixed3fp8": (3, None),
               "decode3": (3, [1, 2, 3]), "decode4": (4, None), "decode5": (5, None),
               "decode1": (1, None)}[args.profile]
    if rows is None:
        rows = list(range(len(workloads.workload_lengths(n)[0])))
    if args.profile_rows:
        rows = rows[:args.profile_rows]
    # mixed3fp8: the mixed workload with fp16 Q and an fp8 E5M2 cache
    over = dict(kv_dtype="e5m2", k_scale=0.5, v_scale=2.0) if args.profile == "mixed3fp8" else {}
    b = workloads.make_workload(n, device="cuda", data_device="cuda", rows=rows, **over)
    torch.cuda.empty_cache()
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache, num_splits=args.num_splits),
                           b.num_rows, b.total_q, "cuda")
    out = torch.empty_like(b.q)
    fn = pa.paged_attn_decode if args.profile.startswith("decode") else pa.paged_attn_mixed
    for _ in range(args.warmup + args.steps):
        fn(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens, out=out,
           workspace=ws, num_splits=args.num_splits, **call_args(b))
    torch.cuda.synchronize()
    print(f"profiled {args.profile}: rows={b.num_rows} total_q={b.total_q} "
          f"cache={2 * b.k_cache.numel() * b.k_cache.element_size() / 2**20:.0f} MiB "
          f"device bytes held={torch.cuda.max_memory_allocated() / 2**20:.0f} MiB")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=4.0)
    ap.add_argument("--profile", choices=["prefill", "mixed3", "mixed3fp8", "decode3", "decode4",
                                          "decode5", "decode1"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--profile-rows", type=int, default=0)
    args = ap.parse_args()
    if args.profile:
        return run_profile(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
