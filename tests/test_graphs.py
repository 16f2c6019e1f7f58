"""The compute calls under CUDA-graph capture and replay.

The calls make no host sync and allocate nothing, and their grids depend only
on the batch's row and token counts, so a serving loop can capture one step
and replay it with new data in the same buffers.  The mixed call with both
kinds of rows forks its decode rows onto the library's second stream, which
must join the capture too.  Each replay is compared bitwise with an eager
call on the same inputs.
"""
import pytest
import torch

import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build
from paged_kv_attention_prefill_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()
    torch.cuda.init()


def _args(b):
    return dict(softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale,
                cu_seqlens_q_host=b.cu_seqlens_q.cpu(), seq_lens_host=b.seq_lens.cpu())


def _bitwise(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("entry,q_lens,kv_lens,kv", [
    ("mixed", [300, 1, 4, 0, 17, 5], [900, 700, 90, 0, 17, 2000], None),
    ("mixed", [129, 1, 3], [2000, 5000, 40], "e5m2"),
    ("decode", [1, 4, 1, 5, 1], [1, 700, 2049, 64, 9000], None),
    ("prefill", [65, 300, 7], [65, 1500, 40], None),
])
def test_capture_and_replay_bitwise(entry, q_lens, kv_lens, kv):
    b = workloads.make_batch(q_lens, kv_lens, num_q_heads=8, num_kv_heads=2, head_dim=128,
                             page_size=16, q_dtype="f16", kv_dtype=kv, seed=51,
                             k_scale=0.5 if kv else 1.0, v_scale=2.0 if kv else 1.0,
                             device="cuda")
    fn = {"mixed": pa.paged_attn_mixed, "decode": pa.paged_attn_decode,
          "prefill": pa.paged_attn_prefill}[entry]
    ws = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    ws_eager = pa.make_workspace(pa.make_params(b.q, b.k_cache), b.num_rows, b.total_q, "cuda")
    out_g = torch.empty_like(b.q)
    kw = _args(b)

    def call(out, workspace):
        fn(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens, out=out,
           workspace=workspace, **kw)

    call(out_g, ws)  # one-time set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(out_g, ws)
    torch.cuda.synchronize()
    for step in range(3):
        # new query values in the captured buffer, then replay vs an eager call
        b.q.copy_(torch.randn(b.q.shape, generator=torch.Generator().manual_seed(60 + step))
                  .to(b.q.dtype).to("cuda"))
        out_g.fill_(float("nan"))
        g.replay()
        out_e = torch.full_like(b.q, float("nan"))
        call(out_e, ws_eager)
        torch.cuda.synchronize()
        assert torch.isfinite(out_g.float()).all()
        assert _bitwise(out_g, out_e)
    assert pa.read_errors(ws) == 0


def test_static_decode_capture_and_replay_bitwise():
    b = workloads.make_batch([1, 4, 1], [33, 700, 4097], num_q_heads=8, num_kv_heads=2,
                             head_dim=128, page_size=16, q_dtype="bf16", seed=52, device="cuda")
    kw = dict(softmax_scale=b.softmax_scale)
    out_g = torch.empty_like(b.q)

    def static(out):
        pa.paged_attn_decode_static(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                                    b.seq_lens, out=out, **kw)

    static(out_g)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        static(out_g)
    for step in range(2):
        b.q.copy_(torch.randn(b.q.shape, generator=torch.Generator().manual_seed(70 + step))
                  .to(b.q.dtype).to("cuda"))
        g.replay()
        out_e = pa.paged_attn_decode(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                                     b.seq_lens, **kw)
        torch.cuda.synchronize()
        assert _bitwise(out_g, out_e)


@pytest.mark.parametrize("entry", ["decode", "mixed"])
def test_capture_and_replay_long_rows_split_by_length(entry):
    # rows over 32768 keys cut into 2048-key parts on the tile kernel (its
    # item list built on the device), with and without a prefill row beside
    # them; replayed bitwise like the eager call, the merge in either place
    q_lens = [1, 4, 1] if entry == "decode" else [200, 1, 4]
    kv_lens = [40000, 36000, 900] if entry == "decode" else [3000, 40000, 36000]
    b = workloads.make_batch(q_lens, kv_lens, num_q_heads=12, num_kv_heads=2, head_dim=256,
                             page_size=16, q_dtype="f16", seed=53, device="cuda",
                             data_device="cuda")
    fn = {"mixed": pa.paged_attn_mixed, "decode": pa.paged_attn_decode}[entry]
    by_len = pa.PA_SPLITS_BY_LENGTH
    prm = pa.make_params(b.q, b.k_cache, num_splits=by_len)
    for mode in (pa.PA_MERGE_SAME_LAUNCH, pa.PA_MERGE_SEPARATE):
        ws = pa.make_workspace(prm, b.num_rows, b.total_q, "cuda")
        ws_eager = pa.make_workspace(prm, b.num_rows, b.total_q, "cuda")
        out_g = torch.empty_like(b.q)
        kw = dict(_args(b), num_splits=by_len, merge_mode=mode)

        def call(out, workspace):
            fn(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens, out=out,
               workspace=workspace, **kw)

        call(out_g, ws)  # one-time set-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call(out_g, ws)
        out_e = torch.empty_like(b.q)
        for _ in range(3):
            out_g.zero_()
            g.replay()
            call(out_e, ws_eager)
            torch.cuda.synchronize()
            assert _bitwise(out_g, out_e)
        assert pa.read_errors(ws) == 0 and pa.read_errors(ws_eager) == 0
        del g
