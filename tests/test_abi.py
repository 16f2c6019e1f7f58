"""The C ABI on the CPU: the library loads, exports what the header declares,
sizes its workspace as documented, and rejects bad arguments before any
launch.  No compute call runs here (without a GPU a valid call stops at the
device check with PA_ERR_NO_DEVICE)."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_attention_prefill_gb300 as pa
from paged_kv_attention_prefill_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_attn.h")

OK, INVALID, UNSUPPORTED, WS_SMALL, CUDA_ERR, NO_DEVICE = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(paged_attn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"paged_attn_prefill", "paged_attn_decode", "paged_attn_mixed",
            "paged_attn_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.paged_attn_version() >= 100
    for code in range(6):
        s = lib.paged_attn_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.paged_attn_status_string(99).decode() == "unknown status"


def params(**kw):
    d = dict(num_q_heads=16, num_kv_heads=4, head_dim=128, page_size=16, q_dtype=pa.PA_BF16,
             kv_dtype=pa.PA_BF16, softmax_scale=0.0, k_scale=1.0, v_scale=1.0, max_decode_q=0,
             num_splits=0)
    d.update(kw)
    return pa.Params(**d)


def test_workspace_matches_the_decode_workspace_figure(lib):
    # fp32 partial state of heads x 16 x (head_dim + 2) x 4 bytes per decode token
    p = params(num_q_heads=16, num_kv_heads=16, head_dim=128)
    per_tok = 16 * 16 * (128 + 2) * 4
    n = pa.workspace_size(p, 64, 64)
    assert 64 * per_tok <= n <= 64 * per_tok + 64 * 1024
    # grows with rows; zero for invalid parameters
    assert pa.workspace_size(p, 128, 128) > n
    assert lib.paged_attn_workspace_size(ctypes.byref(params(page_size=24)), 4, 4) == 0
    assert lib.paged_attn_workspace_size(None, 4, 4) == 0


def test_length_only_split_workspace_and_checks(lib):
    # PA_SPLITS_BY_LENGTH: 128 partial states per decode token and head (the
    # default's 16 times 8) plus the long-row item list; other modes refused
    by_len = pa.PA_SPLITS_BY_LENGTH
    p16 = params(num_q_heads=24, num_kv_heads=4, head_dim=256, q_dtype=pa.PA_F16,
                 kv_dtype=pa.PA_F16)
    plen = params(num_q_heads=24, num_kv_heads=4, head_dim=256, q_dtype=pa.PA_F16,
                  kv_dtype=pa.PA_F16, num_splits=by_len)
    n16, nlen = pa.workspace_size(p16, 8, 40), pa.workspace_size(plen, 8, 40)
    per_split = 24 * (256 + 2) * 4          # one split of one token, all heads
    items = 8 * 128 * 1 * 8                 # rows x splits x 128-row blocks x int2
    assert nlen - n16 >= 40 * (128 - 16) * per_split + items
    assert nlen - n16 <= 40 * (128 - 16) * per_split + items + 4 * 256
    assert lib.paged_attn_workspace_size(ctypes.byref(params(num_splits=-2)), 4, 4) == 0
    for name in ("paged_attn_decode", "paged_attn_mixed"):
        # the decode kernel's cases (16-bit q) with packed verify rows
        for p in (params(head_dim=256, q_dtype=pa.PA_F32, kv_dtype=pa.PA_F32,
                         num_splits=by_len),
                  params(head_dim=64, q_dtype=pa.PA_F16, kv_dtype=pa.PA_E5M2,
                         num_splits=by_len),
                  params(head_dim=256, num_splits=by_len,
                         verify_mode=pa.PA_VERIFY_TOKENWISE)):
            assert FakeCall(lib, p, [1, 1], [10, 20])(name) == UNSUPPORTED
        assert FakeCall(lib, params(num_splits=-2), [1, 1], [10, 20])(name) == UNSUPPORTED
        # the rest pass the argument checks (here they stop at the device)
        for p in (params(num_splits=by_len),
                  params(head_dim=256, q_dtype=pa.PA_F16, kv_dtype=pa.PA_E5M2,
                         num_splits=by_len)):
            rc = FakeCall(lib, p, [1, 1], [10, 20])(name)
            assert rc in (OK, NO_DEVICE) if not torch.cuda.is_available() else True


class FakeCall:
    """Builds argument structs with non-null dummy pointers.  They are never
    dereferenced: every case either fails validation before any launch or,
    on a machine without a GPU, stops at the device check.  Cases that would
    pass validation are skipped where a GPU is present."""

    def __init__(self, lib, p, q_lens, kv_lens, max_pages=64, num_pages=100, ws_bytes=None,
                 host=True):
        self.lib, self.p = lib, p
        self.cu = (ctypes.c_int32 * (len(q_lens) + 1))(*([0] + list(
            __import__("itertools").accumulate(q_lens))))
        self.lens = (ctypes.c_int32 * len(kv_lens))(*kv_lens)
        total = sum(q_lens)
        fake = 0x10000
        self.batch = pa.Batch(len(q_lens), total, num_pages, max_pages, fake, fake, fake,
                              ctypes.cast(self.cu, ctypes.c_void_p) if host else None,
                              ctypes.cast(self.lens, ctypes.c_void_p) if host else None)
        need = lib.paged_attn_workspace_size(ctypes.byref(p), len(q_lens), total)
        self.ws = need if ws_bytes is None else ws_bytes

    def __call__(self, name, **over):
        args = dict(q=0x10000, k=0x10000, v=0x10000, out=0x10000, ws=0x10000)
        args.update(over)
        return getattr(self.lib, name)(ctypes.byref(self.p), ctypes.byref(self.batch), args["q"],
                                       args["k"], args["v"], args["out"], args["ws"], self.ws,
                                       None)


ENTRIES = ["paged_attn_prefill", "paged_attn_decode", "paged_attn_mixed"]


@pytest.mark.parametrize("name", ENTRIES)
def test_rejects_bad_params(lib, name):
    cases = [
        (params(page_size=24), INVALID),
        (params(page_size=0), INVALID),
        (params(num_q_heads=6, num_kv_heads=4), INVALID),
        (params(num_kv_heads=0), INVALID),
        (params(head_dim=96), UNSUPPORTED),
        (params(q_dtype=pa.PA_F32, kv_dtype=pa.PA_E5M2), UNSUPPORTED),
        (params(q_dtype=pa.PA_BF16, kv_dtype=pa.PA_F16), UNSUPPORTED),
        (params(num_splits=8), UNSUPPORTED),
        (params(merge_mode=3), INVALID),
        (params(merge_mode=-1), INVALID),
        (params(softmax_scale=float("nan")), INVALID),
    ]
    for p, want in cases:
        c = FakeCall(lib, p, [1, 1], [10, 20])
        assert c(name) == want, (p.page_size, p.head_dim, want)


@pytest.mark.parametrize("name", ENTRIES)
def test_verify_mode_checks(lib, name):
    # an unknown verify mode is refused by every entry; one-token verify rows
    # run on the 16-bit decode kernel only, so fp32 decode/mixed refuse them
    assert FakeCall(lib, params(verify_mode=7), [1, 1], [10, 20])(name) == INVALID
    if name != "paged_attn_prefill":
        p = params(q_dtype=pa.PA_F32, kv_dtype=pa.PA_F32, verify_mode=pa.PA_VERIFY_TOKENWISE)
        assert FakeCall(lib, p, [1, 1], [10, 20])(name) == UNSUPPORTED


@pytest.mark.parametrize("name", ENTRIES)
def test_rejects_bad_batches(lib, name):
    p = params()
    assert FakeCall(lib, p, [1], [-2])(name) == INVALID                 # negative length
    assert FakeCall(lib, p, [1], [64 * 16 + 1])(name) == INVALID        # L beyond the table
    c = FakeCall(lib, p, [1, 1], [10, 20])
    assert c(name, ws=None) == INVALID                                  # null workspace
    assert c(name, q=None) == INVALID                                   # null q
    assert c(name, k=None) == INVALID                                   # null cache
    small = FakeCall(lib, p, [1, 1], [10, 20], ws_bytes=1024)
    assert small(name) == WS_SMALL
    assert getattr(lib, name)(None, None, None, None, None, None, None, 0, None) == INVALID


def test_decode_rejects_long_rows_with_host_mirrors(lib):
    p = params(max_decode_q=4)
    assert FakeCall(lib, p, [5], [50])("paged_attn_decode") == INVALID
    if torch.cuda.is_available():
        return  # a valid call with dummy pointers must never reach a launch
    # the same row passes validation for the mixed call (routed to prefill) and prefill
    for name in ("paged_attn_mixed", "paged_attn_prefill"):
        assert FakeCall(lib, p, [5], [50])(name) == NO_DEVICE


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
@pytest.mark.parametrize("name", ENTRIES)
def test_valid_call_without_gpu_stops_at_device_check(lib, name):
    ql = [1, 4] if name == "paged_attn_decode" else [1, 70]
    assert FakeCall(lib, params(), ql, [10, 200])(name) == NO_DEVICE
    assert FakeCall(lib, params(), ql, [10, 200], host=False)(name) == NO_DEVICE


def test_empty_batch_is_ok_or_no_device(lib):
    for name in ENTRIES:
        assert FakeCall(lib, params(), [], [])(name) in (OK, NO_DEVICE)


def test_prefill_parts_workspace_and_checks(lib):
    # K prefill parts add K fp32 states (acc[d], m, l) per query token and head
    # (and K times the work-list entries); 0 and 1 leave the workspace as it is
    base = pa.workspace_size(params(), 8, 1000)
    assert pa.workspace_size(params(prefill_kv_parts=1), 8, 1000) == base
    for k in (2, 8, 16):
        grown = pa.workspace_size(params(prefill_kv_parts=k), 8, 1000) - base
        states = 1000 * 16 * k * (128 + 2) * 4
        assert states <= grown <= states + 1000 * 16 * k * 8 + 64 * 1024
    for bad in (-2, 17):
        assert lib.paged_attn_workspace_size(ctypes.byref(params(prefill_kv_parts=bad)), 4, 4) == 0
        for name in ENTRIES:
            assert FakeCall(lib, params(prefill_kv_parts=bad), [1, 1], [10, 20])(name) == INVALID
    # the count chosen per call: the workspace holds 4 parts; -2 is refused
    assert pa.workspace_size(params(prefill_kv_parts=pa.PA_PREFILL_PARTS_AUTO), 8, 1000) == \
        pa.workspace_size(params(prefill_kv_parts=4), 8, 1000)
    assert lib.paged_attn_workspace_size(ctypes.byref(params(prefill_kv_parts=-2)), 4, 4) == 0
    for name in ENTRIES:
        assert FakeCall(lib, params(prefill_kv_parts=-2), [1, 1], [10, 20])(name) == INVALID
        assert FakeCall(lib, params(prefill_kv_parts=-1), [1, 1], [10, 20])(name) in (OK, NO_DEVICE)
    # decode never cuts prefill items: its workspace need is the uncut one
    p = params(prefill_kv_parts=8)
    c = FakeCall(lib, p, [1, 1], [10, 20], ws_bytes=pa.workspace_size(params(), 2, 2))
    assert c("paged_attn_decode") in (OK, NO_DEVICE)
    assert c("paged_attn_prefill") == WS_SMALL


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import importlib
    mod = importlib.reload(pa)
    monkeypatch.setattr(mod, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(mod.PagedAttnError):
        mod.load()
    importlib.reload(pa)
