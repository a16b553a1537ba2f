"""The Python binding only marshals arguments: each wrapper must hand every
tensor, size and option to the C call in the parameter the header names for
it.  Run on the CPU against a stand-in library that records the calls (the
wrappers' CUDA-device check is relaxed to accept CPU tensors; nothing is
launched), so that a swapped, dropped or stale argument fails here and not
only on a GPU."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_attention_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STREAM = 0x5151


def _params():
    """name -> [parameter names] of every PKV_API prototype in include/pkv.h."""
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", src, flags=re.S))
    out = {}
    for name, params in re.findall(r"PKV_API\s+[\w\s\*]*?\b(pkv_\w+)\s*\(([^)]*)\)\s*;", src):
        ps = [p.split()[-1].lstrip("*") for p in params.split(",") if p.strip() != "void"]
        out[name] = ps
    return out


PARAMS = _params()


class _Recorder:
    """Stands in for libpkv: records each entry-point call by parameter name."""

    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("pkv_"):
            raise AttributeError(name)
        if name in ("pkv_minference_sizes", "pkv_status_string"):  # host-only arithmetic
            return getattr(self.real, name)

        def call(*args):
            names = PARAMS[name]
            assert len(args) == len(names), f"{name}: {len(args)} arguments"
            self.calls.append((name, dict(zip(names, args))))
            return 4096 if name.endswith("_workspace_size") else 0
        return call

    def last(self, name):
        hits = [a for n, a in self.calls if n == name]
        assert hits, f"{name} was not called"
        return hits[-1]


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder(pkv.load_library())

    def contig(name, t, dtype=None, ndim=None):  # as the binding's, minus the device check
        pkv._require(t.is_contiguous(), f"{name} must be contiguous")
        if dtype is not None:
            pkv._require(t.dtype == dtype, f"{name} must be {dtype}")
        if ndim is not None:
            pkv._require(t.dim() == ndim, f"{name} must have {ndim} dims")

    monkeypatch.setattr(pkv, "load_library", lambda *a, **k: rec)
    monkeypatch.setattr(pkv, "_cuda_contig", contig)
    monkeypatch.setattr(pkv, "_stream_handle", lambda s: STREAM)
    return rec


def _desc_fields(d):
    return (d.num_blocks, d.block_size, d.num_kv_heads, d.head_dim, d.dtype, d.layout)


BF16, F32, I32, I64 = torch.bfloat16, torch.float32, torch.int32, torch.int64


def _pools(layout="NHD", nb=10, bs=16, hkv=2, d=64, dtype=BF16):
    shape = (nb, bs, hkv, d) if layout == "NHD" else (nb, hkv, bs, d)
    return torch.zeros(shape, dtype=dtype), torch.zeros(shape, dtype=dtype)


def test_reshape_and_cache(lib):
    kc, vc = _pools("HND")
    key, value = torch.zeros(5, 2, 64, dtype=BF16), torch.zeros(5, 2, 64, dtype=BF16)
    slots, err = torch.zeros(5, dtype=I64), torch.zeros(1, dtype=I32)
    pkv.reshape_and_cache(key, value, kc, vc, slots, dev_error=err, layout="HND")
    a = lib.last("pkv_reshape_and_cache")
    assert a["key"] == key.data_ptr() and a["value"] == value.data_ptr()
    assert a["k_cache"] == kc.data_ptr() and a["v_cache"] == vc.data_ptr()
    assert a["slot_mapping"] == slots.data_ptr() and a["num_tokens"] == 5
    assert _desc_fields(a["cache"]) == (10, 16, 2, 64, pkv.PKV_BF16, 1)
    assert a["dev_error"] == err.data_ptr() and a["stream"] == STREAM


@pytest.mark.parametrize("noalloc", [False, True])
def test_paged_decode(lib, noalloc):
    kc, vc = _pools(dtype=F32)
    q, out = torch.zeros(3, 8, 64, dtype=F32), torch.zeros(3, 8, 64, dtype=F32)
    bt, sl = torch.zeros(3, 7, dtype=I32), torch.zeros(3, dtype=I32)
    sink, lse = torch.zeros(8, dtype=F32), torch.zeros(3, 8, dtype=F32)
    err = torch.zeros(1, dtype=I32)
    kw = dict(sink=sink, window_left=5, sm_scale=0.25, partition_size=256, out=out, lse=lse,
              dev_error=err)
    if noalloc:
        got = pkv.paged_decode_noalloc(q, kc, vc, bt, sl, 99, **kw)
        a = lib.last("pkv_paged_decode_noalloc")
    else:
        alibi = torch.zeros(8, dtype=F32)
        ws = torch.zeros(8192, dtype=torch.uint8)
        got = pkv.paged_decode(q, kc, vc, bt, sl, 99, workspace=ws, alibi_slopes=alibi, **kw)
        a = lib.last("pkv_paged_decode")
        assert a["alibi_slopes"] == alibi.data_ptr()
        assert a["workspace"] == ws.data_ptr() and a["workspace_bytes"] == 8192
        size = lib.last("pkv_paged_decode_workspace_size")
        assert list(size.values()) == [3, 8, 64, 99, 256, 5]
    assert got is out
    assert a["out"] == out.data_ptr() and a["q"] == q.data_ptr()
    assert a["k_cache"] == kc.data_ptr() and a["v_cache"] == vc.data_ptr()
    assert _desc_fields(a["cache"]) == (10, 16, 2, 64, pkv.PKV_F32, 0)
    assert a["block_table"] == bt.data_ptr() and a["max_blocks_per_seq"] == 7
    assert a["cache_seqlens"] == sl.data_ptr() and a["max_seqlen"] == 99
    assert a["sink"] == sink.data_ptr() and a["batch"] == 3 and a["num_qo_heads"] == 8
    assert a["window_left"] == 5 and a["sm_scale"] == 0.25 and a["partition_size"] == 256
    assert a["lse_out"] == lse.data_ptr() and a["dev_error"] == err.data_ptr()
    assert a["stream"] == STREAM


def test_paged_decode_defaults(lib):
    kc, vc = _pools()
    q = torch.zeros(2, 4, 64, dtype=BF16)
    pkv.paged_decode(q, kc, vc, torch.zeros(2, 3, dtype=I32), torch.zeros(2, dtype=I32), 48)
    a = lib.last("pkv_paged_decode")
    assert a["sink"] is None and a["alibi_slopes"] is None and a["lse_out"] is None
    assert a["dev_error"] is None and a["window_left"] == -1 and a["partition_size"] == 512
    assert a["sm_scale"] == 64 ** -0.5
    assert a["workspace_bytes"] >= 4096  # the size the library asked for


def test_varlen_prefill(lib):
    kc, vc = _pools()
    q, out = torch.zeros(20, 8, 64, dtype=BF16), torch.zeros(20, 8, 64, dtype=BF16)
    bt = torch.zeros(2, 9, dtype=I32)
    cuq, cuk = torch.zeros(3, dtype=I32), torch.zeros(3, dtype=I32)
    sink, alibi = torch.zeros(8, dtype=F32), torch.zeros(8, dtype=F32)
    lse, err = torch.zeros(20, 8, dtype=F32), torch.zeros(1, dtype=I32)
    pkv.varlen_prefill(q, kc, vc, bt, cuq, cuk, 12, 140, sink=sink, causal=False,
                       window_left=7, sm_scale=0.5, out=out, lse=lse, dev_error=err,
                       alibi_slopes=alibi, max_ctas=37)
    a = lib.last("pkv_varlen_prefill")
    assert a["max_ctas"] == 37
    assert a["out"] == out.data_ptr() and a["q"] == q.data_ptr()
    assert a["k_cache"] == kc.data_ptr() and a["v_cache"] == vc.data_ptr()
    assert _desc_fields(a["cache"]) == (10, 16, 2, 64, pkv.PKV_BF16, 0)
    assert a["block_table"] == bt.data_ptr() and a["max_blocks_per_seq"] == 9
    assert a["cu_seq_lens_q"] == cuq.data_ptr() and a["cu_seq_lens_k"] == cuk.data_ptr()
    assert a["max_seqlen_q"] == 12 and a["max_seqlen_k"] == 140 and a["total_q"] == 20
    assert a["sink"] == sink.data_ptr() and a["alibi_slopes"] == alibi.data_ptr()
    assert a["batch"] == 2 and a["num_qo_heads"] == 8 and a["causal"] == 0
    assert a["window_left"] == 7 and a["sm_scale"] == 0.5
    assert a["lse_out"] == lse.data_ptr() and a["dev_error"] == err.data_ptr()
    assert a["stream"] == STREAM
    size = lib.last("pkv_varlen_prefill_workspace_size")
    assert list(size.values()) == [2, 8, 2, 20, 12]


def test_varlen_prefill_contiguous(lib):
    q = torch.zeros(20, 8, 64, dtype=BF16)
    k, v = torch.zeros(50, 2, 64, dtype=BF16), torch.zeros(50, 2, 64, dtype=BF16)
    cuq, cuk = torch.zeros(4, dtype=I32), torch.zeros(4, dtype=I32)
    sink, alibi = torch.zeros(8, dtype=F32), torch.zeros(8, dtype=F32)
    out = pkv.varlen_prefill_contiguous(q, k, v, cuq, cuk, 11, 30, sink=sink, causal=True,
                                        window_left=-1, sm_scale=0.125, alibi_slopes=alibi)
    a = lib.last("pkv_varlen_prefill_contiguous")
    assert a["out"] == out.data_ptr() and a["q"] == q.data_ptr()
    assert a["k"] == k.data_ptr() and a["v"] == v.data_ptr()
    assert (a["total_k"], a["num_kv_heads"], a["head_dim"], a["dtype"]) == (50, 2, 64,
                                                                            pkv.PKV_BF16)
    assert a["cu_seq_lens_q"] == cuq.data_ptr() and a["cu_seq_lens_k"] == cuk.data_ptr()
    assert (a["max_seqlen_q"], a["max_seqlen_k"], a["total_q"]) == (11, 30, 20)
    assert a["sink"] == sink.data_ptr() and a["alibi_slopes"] == alibi.data_ptr()
    assert (a["batch"], a["num_qo_heads"], a["causal"], a["window_left"]) == (3, 8, 1, -1)
    assert a["sm_scale"] == 0.125 and a["lse_out"] is None and a["stream"] == STREAM


def test_rope(lib, monkeypatch):
    tab = pkv.rope_cos_sin_table(33, 32, base=5e5, position_scale=4.0, ntk_alpha=2.5,
                                 device="cpu")
    a = lib.last("pkv_rope_cos_sin_table")
    assert tuple(tab.shape) == (33, 16, 2)
    assert a["cos_sin"] == tab.data_ptr() and a["max_position"] == 33
    assert (a["rotary_dim"], a["base"], a["position_scale"]) == (32, 5e5, 4.0)
    assert a["ntk_alpha"] == 2.5 and a["stream"] == STREAM
    kc, vc = _pools()
    query = torch.zeros(6, 4, 64, dtype=BF16)
    key, value = torch.zeros(6, 2, 64, dtype=BF16), torch.zeros(6, 2, 64, dtype=BF16)
    pos, slots = torch.zeros(6, dtype=I64), torch.zeros(6, dtype=I64)
    err = torch.zeros(1, dtype=I32)
    pkv.rope_reshape_and_cache(query, key, value, kc, vc, pos, slots, tab,
                               is_neox_style=False, dev_error=err)
    a = lib.last("pkv_rope_reshape_and_cache")
    assert a["query"] == query.data_ptr() and a["key"] == key.data_ptr()
    assert a["value"] == value.data_ptr()
    assert a["k_cache"] == kc.data_ptr() and a["v_cache"] == vc.data_ptr()
    assert a["positions"] == pos.data_ptr() and a["slot_mapping"] == slots.data_ptr()
    assert (a["num_tokens"], a["num_qo_heads"]) == (6, 4)
    assert _desc_fields(a["cache"]) == (10, 16, 2, 64, pkv.PKV_BF16, 0)
    assert a["cos_sin"] == tab.data_ptr() and a["max_position"] == 33
    assert (a["rotary_dim"], a["is_neox_style"]) == (32, 0)
    assert a["dev_error"] == err.data_ptr() and a["stream"] == STREAM


def test_minference_prefill(lib):
    q = torch.zeros(300, 8, 64, dtype=BF16)
    k, v = torch.zeros(300, 2, 64, dtype=BF16), torch.zeros(300, 2, 64, dtype=BF16)
    err = torch.zeros(1, dtype=I32)
    out, vi, si = pkv.minference_prefill(q, k, v, vertical_size=40, slash_size=90,
                                         adaptive_budget=None, num_sink_tokens=3,
                                         num_recent_diags=5, sm_scale=0.2, return_pattern=True,
                                         dev_error=err)
    a = lib.last("pkv_minference_prefill")
    assert tuple(vi.shape) == (8, 40) and tuple(si.shape) == (8, 90)
    assert a["out"] == out.data_ptr() and a["q"] == q.data_ptr()
    assert a["k"] == k.data_ptr() and a["v"] == v.data_ptr()
    assert (a["seq_len"], a["num_qo_heads"], a["num_kv_heads"], a["head_dim"]) == (300, 8, 2, 64)
    assert a["dtype"] == pkv.PKV_BF16
    assert (a["vertical_size"], a["slash_size"], a["adaptive_budget"]) == (40, 90, 0.0)
    assert (a["num_sink_tokens"], a["num_recent_diags"], a["sm_scale"]) == (3, 5, 0.2)
    assert a["vertical_indices"] == vi.data_ptr() and a["slash_indices"] == si.data_ptr()
    assert a["dev_error"] == err.data_ptr() and a["stream"] == STREAM
    size = lib.last("pkv_minference_workspace_size")
    assert list(size.values()) == [300, 8, 2, 40, 90, 0.0, 3, 5]


def test_get_device_error(lib, monkeypatch):
    err = torch.zeros(1, dtype=I32)
    assert pkv.get_device_error(err, clear=True) == 0
    a = lib.last("pkv_get_device_error")
    assert a["dev_error"] == err.data_ptr() and a["clear"] == 1 and a["stream"] == STREAM
    assert isinstance(a["bits"], int) and a["bits"] != 0  # a host int32 the call fills


def test_every_wrapped_entry_point_is_covered_here():
    src = open(os.path.abspath(__file__)).read()
    for name in ("pkv_reshape_and_cache", "pkv_paged_decode", "pkv_paged_decode_noalloc",
                 "pkv_varlen_prefill", "pkv_varlen_prefill_contiguous", "pkv_rope_cos_sin_table",
                 "pkv_rope_reshape_and_cache", "pkv_minference_prefill",
                 "pkv_get_device_error"):
        assert f'lib.last("{name}")' in src
