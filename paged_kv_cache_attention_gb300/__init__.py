"""Paged KV-cache attention for GB300 (sm_103a): Python binding of libpkv.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``libpkv.so`` (built from ``csrc/`` by ``build()``); this module
checks shapes and dtypes, takes raw device pointers from torch tensors and
the current torch stream, and calls the C ABI declared in ``include/pkv.h``.
There is no CPU or PyTorch fallback: if the library is missing or a call
fails, an exception is raised.

Operations (same names as the C ABI):
  * ``reshape_and_cache`` -- write new K/V rows into the paged pools at
    ``slot_mapping`` (vLLM attention.py, PagedAttention.forward);
  * ``rope_reshape_and_cache`` -- the rotary embedding of q and k by position
    (neox or GPT-J pairing, partial rotary_dim, scaled tables from
    ``rope_cos_sin_table``) fused with that write (vLLM attention.py,
    PagedAttentionWithRoPE);
  * ``paged_decode`` (and ``paged_decode_noalloc``, which needs no workspace)
    -- one query per sequence over its pages through ``block_table`` /
    ``cache_seqlens`` (transformers docs "paged_attention", decode path),
    split-KV with 512-token partitions;
  * ``varlen_prefill`` -- varlen / chunk prefill addressed by
    ``cu_seq_lens_q`` / ``cu_seq_lens_k`` (transformers docs
    "paged_attention", varlen path), keys read from the pages, causal or not;
    ``varlen_prefill_contiguous`` reads them from [total_k, Hkv, D] arrays;
  * ``minference_prefill`` -- MInference's vertical + slash sparse prefill of
    one sequence (nano-vllm minference.py): pattern estimate, top-k, then
    attention over the kept keys.
The attention calls support GQA, ``window_left``, the per-head attention sink
of FlashInfer's sink_attention_reference.py, ALiBi slopes, head sizes 64, 80,
96, 112, 128 and 256, and NHD or HND page layouts.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from ._build import LIB_PATH, build as _build_lib

__all__ = [
    "build", "load_library", "PkvError", "reshape_and_cache", "paged_decode",
    "varlen_prefill", "varlen_prefill_contiguous", "paged_decode_noalloc",
    "paged_decode_workspace_size", "varlen_prefill_workspace_size",
    "rope_cos_sin_table", "rope_reshape_and_cache", "get_device_error",
    "selftest_bounded_wait",
    "minference_sizes", "minference_prefill",
    "DEVERR_BLOCK_ID", "DEVERR_SLOT", "DEVERR_SEQLEN", "DEVERR_TIMEOUT", "DEVERR_POSITION",
    "EXPORTED_SYMBOLS",
]

PKV_F32 = 0
PKV_BF16 = 1
DEVERR_BLOCK_ID = 1
DEVERR_SLOT = 2
DEVERR_SEQLEN = 4
DEVERR_TIMEOUT = 8
DEVERR_POSITION = 16

EXPORTED_SYMBOLS = (
    "pkv_status_string", "pkv_version", "pkv_reshape_and_cache",
    "pkv_paged_decode_workspace_size", "pkv_paged_decode",
    "pkv_varlen_prefill_workspace_size", "pkv_varlen_prefill",
    "pkv_varlen_prefill_contiguous", "pkv_rope_cos_sin_table", "pkv_rope_reshape_and_cache",
    "pkv_minference_sizes", "pkv_minference_workspace_size", "pkv_minference_prefill",
    "pkv_paged_decode_noalloc", "pkv_get_device_error", "pkv_selftest_bounded_wait",
)


class PkvError(RuntimeError):
    """A libpkv call returned a non-OK status."""

    def __init__(self, fn: str, status: int, name: str):
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status
        self.status_name = name


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32)]


LAYOUTS = {"NHD": 0, "HND": 1}


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile libpkv.so for sm_103a (in-tree)."""
    return _build_lib(force=force)


def load_library(path: Optional[str] = None):
    """Load libpkv.so (building it first if it is absent) and declare the ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            p = _build_lib()
        lib = ctypes.CDLL(p)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        lib.pkv_status_string.argtypes = [i32]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = i32
        lib.pkv_reshape_and_cache.argtypes = [P, P, P, P, P, i64, CacheDesc, P, P]
        lib.pkv_reshape_and_cache.restype = i32
        lib.pkv_paged_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.pkv_paged_decode_workspace_size.restype = sz
        lib.pkv_paged_decode.argtypes = [P, P, P, P, CacheDesc, P, i32, P, i32, P, P, i32, i32,
                                         i32, f32, i32, P, P, sz, P, P]
        lib.pkv_paged_decode.restype = i32
        lib.pkv_varlen_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.pkv_varlen_prefill_workspace_size.restype = sz
        lib.pkv_varlen_prefill.argtypes = [P, P, P, P, CacheDesc, P, i32, P, P, i32, i32, i32, P,
                                           P, i32, i32, i32, i32, f32, P, P, sz, i32, P, P]
        lib.pkv_varlen_prefill.restype = i32
        lib.pkv_varlen_prefill_contiguous.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, i32,
                                                      i32, i32, P, P, i32, i32, i32, i32, f32, P,
                                                      P, sz, P, P]
        lib.pkv_varlen_prefill_contiguous.restype = i32
        f64 = ctypes.c_double
        lib.pkv_rope_cos_sin_table.argtypes = [P, i32, i32, f64, f64, f64, P]
        lib.pkv_rope_cos_sin_table.restype = i32
        lib.pkv_rope_reshape_and_cache.argtypes = [P, P, P, P, P, P, P, i64, i32, CacheDesc, P,
                                                   i32, i32, i32, P, P]
        lib.pkv_rope_reshape_and_cache.restype = i32
        lib.pkv_minference_sizes.argtypes = [i32, i32, i32, f64, i32, i32, P, P]
        lib.pkv_minference_sizes.restype = i32
        lib.pkv_minference_workspace_size.argtypes = [i32, i32, i32, i32, i32, f64, i32, i32]
        lib.pkv_minference_workspace_size.restype = sz
        lib.pkv_minference_prefill.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, f64,
                                               i32, i32, f32, P, P, P, sz, P, P]
        lib.pkv_minference_prefill.restype = i32
        lib.pkv_paged_decode_noalloc.argtypes = [P, P, P, P, CacheDesc, P, i32, P, i32, P, i32,
                                                 i32, i32, f32, i32, P, P, P]
        lib.pkv_paged_decode_noalloc.restype = i32
        lib.pkv_get_device_error.argtypes = [P, P, i32, P]
        lib.pkv_get_device_error.restype = i32
        lib.pkv_selftest_bounded_wait.argtypes = [P, P]
        lib.pkv_selftest_bounded_wait.restype = i32
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _check(fn: str, status: int):
    if status != 0:
        name = load_library().pkv_status_string(status).decode()
        raise PkvError(fn, status, name)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(dtype) -> int:
    torch = _torch()
    if dtype == torch.float32:
        return PKV_F32
    if dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {dtype}: use torch.bfloat16 or torch.float32")


def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(name, t, dtype=None, ndim=None):
    _require(t.is_cuda, f"{name} must be a CUDA tensor")
    _require(t.is_contiguous(), f"{name} must be contiguous")
    if dtype is not None:
        _require(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None:
        _require(t.dim() == ndim, f"{name} must have {ndim} dims, got {t.dim()}")


def _pool_dims(k_cache, layout: str):
    """(num_blocks, block_size, num_kv_heads, head_dim) of a pool: NHD pools
    are [num_blocks, block_size, Hkv, D], HND pools [num_blocks, Hkv,
    block_size, D]."""
    _require(layout in LAYOUTS, f"layout must be one of {sorted(LAYOUTS)}")
    nb, a, b, d = k_cache.shape
    return (nb, a, b, d) if layout == "NHD" else (nb, b, a, d)


def _cache_desc(k_cache, v_cache, layout: str = "NHD") -> CacheDesc:
    _cuda_contig("k_cache", k_cache, ndim=4)
    _cuda_contig("v_cache", v_cache, ndim=4)
    _require(k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype,
             "k_cache and v_cache must have the same shape and dtype")
    nb, bs, hkv, d = _pool_dims(k_cache, layout)
    return CacheDesc(nb, bs, hkv, d, _dtype_code(k_cache.dtype), LAYOUTS[layout])


def _head_vector(name, t, Hq):
    if t is not None:
        _cuda_contig(name, t, _torch().float32, 1)
        _require(t.shape[0] == Hq, f"{name} must have num_qo_heads entries")


def paged_decode_workspace_size(batch: int, num_qo_heads: int, head_dim: int, max_seqlen: int,
                                partition_size: int = 512, window_left: int = -1) -> int:
    return int(load_library().pkv_paged_decode_workspace_size(
        batch, num_qo_heads, head_dim, max_seqlen, partition_size, window_left))


def varlen_prefill_workspace_size(batch: int, num_qo_heads: int, num_kv_heads: int,
                                  total_q: int, max_seqlen_q: int) -> int:
    return int(load_library().pkv_varlen_prefill_workspace_size(
        batch, num_qo_heads, num_kv_heads, total_q, max_seqlen_q))


def _workspace(nbytes: int, device, workspace):
    torch = _torch()
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    _cuda_contig("workspace", workspace)
    _require(workspace.numel() * workspace.element_size() >= nbytes,
             f"workspace too small: need {nbytes} bytes")
    return workspace


# ---------------------------------------------------------------------------
# public operations
# ---------------------------------------------------------------------------

def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, dev_error=None,
                      stream=None, layout: str = "NHD") -> None:
    """k_cache/v_cache flat slot slot_mapping[t] <- key/value[t] (in place).

    key, value: [T, Hkv, D] contiguous, dtype of the cache; slot_mapping: [T]
    int64, negative = skip.  dev_error: optional int32 device tensor that
    receives PKV_DEVERR_SLOT for slots outside the pool.
    """
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache, layout)
    _cuda_contig("key", key, k_cache.dtype, 3)
    _cuda_contig("value", value, k_cache.dtype, 3)
    _cuda_contig("slot_mapping", slot_mapping, torch.int64, 1)
    _require(key.shape == value.shape and key.shape[1:] == (desc.num_kv_heads, desc.head_dim),
             "key/value must be [T, num_kv_heads, head_dim] matching the cache")
    _require(slot_mapping.shape[0] == key.shape[0], "slot_mapping must have T entries")
    st = load_library().pkv_reshape_and_cache(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
        key.shape[0], desc, _ptr(dev_error), _stream_handle(stream))
    _check("pkv_reshape_and_cache", st)


def get_device_error(dev_error, clear: bool = False, stream=None, raise_on_error: bool = False):
    """The PKV_DEVERR_* bits the calls so far ORed into ``dev_error`` (an int32
    device tensor of one element).  Waits for ``stream`` (the current one by
    default); with ``clear`` the word is then zeroed on that stream.  With
    ``raise_on_error`` a set bit raises PkvError (PKV_ERR_OUT_OF_RANGE, or
    PKV_ERR_TIMEOUT for a pipeline wait that gave up)."""
    torch = _torch()
    _cuda_contig("dev_error", dev_error, torch.int32, 1)
    bits = ctypes.c_int32(0)
    st = load_library().pkv_get_device_error(_ptr(dev_error), ctypes.addressof(bits),
                                             int(bool(clear)), _stream_handle(stream))
    if st != 0 and (raise_on_error or st not in (5, 6)):
        _check("pkv_get_device_error", st)
    return int(bits.value)


def selftest_bounded_wait(dev_error, stream=None):
    """Run one bounded pipeline wait that nothing completes on ``stream``: it
    gives up by itself and ORs DEVERR_TIMEOUT into ``dev_error`` (an int32
    device tensor of one element); see get_device_error."""
    _cuda_contig("dev_error", dev_error, _torch().int32, 1)
    _check("pkv_selftest_bounded_wait",
           load_library().pkv_selftest_bounded_wait(_ptr(dev_error), _stream_handle(stream)))


def rope_cos_sin_table(max_position: int, rotary_dim: int, base: float = 10000.0,
                       position_scale: float = 1.0, ntk_alpha: float = 1.0, device=None,
                       stream=None):
    """The rotary table [max_position, rotary_dim // 2, 2] float32 of
    (cos, sin) of (pos / position_scale) * b^(-2i / rotary_dim), computed in
    fp64 on the GPU, b = base * ntk_alpha^(rotary_dim / (rotary_dim - 2)).
    position_scale is the linear scaling factor, ntk_alpha the NTK-aware
    context stretch (1: none)."""
    torch = _torch()
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    tab = torch.empty(max(max_position, 0), rotary_dim // 2, 2, dtype=torch.float32, device=dev)
    st = load_library().pkv_rope_cos_sin_table(_ptr(tab) if tab.numel() else None,
                                               int(max_position), int(rotary_dim), float(base),
                                               float(position_scale), float(ntk_alpha),
                                               _stream_handle(stream))
    _check("pkv_rope_cos_sin_table", st)
    return tab


def rope_reshape_and_cache(query, key, value, k_cache, v_cache, positions, slot_mapping,
                           cos_sin, rotary_dim: Optional[int] = None, is_neox_style: bool = True,
                           dev_error=None, stream=None, layout: str = "NHD") -> None:
    """Rotate query [T, Hq, D] and key [T, Hkv, D] in place by positions [T]
    (int64) using the table cos_sin ([max_position, rotary_dim // 2, 2]), then
    write the rotated key and the value to the pools at slot_mapping [T]
    (int64; negative = not cached).  query may be None."""
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache, layout)
    _cuda_contig("key", key, k_cache.dtype, 3)
    _cuda_contig("value", value, k_cache.dtype, 3)
    _cuda_contig("positions", positions, torch.int64, 1)
    _cuda_contig("slot_mapping", slot_mapping, torch.int64, 1)
    _cuda_contig("cos_sin", cos_sin, torch.float32, 3)
    T = key.shape[0]
    _require(key.shape == value.shape and key.shape[1:] == (desc.num_kv_heads, desc.head_dim),
             "key/value must be [T, num_kv_heads, head_dim] matching the cache")
    _require(positions.shape[0] == T and slot_mapping.shape[0] == T,
             "positions and slot_mapping must have T entries")
    rd = int(rotary_dim) if rotary_dim is not None else 2 * cos_sin.shape[1]
    _require(cos_sin.shape[1] * 2 == rd and cos_sin.shape[2] == 2,
             "cos_sin must be [max_position, rotary_dim // 2, 2]")
    Hq = 0
    if query is not None:
        _cuda_contig("query", query, k_cache.dtype, 3)
        _require(query.shape[0] == T and query.shape[2] == key.shape[2],
                 "query must be [T, num_qo_heads, head_dim]")
        Hq = query.shape[1]
    st = load_library().pkv_rope_reshape_and_cache(
        _ptr(query), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(positions),
        _ptr(slot_mapping), T, Hq, desc, _ptr(cos_sin), cos_sin.shape[0], rd,
        int(bool(is_neox_style)), _ptr(dev_error), _stream_handle(stream))
    _check("pkv_rope_reshape_and_cache", st)


def _decode_args(q, k_cache, v_cache, block_table, cache_seqlens, sink, out, lse, layout):
    """Checks shared by the two decode entry points; returns (cache desc, out)."""
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache, layout)
    _cuda_contig("q", q, k_cache.dtype, 3)
    _cuda_contig("block_table", block_table, torch.int32, 2)
    _cuda_contig("cache_seqlens", cache_seqlens, torch.int32, 1)
    B, Hq, D = q.shape
    _require(D == desc.head_dim, "head_dim of q and cache differ")
    _require(block_table.shape[0] == B and cache_seqlens.shape[0] == B,
             "block_table / cache_seqlens batch mismatch")
    if sink is not None:
        _cuda_contig("sink", sink, torch.float32, 1)
        _require(sink.shape[0] == Hq, "sink must have num_qo_heads entries")
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_contig("out", out, q.dtype, 3)
        _require(out.shape == q.shape, "out must be shaped like q")
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32, 2)
        _require(tuple(lse.shape) == (B, Hq), "lse must be [B, Hq]")
    return desc, out


def paged_decode(q, k_cache, v_cache, block_table, cache_seqlens, max_seqlen: int,
                 sink=None, window_left: int = -1, sm_scale: Optional[float] = None,
                 partition_size: int = 512, out=None, lse=None, workspace=None,
                 dev_error=None, stream=None, alibi_slopes=None, layout: str = "NHD"):
    """Single-token decode over the paged pools; returns out [B, Hq, D].

    q: [B, Hq, D] (dtype of the cache); block_table: [B, max_blocks] int32;
    cache_seqlens: [B] int32, the attended length (query at position L-1);
    max_seqlen: host int >= max(cache_seqlens); sink: [Hq] float32 or None;
    lse: optional [B, Hq] float32 output (natural log, sink included);
    alibi_slopes: [Hq] float32 or None (bias slope * (j - (L - 1)));
    layout: "NHD" pools [num_blocks, block_size, Hkv, D] or "HND" pools
    [num_blocks, Hkv, block_size, D].
    """
    torch = _torch()
    desc, out = _decode_args(q, k_cache, v_cache, block_table, cache_seqlens, sink, out, lse,
                             layout)
    B, Hq, D = q.shape
    _head_vector("alibi_slopes", alibi_slopes, Hq)
    scale = float(sm_scale) if sm_scale is not None else D ** -0.5
    need = paged_decode_workspace_size(B, Hq, D, max_seqlen, partition_size, window_left)
    ws = _workspace(need, q.device, workspace)
    st = load_library().pkv_paged_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), desc, _ptr(block_table),
        block_table.shape[1], _ptr(cache_seqlens), int(max_seqlen), _ptr(sink),
        _ptr(alibi_slopes), B, Hq, int(window_left), scale, int(partition_size), _ptr(lse),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_error), _stream_handle(stream))
    _check("pkv_paged_decode", st)
    return out


def varlen_prefill(q, k_cache, v_cache, block_table, cu_seq_lens_q, cu_seq_lens_k,
                   max_seqlen_q: int, max_seqlen_k: int, sink=None, causal: bool = True,
                   window_left: int = -1, sm_scale: Optional[float] = None, out=None, lse=None,
                   workspace=None, dev_error=None, stream=None, alibi_slopes=None,
                   layout: str = "NHD", max_ctas: int = 0):
    """Varlen / chunk prefill over the paged pools; returns out [total_q, Hq, D].

    q: [total_q, Hq, D] bf16; cu_seq_lens_q / cu_seq_lens_k: [B+1] int32;
    max_seqlen_q / max_seqlen_k: host ints; request r's queries sit at the end
    of its kv_len keys.  causal=False drops the j <= position bound (a window
    still bounds keys from below).  max_ctas: at most this many attention
    CTAs (one SM each) at once, 0 = one per SM; fewer leave SMs free for
    work on another stream.
    """
    torch = _torch()
    desc = _cache_desc(k_cache, v_cache, layout)
    _cuda_contig("q", q, k_cache.dtype, 3)
    _cuda_contig("block_table", block_table, torch.int32, 2)
    _cuda_contig("cu_seq_lens_q", cu_seq_lens_q, torch.int32, 1)
    _cuda_contig("cu_seq_lens_k", cu_seq_lens_k, torch.int32, 1)
    total_q, Hq, D = q.shape
    B = cu_seq_lens_q.shape[0] - 1
    _require(cu_seq_lens_k.shape[0] == B + 1, "cu_seq_lens_q/k lengths differ")
    _require(block_table.shape[0] == B, "block_table must have one row per request")
    if sink is not None:
        _cuda_contig("sink", sink, torch.float32, 1)
        _require(sink.shape[0] == Hq, "sink must have num_qo_heads entries")
    _head_vector("alibi_slopes", alibi_slopes, Hq)
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_contig("out", out, q.dtype, 3)
        _require(out.shape == q.shape, "out must be shaped like q")
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32, 2)
        _require(tuple(lse.shape) == (total_q, Hq), "lse must be [total_q, Hq]")
    scale = float(sm_scale) if sm_scale is not None else D ** -0.5
    need = varlen_prefill_workspace_size(B, Hq, desc.num_kv_heads, total_q, max_seqlen_q)
    ws = _workspace(need, q.device, workspace)
    st = load_library().pkv_varlen_prefill(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), desc, _ptr(block_table),
        block_table.shape[1], _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k), int(max_seqlen_q),
        int(max_seqlen_k), int(total_q), _ptr(sink), _ptr(alibi_slopes), B, Hq,
        int(bool(causal)), int(window_left), scale, _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), int(max_ctas), _ptr(dev_error), _stream_handle(stream))
    _check("pkv_varlen_prefill", st)
    return out


def varlen_prefill_contiguous(q, k, v, cu_seq_lens_q, cu_seq_lens_k, max_seqlen_q: int,
                              max_seqlen_k: int, sink=None, causal: bool = True,
                              window_left: int = -1, sm_scale: Optional[float] = None, out=None,
                              lse=None, workspace=None, dev_error=None, stream=None,
                              alibi_slopes=None):
    """Varlen prefill with contiguous keys: request r's keys and values are
    rows cu_seq_lens_k[r] .. cu_seq_lens_k[r+1]-1 of k and v ([total_k, Hkv, D]
    bf16).  Otherwise as varlen_prefill; returns out [total_q, Hq, D]."""
    torch = _torch()
    _cuda_contig("q", q, ndim=3)
    _cuda_contig("k", k, q.dtype, 3)
    _cuda_contig("v", v, q.dtype, 3)
    _cuda_contig("cu_seq_lens_q", cu_seq_lens_q, torch.int32, 1)
    _cuda_contig("cu_seq_lens_k", cu_seq_lens_k, torch.int32, 1)
    _require(k.shape == v.shape, "k and v must have the same shape")
    total_q, Hq, D = q.shape
    total_k, Hkv, Dk = k.shape
    _require(Dk == D, "head_dim of q and k differ")
    B = cu_seq_lens_q.shape[0] - 1
    _require(cu_seq_lens_k.shape[0] == B + 1, "cu_seq_lens_q/k lengths differ")
    if sink is not None:
        _cuda_contig("sink", sink, torch.float32, 1)
        _require(sink.shape[0] == Hq, "sink must have num_qo_heads entries")
    _head_vector("alibi_slopes", alibi_slopes, Hq)
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_contig("out", out, q.dtype, 3)
        _require(out.shape == q.shape, "out must be shaped like q")
    if lse is not None:
        _cuda_contig("lse", lse, torch.float32, 2)
        _require(tuple(lse.shape) == (total_q, Hq), "lse must be [total_q, Hq]")
    scale = float(sm_scale) if sm_scale is not None else D ** -0.5
    need = varlen_prefill_workspace_size(B, Hq, Hkv, total_q, max_seqlen_q)
    ws = _workspace(need, q.device, workspace)
    st = load_library().pkv_varlen_prefill_contiguous(
        _ptr(out), _ptr(q), _ptr(k) if total_k else None, _ptr(v) if total_k else None,
        int(total_k), Hkv, D, _dtype_code(q.dtype), _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k),
        int(max_seqlen_q), int(max_seqlen_k), int(total_q), _ptr(sink), _ptr(alibi_slopes), B,
        Hq, int(bool(causal)), int(window_left), scale, _ptr(lse), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(dev_error), _stream_handle(stream))
    _check("pkv_varlen_prefill_contiguous", st)
    return out


def minference_sizes(seq_len: int, vertical_size: int = 1000, slash_size: int = 6096,
                     adaptive_budget: Optional[float] = 0.3, num_sink_tokens: int = 30,
                     num_recent_diags: int = 100):
    """(nv, ns): how many vertical columns and slash diagonals are kept."""
    nv, ns = ctypes.c_int(), ctypes.c_int()
    st = load_library().pkv_minference_sizes(
        int(seq_len), int(vertical_size), int(slash_size),
        float(adaptive_budget) if adaptive_budget is not None else 0.0, int(num_sink_tokens),
        int(num_recent_diags), ctypes.byref(nv), ctypes.byref(ns))
    _check("pkv_minference_sizes", st)
    return nv.value, ns.value


def lib_minference_workspace(seq_len: int, num_qo_heads: int, num_kv_heads: int,
                             vertical_size: int = 1000, slash_size: int = 6096,
                             adaptive_budget: Optional[float] = 0.3, num_sink_tokens: int = 30,
                             num_recent_diags: int = 100) -> int:
    """Workspace bytes minference_prefill needs."""
    return int(load_library().pkv_minference_workspace_size(
        int(seq_len), int(num_qo_heads), int(num_kv_heads), int(vertical_size), int(slash_size),
        float(adaptive_budget) if adaptive_budget is not None else 0.0, int(num_sink_tokens),
        int(num_recent_diags)))


def minference_prefill(q, k, v, vertical_size: int = 1000, slash_size: int = 6096,
                       adaptive_budget: Optional[float] = 0.3, num_sink_tokens: int = 30,
                       num_recent_diags: int = 100, sm_scale: Optional[float] = None, out=None,
                       return_pattern: bool = False, workspace=None, dev_error=None,
                       stream=None):
    """MInference vertical + slash sparse prefill of one sequence: q [S, Hq, D],
    k, v [S, Hkv, D] bf16.  Returns out [S, Hq, D] (and, with
    return_pattern, the kept vertical [Hq, nv] and slash [Hq, ns] indices)."""
    torch = _torch()
    _cuda_contig("q", q, torch.bfloat16, 3)
    _cuda_contig("k", k, torch.bfloat16, 3)
    _cuda_contig("v", v, torch.bfloat16, 3)
    S, Hq, D = q.shape
    _require(k.shape == v.shape and k.shape[0] == S and k.shape[2] == D,
             "k and v must be [S, num_kv_heads, head_dim] like q")
    Hkv = k.shape[1]
    budget = float(adaptive_budget) if adaptive_budget is not None else 0.0
    nv, ns = minference_sizes(S, vertical_size, slash_size, adaptive_budget, num_sink_tokens,
                              num_recent_diags)
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_contig("out", out, q.dtype, 3)
        _require(out.shape == q.shape, "out must be shaped like q")
    vi = torch.empty(Hq, nv, dtype=torch.int32, device=q.device) if return_pattern else None
    si = torch.empty(Hq, ns, dtype=torch.int32, device=q.device) if return_pattern else None
    need = int(load_library().pkv_minference_workspace_size(
        S, Hq, Hkv, int(vertical_size), int(slash_size), budget, int(num_sink_tokens),
        int(num_recent_diags)))
    ws = _workspace(need, q.device, workspace)
    scale = float(sm_scale) if sm_scale is not None else D ** -0.5
    st = load_library().pkv_minference_prefill(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), S, Hq, Hkv, D, PKV_BF16, int(vertical_size),
        int(slash_size), budget, int(num_sink_tokens), int(num_recent_diags), scale, _ptr(vi),
        _ptr(si), _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_error),
        _stream_handle(stream))
    _check("pkv_minference_prefill", st)
    return (out, vi, si) if return_pattern else out


def paged_decode_noalloc(q, k_cache, v_cache, block_table, cache_seqlens, max_seqlen: int,
                         sink=None, window_left: int = -1, sm_scale: Optional[float] = None,
                         partition_size: int = 512, out=None, lse=None, dev_error=None,
                         stream=None, layout: str = "NHD"):
    """paged_decode without a caller workspace, for callers that cannot
    allocate device memory at the call site.  The library's fixed device
    scratch array (PKV_NOALLOC_DECODE_SCRATCH_BYTES, 32 MiB) replaces the
    workspace; problems that need more are rejected (PkvError
    PKV_ERR_WORKSPACE).  Calls share the array: do not overlap them on the
    GPU.  The first call on a device should come before any stream capture.
    ``out`` (and ``lse``) should be preallocated when the caller must not
    allocate at all."""
    desc, out = _decode_args(q, k_cache, v_cache, block_table, cache_seqlens, sink, out, lse,
                             layout)
    B, Hq, D = q.shape
    scale = float(sm_scale) if sm_scale is not None else D ** -0.5
    st = load_library().pkv_paged_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), desc, _ptr(block_table),
        block_table.shape[1], _ptr(cache_seqlens), int(max_seqlen), _ptr(sink), B, Hq,
        int(window_left), scale, int(partition_size), _ptr(lse), _ptr(dev_error),
        _stream_handle(stream))
    _check("pkv_paged_decode_noalloc", st)
    return out
