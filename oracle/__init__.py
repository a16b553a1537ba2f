"""fp64 CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package imports
nothing from the product path.

The arithmetic lives in ``pkv_oracle.c`` (plain loops in double precision);
this module compiles it with gcc and marshals numpy arrays through ctypes.
bf16 tensors travel as their raw 16-bit patterns (``numpy.uint16``).

Definitions followed (page title, section):
  * sink_attention_reference.py (FlashInfer tests): ``sink_softmax`` and the
    varlen / incremental branches of ``sink_attention_unified``;
  * vLLM ``attention.py``: ``PagedAttention.head_mapping`` (GQA) and the
    ``reshape_and_cache`` step of ``PagedAttention.forward``;
  * transformers docs "paged_attention": the varlen worked example
    (cu_seq_lens) and the decode worked example (block_table, cache_seqlens).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F32 = 0
BF16 = 1

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, no fast-math) and return the path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PKV_ORACLE_LIB lets the mutation test load a deliberately broken
            # copy of the oracle and check that the pins reject it.
            override = os.environ.get("PKV_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_token_to_request.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
            lib.oracle_token_to_request.restype = ctypes.c_int
            lib.oracle_slot.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.oracle_slot.restype = i64
            lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, ctypes.c_int, i64]
            lib.oracle_reshape_and_cache.restype = None
            lib.oracle_attention.argtypes = [
                P, P, P, ctypes.c_int, P, P, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, P, ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, P, P,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, P, ctypes.c_int, ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_rope.argtypes = [P, P, ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, P,
                                        ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_int]
            lib.oracle_rope.restype = None
            lib.oracle_minference_scores.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_double]
            lib.oracle_minference_scores.restype = None
            lib.oracle_sparse_attention.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                                    ctypes.c_int, P, ctypes.c_int, ctypes.c_double]
            lib.oracle_sparse_attention.restype = None
            lib.oracle_online_cores.argtypes = []
            lib.oracle_online_cores.restype = ctypes.c_int
            _ = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or uint16 (bf16 bits), got {a.dtype}")


def online_cores() -> int:
    return int(_load().oracle_online_cores())


def token_to_request(cu_seq_lens, total: int) -> np.ndarray:
    """Request index of every token, from cumulative sequence lengths."""
    cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
    out = np.empty(total, dtype=np.int32)
    rc = _load().oracle_token_to_request(_ptr(cu), len(cu) - 1, total, _ptr(out))
    if rc != 0:
        raise ValueError("cu_seq_lens does not cover every token")
    return out


def slot(block_table, b: int, pos: int, block_size: int) -> int:
    """Flat cache slot of logical position ``pos`` of sequence ``b``."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    return int(_load().oracle_slot(_ptr(bt), bt.shape[1], b, pos, block_size))


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping) -> None:
    """In place: k_cache/v_cache rows at slot_mapping[t] <- key/value row t.

    key/value: [T, Hkv, D]; caches: [num_blocks, block_size, Hkv, D]
    (any dtype; rows are copied as bytes).  slot < 0 skips the token.
    """
    assert key.flags.c_contiguous and value.flags.c_contiguous
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = key.shape[0]
    row_bytes = key.dtype.itemsize * int(np.prod(key.shape[1:]))
    cap = k_cache.shape[0] * k_cache.shape[1]
    if np.any(sm >= cap):
        raise ValueError("slot out of the pool")
    _load().oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(sm), T, row_bytes)


def attention(q, k_cache, v_cache, block_table, cu_seq_lens_q, kv_lens, sink=None,
              causal: bool = True, window_left: int = -1, sm_scale: float = 1.0,
              rows=None, threads: int = 0, with_lse: bool = False, alibi_slopes=None):
    """Paged attention of every query row (or of ``rows``) in fp64.

    q: [total_q, Hq, D]; caches: [num_blocks, block_size, Hkv, D] (NHD pages);
    block_table: [batch, max_blocks_per_seq] int32; cu_seq_lens_q: [batch+1];
    kv_lens: [batch]; sink: [Hq] float32 or None (no sink); alibi_slopes: [Hq]
    float32 or None (no ALiBi bias).
    Returns out [nrows, Hq, D] float64 (and lse [nrows, Hq] if with_lse).
    """
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    qd, kd = _dtype_code(q), _dtype_code(k_cache)
    if _dtype_code(v_cache) != kd:
        raise TypeError("k_cache and v_cache dtypes differ")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seq_lens_q, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    batch = len(cu) - 1
    total_q, Hq, D = q.shape
    num_blocks, block_size, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim mismatch")
    sk = None if sink is None else np.ascontiguousarray(sink, dtype=np.float32)
    al = None if alibi_slopes is None else np.ascontiguousarray(alibi_slopes, dtype=np.float32)
    if al is not None and al.shape != (Hq,):
        raise ValueError("alibi_slopes must have num_qo_heads entries")
    if rows is None:
        rw = None
        nrows = int(cu[-1]) if batch > 0 else 0
    else:
        rw = np.ascontiguousarray(rows, dtype=np.int32)
        nrows = len(rw)
    out = np.zeros((nrows, Hq, D), dtype=np.float64)
    lse = np.zeros((nrows, Hq), dtype=np.float64) if with_lse else None
    rc = _load().oracle_attention(
        _ptr(out), _ptr(lse), _ptr(q), qd, _ptr(k_cache), _ptr(v_cache), kd, num_blocks,
        block_size, Hkv, D, _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0, _ptr(cu), _ptr(kl),
        batch, Hq, _ptr(sk), _ptr(al), int(bool(causal)), int(window_left), float(sm_scale), _ptr(rw),
        nrows, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with code {rc}")
    return (out, lse) if with_lse else out


def rope(x, positions, rotary_dim: int, base: float = 10000.0, position_scale: float = 1.0,
         neox: bool = True, ntk_alpha: float = 1.0) -> np.ndarray:
    """Rotary position embedding of x [T, H, D] (float32, or uint16 bf16 bits)
    at positions [T]; returns float64 [T, H, D].  Dimensions past rotary_dim
    are copied.  position_scale divides the positions (linear scaling);
    ntk_alpha != 1 raises the base for NTK-aware scaling (vLLM attention.py,
    PagedAttentionWithRoPE's "dynamic" rope_scaling, read as NTK)."""
    if ntk_alpha != 1.0 and not (ntk_alpha > 0 and rotary_dim > 2):
        raise ValueError("rope: ntk_alpha > 0 and rotary_dim > 2")
    x = np.ascontiguousarray(x)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    T, H, D = x.shape
    if pos.shape != (T,) or rotary_dim % 2 or not 0 < rotary_dim <= D:
        raise ValueError("rope: positions must be [T]; rotary_dim even, 0 < rotary_dim <= D")
    out = np.empty((T, H, D), dtype=np.float64)
    _load().oracle_rope(_ptr(out), _ptr(x), _dtype_code(x), T, H, D, _ptr(pos), int(rotary_dim),
                        float(base), float(position_scale), float(ntk_alpha), int(bool(neox)))
    return out


def paged_decode(q, k_cache, v_cache, block_table, cache_seqlens, sink=None,
                 window_left: int = -1, sm_scale: float = 1.0, rows=None, threads: int = 0,
                 with_lse: bool = False, alibi_slopes=None):
    """Single-token decode: one query per sequence at position cache_seqlens[b]-1."""
    B = q.shape[0]
    cu = np.arange(B + 1, dtype=np.int32)
    return attention(q, k_cache, v_cache, block_table, cu, cache_seqlens, sink=sink,
                     causal=True, window_left=window_left, sm_scale=sm_scale, rows=rows,
                     threads=threads, with_lse=with_lse, alibi_slopes=alibi_slopes)


# ---------------------------------------------------------------------------
# MInference vertical + slash sparse prefill (nano-vllm minference.py)
# ---------------------------------------------------------------------------

def minference_sizes(seq_len: int, vertical_size: int = 1000, slash_size: int = 6096,
                     adaptive_budget=0.3, num_sink_tokens: int = 30,
                     num_recent_diags: int = 100):
    """Numbers of vertical and slash indices kept (MInferencePolicy
    .estimate_pattern): with an adaptive budget b = int(S * budget) they are
    max(num_sink + 1, int(0.2 b)) and max(num_recent + 1, int(0.8 b)); both
    are capped at S."""
    if adaptive_budget is not None:
        budget = int(seq_len * adaptive_budget)
        vertical_size = max(num_sink_tokens + 1, int(budget * 0.2))
        slash_size = max(num_recent_diags + 1, int(budget * 0.8))
    return min(vertical_size, seq_len), min(slash_size, seq_len)


def minference_scores(q, k, last_q: int = 64, scale=None):
    """(vertical [Hq, S], slash [Hq, S]) fp64 pattern scores of the last
    min(last_q, S) queries (see oracle_minference_scores)."""
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    lq = min(last_q, S)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    vert = np.zeros((Hq, S), np.float64)
    sl = np.zeros((Hq, S), np.float64)
    _load().oracle_minference_scores(_ptr(vert), _ptr(sl), _ptr(q), _ptr(k), _dtype_code(q), S,
                                     Hq, Hkv, D, lq, sc)
    return vert, sl


def topk_sorted(scores, k: int, n_force: int):
    """The page's selection: the first n_force entries forced to +inf, the k
    largest kept (equal values: lower index first), returned in ascending
    index order.  scores: [H, S]; returns int32 [H, k]."""
    sc = np.array(scores, np.float64, copy=True)
    sc[:, :n_force] = np.inf
    H, S = sc.shape
    out = np.empty((H, k), np.int32)
    for h in range(H):
        order = np.lexsort((np.arange(S), -sc[h]))  # by value descending, then index
        out[h] = np.sort(order[:k])
    return out


def minference_pattern(q, k, last_q: int = 64, scale=None, vertical_size: int = 1000,
                       slash_size: int = 6096, adaptive_budget=0.3, num_sink_tokens: int = 30,
                       num_recent_diags: int = 100):
    """(vertical_indices [Hq, nv], slash_indices [Hq, ns], vertical_scores,
    slash_scores): the estimate_pattern steps in fp64."""
    S = q.shape[0]
    nv, ns = minference_sizes(S, vertical_size, slash_size, adaptive_budget, num_sink_tokens,
                              num_recent_diags)
    vsc, ssc = minference_scores(q, k, last_q, scale)
    return (topk_sorted(vsc, nv, num_sink_tokens), topk_sorted(ssc, ns, num_recent_diags),
            vsc, ssc)


def sparse_attention(q, k, v, vertical_indices, slash_indices, scale=None):
    """Vertical + slash sparse causal attention of one sequence, fp64
    [S, Hq, D] (see oracle_sparse_attention)."""
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    S, Hq, D = q.shape
    Hkv = k.shape[1]
    vi = np.ascontiguousarray(vertical_indices, dtype=np.int32)
    si = np.ascontiguousarray(slash_indices, dtype=np.int32)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    out = np.zeros((S, Hq, D), np.float64)
    _load().oracle_sparse_attention(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _dtype_code(q), S, Hq,
                                    Hkv, D, _ptr(vi), vi.shape[1], _ptr(si), si.shape[1], sc)
    return out
