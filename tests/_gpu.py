"""Shared plumbing of the GPU parity tests: run a case through the C ABI
(via the binding) and through the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W

# max-abs-error bars on attention outputs
TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-5}
# log-sum-exp (natural log) bars: fp32 logits of bf16 / fp32 inputs
LSE_TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def to_dev(t):
    return None if t is None else t.to(dev())


def to_hnd(pool):
    """An NHD pool [num_blocks, block_size, Hkv, D] as the same pages in the
    HND layout [num_blocks, Hkv, block_size, D] (pure re-indexing)."""
    return pool.permute(0, 2, 1, 3).contiguous()


def from_hnd(pool):
    return pool.permute(0, 2, 1, 3).contiguous()


def _pools(case, layout):
    k, v = case.k_cache, case.v_cache
    if layout == "HND":
        k, v = to_hnd(k), to_hnd(v)
    return to_dev(k), to_dev(v)


def gpu_decode(case, partition_size=None, with_lse=False, err=None, max_seqlen=None,
               layout="NHD"):
    d = dev()
    lse = torch.empty(case.batch, case.num_qo_heads, dtype=torch.float32, device=d) \
        if with_lse else None
    kc, vc = _pools(case, layout)
    out = pkv.paged_decode(to_dev(case.q), kc, vc,
                           to_dev(case.block_table), to_dev(case.cache_seqlens),
                           max_seqlen=case.max_seqlen if max_seqlen is None else max_seqlen,
                           sink=to_dev(case.sink), window_left=case.window_left,
                           sm_scale=case.sm_scale,
                           partition_size=partition_size or case.partition_size, lse=lse,
                           dev_error=err, alibi_slopes=to_dev(case.alibi), layout=layout)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    return (o, lse.cpu().numpy().astype(np.float64)) if with_lse else o


def oracle_decode(case, rows=None, with_lse=False):
    return oracle.paged_decode(
        W.to_oracle(case.q), W.to_oracle(case.k_cache), W.to_oracle(case.v_cache),
        case.block_table.numpy(), case.cache_seqlens.numpy(),
        sink=None if case.sink is None else case.sink.numpy(), window_left=case.window_left,
        sm_scale=case.sm_scale, rows=rows, with_lse=with_lse,
        alibi_slopes=None if case.alibi is None else case.alibi.numpy())


def gpu_prefill(case, with_lse=False, err=None, layout="NHD"):
    d = dev()
    lse = torch.empty(case.total_q, case.q.shape[1], dtype=torch.float32, device=d) \
        if with_lse else None
    kc, vc = _pools(case, layout)
    out = pkv.varlen_prefill(to_dev(case.q), kc, vc,
                             to_dev(case.block_table), to_dev(case.cu_seq_lens_q),
                             to_dev(case.cu_seq_lens_k), case.max_seqlen_q, case.max_seqlen_k,
                             sink=to_dev(case.sink), causal=case.causal,
                             window_left=case.window_left, sm_scale=case.sm_scale, lse=lse,
                             dev_error=err, alibi_slopes=to_dev(case.alibi), layout=layout)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    return (o, lse.cpu().numpy().astype(np.float64)) if with_lse else o


def contiguous_kv(case, pad_rows=0):
    """The case's keys and values packed request after request ([total_k, Hkv,
    D], the layout cu_seq_lens_k addresses), gathered from the pool by plain
    indexing; pad_rows NaN rows follow the last request."""
    bs = case.k_cache.shape[1]
    ks, vs = [], []
    for r, L in enumerate(case.kv_lens.tolist()):
        pos = torch.arange(L)
        pages = case.block_table[r, (pos // bs)].long()
        ks.append(case.k_cache[pages, pos % bs])
        vs.append(case.v_cache[pages, pos % bs])
    tail = torch.full((pad_rows,) + tuple(case.k_cache.shape[2:]), float("nan"),
                      dtype=case.k_cache.dtype)
    return torch.cat(ks + [tail]), torch.cat(vs + [tail])


def gpu_prefill_contiguous(case, k, v, with_lse=False, err=None):
    d = dev()
    lse = torch.empty(case.total_q, case.q.shape[1], dtype=torch.float32, device=d) \
        if with_lse else None
    out = pkv.varlen_prefill_contiguous(
        to_dev(case.q), to_dev(k), to_dev(v), to_dev(case.cu_seq_lens_q),
        to_dev(case.cu_seq_lens_k), case.max_seqlen_q, case.max_seqlen_k,
        sink=to_dev(case.sink), causal=case.causal, window_left=case.window_left,
        sm_scale=case.sm_scale, lse=lse, dev_error=err, alibi_slopes=to_dev(case.alibi))
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    return (o, lse.cpu().numpy().astype(np.float64)) if with_lse else o


def oracle_prefill(case, rows=None, with_lse=False):
    return oracle.attention(
        W.to_oracle(case.q), W.to_oracle(case.k_cache), W.to_oracle(case.v_cache),
        case.block_table.numpy(), case.cu_seq_lens_q.numpy(), case.kv_lens.numpy(),
        sink=None if case.sink is None else case.sink.numpy(), causal=case.causal,
        window_left=case.window_left, sm_scale=case.sm_scale, rows=rows, with_lse=with_lse,
        alibi_slopes=None if case.alibi is None else case.alibi.numpy())


def max_abs(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    if a.size == 0:
        return 0.0
    assert np.isfinite(a).all(), "non-finite values in the GPU output"
    return float(np.abs(a - b).max())


def lse_err(a, b):
    """max |a-b| over entries where both are finite; -inf must match -inf."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb), "finite/-inf pattern of lse differs"
    return float(np.abs(a[fa] - b[fb]).max()) if fa.any() else 0.0
