"""Test helpers: dense per-request K/V laid out into a shuffled page pool, and an
independent brute-force dense attention in numpy.

The brute-force routine is a second, separately written statement of the same
definition (sink_attention_reference.py, FlashInfer tests: sink_softmax and the
varlen branch of sink_attention_unified): it builds the whole mask matrix,
appends the sink as one more softmax column and drops that column after
normalising.  It shares nothing with the C oracle.
"""
from __future__ import annotations

import numpy as np


def paginate(dense_k, dense_v, block_size, rng, spare=3, max_blocks=None):
    """Place per-request dense K/V ([kv_len, Hkv, D] float32 each) into a pool
    of [num_blocks, block_size, Hkv, D] pages in random physical order.
    Unowned pages are NaN.  Returns (k_pool, v_pool, block_table)."""
    n_req = len(dense_k)
    pages = [(k.shape[0] + block_size - 1) // block_size for k in dense_k]
    Hkv, D = dense_k[0].shape[1], dense_k[0].shape[2]
    nb = sum(pages) + spare
    perm = rng.permutation(nb).astype(np.int32)
    mb = max(max(pages) if pages else 1, 1)
    if max_blocks is not None:
        mb = max(mb, max_blocks)
    bt = np.full((n_req, mb), -1, dtype=np.int32)
    kp = np.full((nb, block_size, Hkv, D), np.nan, dtype=np.float32)
    vp = np.full((nb, block_size, Hkv, D), np.nan, dtype=np.float32)
    cur = 0
    for r in range(n_req):
        L = dense_k[r].shape[0]
        for i in range(pages[r]):
            blk = perm[cur]
            cur += 1
            bt[r, i] = blk
            lo, hi = i * block_size, min(L, (i + 1) * block_size)
            kp[blk, : hi - lo] = dense_k[r][lo:hi]
            vp[blk, : hi - lo] = dense_v[r][lo:hi]
    return kp, vp, bt


def brute_force(q_list, k_list, v_list, sink, causal, window_left, sm_scale, alibi=None):
    """Dense fp64 attention per request; returns (out [total_q, Hq, D], lse).
    alibi: [Hq] slopes; the logit of key j for the query at position pos gains
    slope * (j - pos)."""
    outs, lses = [], []
    for q, k, v in zip(q_list, k_list, v_list):
        q = q.astype(np.float64)
        k = k.astype(np.float64)
        v = v.astype(np.float64)
        q_len, Hq, D = q.shape
        kv_len, Hkv, _ = k.shape
        G = Hq // Hkv
        kk = np.repeat(k, G, axis=1)  # [kv, Hq, D]
        vv = np.repeat(v, G, axis=1)
        logits = np.einsum("qhd,khd->hqk", q, kk) * sm_scale  # [Hq, q, kv]
        pos = (kv_len - q_len + np.arange(q_len))[:, None]
        col = np.arange(kv_len)[None, :]
        if alibi is not None:
            logits = logits + np.asarray(alibi, np.float64)[:, None, None] * (col - pos)[None]
        mask = np.ones((q_len, kv_len), dtype=bool)
        if causal:
            mask &= col <= pos
        if window_left >= 0:
            mask &= col >= pos - window_left
        logits = np.where(mask[None], logits, -np.inf)
        s = np.full((Hq, q_len, 1), -np.inf) if sink is None else \
            np.broadcast_to(np.asarray(sink, np.float64)[:, None, None], (Hq, q_len, 1))
        ext = np.concatenate([logits, s], axis=-1)  # [Hq, q, kv+1]
        mx = ext.max(axis=-1, keepdims=True)
        dead = ~np.isfinite(mx)
        mx = np.where(dead, 0.0, mx)
        e = np.exp(ext - mx)
        z = e.sum(axis=-1, keepdims=True)
        zsafe = np.where(z > 0, z, 1.0)
        p = (e / zsafe)[..., :-1]
        o = np.einsum("hqk,khd->qhd", p, vv)
        with np.errstate(divide="ignore"):
            lse = (np.log(z) + mx)[..., 0].T  # [q, Hq]
        lse = np.where(dead[..., 0].T, -np.inf, lse)
        outs.append(o)
        lses.append(lse)
    Hq = q_list[0].shape[1]
    D = q_list[0].shape[2]
    out = np.concatenate(outs, 0) if outs else np.zeros((0, Hq, D))
    lse = np.concatenate(lses, 0) if lses else np.zeros((0, Hq))
    return out, lse


def random_dense(rng, q_lens, kv_lens, Hq, Hkv, D):
    q = [rng.standard_normal((ql, Hq, D)).astype(np.float32) for ql in q_lens]
    k = [rng.standard_normal((kl, Hkv, D)).astype(np.float32) for kl in kv_lens]
    v = [rng.standard_normal((kl, Hkv, D)).astype(np.float32) for kl in kv_lens]
    return q, k, v


def cu(lens):
    out = np.zeros(len(lens) + 1, dtype=np.int32)
    out[1:] = np.cumsum(lens)
    return out
