"""MInference vertical + slash sparse prefill on the GPU against the fp64
oracle.

The pattern is an integer decision taken on floating-point scores (fp32 on
the GPU, fp64 in the oracle), so the test first checks the GPU's kept sets
against the oracle's scores (every kept index scores at least as much as
every dropped one, within the fp32 error of a sum of probabilities) and then
requires the sets to be identical on these seeded inputs; the attention is
compared with the oracle's sparse attention over the oracle's own pattern.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import TOL, dev, max_abs

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _case(S, Hq, Hkv, D, seed):
    gen = torch.Generator().manual_seed(seed)
    q = W.randn((S, Hq, D), BF16, gen)
    k = W.randn((S, Hkv, D), BF16, gen)
    v = W.randn((S, Hkv, D), BF16, gen)
    return q, k, v


def _valid(kept, scores, n_force, tol):
    """kept indices (beyond the forced ones) outscore every dropped index."""
    S = scores.shape[0]
    mask = np.zeros(S, bool)
    mask[kept] = True
    mask[:n_force] = False
    free = scores[mask]
    drop = np.ones(S, bool)
    drop[kept] = False
    drop[:n_force] = False
    if free.size == 0 or not drop.any():
        return True
    return free.min() >= scores[drop].max() - tol


def _run(q, k, v, **kw):
    d = dev()
    out, vi, si = pkv.minference_prefill(q.to(d), k.to(d), v.to(d), return_pattern=True, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), vi.cpu().numpy(), si.cpu().numpy()


def _check(S, Hq, Hkv, D, seed, structured=False, **kw):
    q, k, v = (W.make_long_sequence(S, Hq, Hkv, D, seed) if structured
               else _case(S, Hq, Hkv, D, seed))
    out, vi, si = _run(q, k, v, **kw)
    ovi, osi, vsc, ssc = oracle.minference_pattern(W.to_oracle(q), W.to_oracle(k), **kw)
    assert vi.shape == ovi.shape and si.shape == osi.shape
    n_sink = kw.get("num_sink_tokens", 30)
    n_recent = kw.get("num_recent_diags", 100)
    for h in range(Hq):
        assert np.all(np.diff(vi[h]) > 0) and np.all(np.diff(si[h]) > 0)
        assert _valid(vi[h], vsc[h], n_sink, 1e-5)
        assert _valid(si[h], ssc[h], n_recent, 1e-5)
    np.testing.assert_array_equal(vi, ovi)
    np.testing.assert_array_equal(si, osi)
    ref = oracle.sparse_attention(W.to_oracle(q), W.to_oracle(k), W.to_oracle(v), ovi, osi)
    assert max_abs(out, ref) <= TOL[BF16]
    return out, vi, si


@pytest.mark.parametrize("S,Hq,Hkv,D", [(500, 8, 2, 128), (1100, 4, 4, 64), (2048, 8, 2, 128),
                                        (129, 16, 1, 96)])
def test_adaptive_budget(S, Hq, Hkv, D):
    _check(S, Hq, Hkv, D, seed=S + D)


@pytest.mark.parametrize("S,Hq,Hkv", [(1800, 8, 2), (2048, 16, 4), (16384, 4, 2)])
def test_structured_long_sequence(S, Hq, Hkv):
    """Attention with local (slash) and stripe (vertical) structure, the kind
    the pattern is built to capture."""
    _check(S, Hq, Hkv, 128, seed=S + Hq, structured=True)


@pytest.mark.parametrize("S", [1, 7, 63, 64, 65])
def test_short_sequences(S):
    """Fewer than 64 queries: every query estimates; the forced sinks and
    recent diagonals cover the whole (tiny) sequence."""
    _check(S, 4, 2, 64, seed=S)


def test_fixed_sizes():
    _check(1500, 8, 2, 128, seed=3, adaptive_budget=None, vertical_size=100, slash_size=200,
           num_sink_tokens=8, num_recent_diags=16)


def test_keeping_every_key_is_dense_causal_prefill():
    """With every column kept the sparse prefill is dense causal attention
    (the sparse form walks the key tiles from the query's end and rescales on
    every new maximum, so it agrees with the dense kernel to rounding, not bit
    for bit)."""
    S, Hq, Hkv, D = 700, 8, 2, 128
    q, k, v = _case(S, Hq, Hkv, D, seed=4)
    out, vi, _ = _run(q, k, v, adaptive_budget=None, vertical_size=S, slash_size=1)
    assert vi.shape == (Hq, S)
    d = dev()
    cu = torch.tensor([0, S], dtype=torch.int32, device=d)
    dense = pkv.varlen_prefill_contiguous(q.to(d), k.to(d), v.to(d), cu, cu, S, S)
    torch.cuda.synchronize()
    assert np.abs(out - dense.float().cpu().numpy()).max() <= 2e-2
    kp = k.unsqueeze(1).contiguous()  # one-row pages: page j holds key j
    vp = v.unsqueeze(1).contiguous()
    bt = np.arange(S, dtype=np.int32)[None, :]
    ref = oracle.attention(W.to_oracle(q), W.to_oracle(kp), W.to_oracle(vp), bt,
                           np.array([0, S], np.int32), np.array([S], np.int32), causal=True,
                           sm_scale=D ** -0.5)
    assert max_abs(out, ref) <= TOL[BF16]
