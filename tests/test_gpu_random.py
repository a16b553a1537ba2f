"""Seeded random configurations of paged_decode and varlen_prefill against the
fp64 oracle: each draw mixes a head size, a group size, a page size, a pool
layout, lengths (including empty and page-boundary ones), a window, a sink,
ALiBi slopes and, for prefill, causal or not, so that combinations no
hand-written case pairs up still meet the same bar (max-abs 2e-2 on bf16
outputs, 1e-5 on fp32, log-sum-exp within 2e-3 / 1e-5)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import (LSE_TOL, TOL, gpu_decode, gpu_prefill, lse_err, max_abs,
                        oracle_decode, oracle_prefill)

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _lengths(g, n, lo, hi, bs):
    """n lengths in [lo, hi], a few of them on or next to a page boundary."""
    out = g.integers(lo, hi + 1, n)
    for i in range(0, n, 3):
        edge = bs * int(g.integers(0, hi // bs + 1)) + int(g.integers(-1, 2))
        out[i] = max(lo, min(hi, edge))
    return [int(x) for x in out]


@pytest.mark.parametrize("draw", range(32))
def test_random_decode(draw):
    g = np.random.default_rng(9100 + draw)
    dtype = BF16 if draw % 4 else torch.float32
    D = int(g.choice([64, 80, 96, 112, 128] + ([256] if dtype == BF16 else [])))
    G = int(g.choice([1, 2, 4, 8, 16]))
    Hkv = int(g.choice([1, 2, 4]))
    bs = int(g.choice([16, 32]))
    B = int(g.integers(1, 13))
    lens = _lengths(g, B, 0, 6000, bs)
    window = int(g.choice([-1, -1, 0, 31, 700]))
    sink = str(g.choice(["none", "randn"]))
    alibi = str(g.choice(["none", "none", "geometric", "uniform"]))
    layout = "HND" if (dtype == BF16 and g.random() < 0.3) else "NHD"
    case = W.make_decode(lens, G * Hkv, Hkv, D, bs, dtype, seed=9200 + draw, sink=sink,
                         window_left=window, alibi=alibi)
    got, glse = gpu_decode(case, with_lse=True, layout=layout)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[dtype]
    assert lse_err(glse, rlse) <= LSE_TOL[dtype]


@pytest.mark.parametrize("draw", range(32))
def test_random_prefill(draw):
    g = np.random.default_rng(9300 + draw)
    D = int(g.choice([64, 80, 96, 112, 128, 256]))
    G = int(g.choice([1, 2, 4, 8, 16]))
    Hkv = int(g.choice([1, 2, 4]))
    bs = int(g.choice([16, 32]))
    B = int(g.integers(1, 6))
    q_lens = _lengths(g, B, 0, 600, bs)
    prefix = _lengths(g, B, 0, 2500, bs)
    causal = bool(g.random() < 0.7)
    window = int(g.choice([-1, -1, 0, 63, 500]))
    sink = str(g.choice(["none", "randn"]))
    alibi = str(g.choice(["none", "none", "geometric", "uniform"]))
    layout = "HND" if g.random() < 0.3 else "NHD"
    case = W.make_varlen(q_lens, prefix, G * Hkv, Hkv, D, bs, BF16, seed=9400 + draw,
                         sink=sink, window_left=window, causal=causal, alibi=alibi)
    got, glse = gpu_prefill(case, with_lse=True, layout=layout)
    ref, rlse = oracle_prefill(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[BF16]
    assert lse_err(glse, rlse) <= LSE_TOL[BF16]
