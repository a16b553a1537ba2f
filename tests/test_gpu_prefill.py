"""varlen_prefill on the GPU against the fp64 oracle on the same seeded inputs.

Bar: max-abs error 2e-2 on bf16 outputs (P is rounded to bf16 before the PV
product, the oracle is exact), lse within 2e-3.
"""
import json
import os

import numpy as np
import pytest
import torch

import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import (LSE_TOL, TOL, contiguous_kv, dev, gpu_decode, gpu_prefill,
                        gpu_prefill_contiguous, lse_err, max_abs, oracle_decode, oracle_prefill,
                        to_dev)

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _check(case, rows=None, lse=True):
    got, glse = gpu_prefill(case, with_lse=True)
    ref, rlse = oracle_prefill(case, rows=rows, with_lse=True)
    if rows is not None:
        got, glse = got[rows], glse[rows]
    assert max_abs(got, ref) <= TOL[BF16]
    if lse:
        assert lse_err(glse, rlse) <= LSE_TOL[BF16]
    return got


def test_varlen_example_of_the_page():
    """cu_seq_lens_q [0,10,13,14], cu_seq_lens_k [0,0,1,8]: request 0 has no
    key (10 zero rows), request 1 has 3 queries over 1 key (rows at positions
    -2, -1 see nothing, the last sees key 0), request 2 one query over 7 keys."""
    g = json.load(open(os.path.join(GOLDEN, "varlen_example.json")))
    case = W.make_varlen_kv(g["q_lens"], g["k_lens"], 8, 2, 128, 16, BF16, seed=21,
                            sink="randn")
    assert case.cu_seq_lens_q.tolist() == g["cu_seq_lens_q"]
    assert case.cu_seq_lens_k.tolist() == g["cu_seq_lens_k"]
    got = _check(case)
    assert np.all(got[:12] == 0) and np.all(got[12:] != 0)


@pytest.mark.parametrize("G,Hkv", [(1, 4), (2, 4), (4, 8), (8, 2), (16, 1)])
@pytest.mark.parametrize("bs", [16, 32])
def test_group_sizes_and_pages(G, Hkv, bs):
    q_lens = [1, 7, 33, 64, 129, 300]
    prefix = [0, 100, 5, 128, 1000, 77]
    case = W.make_varlen(q_lens, prefix, G * Hkv, Hkv, 128, bs, BF16, seed=G * 31 + bs,
                         sink="randn")
    _check(case)


@pytest.mark.parametrize("sink", ["none", "randn"])
@pytest.mark.parametrize("window", [-1, 0, 7, 127, 128, 1000])
def test_windows_and_sinks(sink, window):
    q_lens = [200, 1, 513, 64]
    prefix = [300, 2000, 0, 64]
    case = W.make_varlen(q_lens, prefix, 32, 8, 128, 16, BF16, seed=window + 50, sink=sink,
                         window_left=window)
    _check(case)


def test_empty_requests_and_ragged_tails():
    q_lens = [0, 5, 0, 127, 128, 129, 1]
    kv_lens = [10, 5, 0, 127, 1000, 129, 0]
    case = W.make_varlen_kv(q_lens, kv_lens, 16, 4, 128, 16, BF16, seed=22, sink="randn")
    _check(case)


# ---------------------------------------------------------------------------
# non-causal varlen (no upper bound on keys; a window still bounds them below)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("sink", ["none", "randn"])
@pytest.mark.parametrize("window", [-1, 0, 7, 128, 1000])
def test_non_causal_windows_and_sinks(sink, window):
    q_lens = [200, 1, 513, 64, 300, 9]
    kv_lens = [500, 2001, 513, 64, 40, 0]   # q_len > kv_len in request 4
    case = W.make_varlen_kv(q_lens, kv_lens, 32, 8, 128, 16, BF16, seed=window + 70,
                            sink=sink, window_left=window, causal=False)
    _check(case)


@pytest.mark.parametrize("G,Hkv,bs", [(1, 4, 32), (4, 4, 16), (16, 1, 16)])
def test_non_causal_group_sizes(G, Hkv, bs):
    case = W.make_varlen_kv([1, 33, 129, 250], [1, 300, 129, 1000], G * Hkv, Hkv, 128, bs, BF16,
                            seed=G * 13 + bs, sink="randn", causal=False)
    _check(case)


def test_non_causal_rows_see_the_same_keys():
    """Without the causal bound and window every row of a request attends to
    the same key set: permuting the queries of a request permutes the outputs."""
    case = W.make_varlen_kv([100], [700], 16, 4, 128, 16, BF16, seed=27, causal=False)
    a = gpu_prefill(case)
    perm = torch.randperm(100, generator=torch.Generator().manual_seed(5))
    case.q = case.q[perm].contiguous()
    b = gpu_prefill(case)
    assert np.array_equal(a[perm.numpy()], b)


# ---------------------------------------------------------------------------
# contiguous (unpaged) keys and values addressed by cu_seq_lens_k
# ---------------------------------------------------------------------------

def _check_contig(case, pad_rows=0, rows=None):
    k, v = contiguous_kv(case, pad_rows)
    got, glse = gpu_prefill_contiguous(case, k, v, with_lse=True)
    ref, rlse = oracle_prefill(case, rows=rows, with_lse=True)
    if rows is not None:
        got, glse = got[rows], glse[rows]
    assert max_abs(got, ref) <= TOL[BF16]
    assert lse_err(glse, rlse) <= LSE_TOL[BF16]
    return got


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window,sink", [(-1, "randn"), (0, "none"), (100, "randn")])
def test_contiguous_matches_oracle(causal, window, sink):
    """NaN rows after the last request: a tile that runs past a request's keys
    must mask them (keys) and zero them (values)."""
    q_lens = [0, 5, 127, 128, 300, 1, 64]
    kv_lens = [10, 5, 127, 1000, 300, 0, 129]
    case = W.make_varlen_kv(q_lens, kv_lens, 32, 8, 128, 16, BF16, seed=window + 90,
                            sink=sink, window_left=window, causal=causal)
    _check_contig(case, pad_rows=200)


@pytest.mark.parametrize("G,Hkv", [(1, 8), (2, 4), (8, 2), (16, 1)])
def test_contiguous_group_sizes(G, Hkv):
    case = W.make_varlen([1, 70, 129, 256], [0, 100, 1000, 3], G * Hkv, Hkv, 128, 16, BF16,
                         seed=G + 40, sink="randn")
    _check_contig(case)


def test_contiguous_equals_paged():
    """Same tiles, same arithmetic order: the contiguous and paged forms give
    identical bits."""
    case = W.make_varlen([150, 40, 300], [500, 9, 0], 32, 8, 128, 16, BF16, seed=28,
                         sink="randn", window_left=200)
    a = gpu_prefill(case)
    k, v = contiguous_kv(case)
    b = gpu_prefill_contiguous(case, k, v)
    assert np.array_equal(a, b)


def test_contiguous_without_keys():
    case = W.make_varlen_kv([3, 4], [0, 0], 8, 2, 128, 16, BF16, seed=29, sink="randn")
    k, v = contiguous_kv(case)
    assert k.shape[0] == 0
    got, glse = gpu_prefill_contiguous(case, k, v, with_lse=True)
    assert np.all(got == 0)
    np.testing.assert_allclose(glse, np.broadcast_to(case.sink.numpy(), glse.shape), atol=1e-6)


def test_contiguous_rows_past_the_arrays_are_flagged():
    """cu_seq_lens_k running past total_k: the request is clipped to the rows
    that exist, PKV_DEVERR_SEQLEN is raised and the other requests are exact."""
    case = W.make_varlen_kv([40, 40], [100, 100], 8, 2, 128, 16, BF16, seed=30, sink="randn")
    k, v = contiguous_kv(case)
    k, v = k[:150].contiguous(), v[:150].contiguous()
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    got = gpu_prefill_contiguous(case, k, v, err=err)
    assert int(err.item()) & pkv.DEVERR_SEQLEN
    assert np.isfinite(got).all()
    ref = oracle_prefill(case, rows=list(range(40)))
    assert max_abs(got[:40], ref) <= TOL[BF16]


# ---------------------------------------------------------------------------
# ALiBi
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window,sink,alibi", [(-1, "randn", "geometric"), (-1, "none", "uniform"),
                                               (127, "randn", "uniform"), (0, "randn", "geometric")])
def test_alibi_prefill(causal, window, sink, alibi):
    q_lens = [200, 1, 513, 64, 300]
    kv_lens = [500, 2001, 513, 64, 40]
    case = W.make_varlen_kv(q_lens, kv_lens, 32, 8, 128, 16, BF16, seed=window + 110,
                            sink=sink, window_left=window, causal=causal, alibi=alibi)
    _check(case)


@pytest.mark.parametrize("G,Hkv,bs", [(1, 8, 32), (4, 4, 16), (16, 1, 16)])
def test_alibi_prefill_group_sizes(G, Hkv, bs):
    case = W.make_varlen([1, 33, 129, 250], [0, 300, 128, 1000], G * Hkv, Hkv, 128, bs, BF16,
                         seed=G * 17 + bs, sink="randn", alibi="uniform")
    _check(case)


@pytest.mark.parametrize("causal", [True, False])
def test_alibi_steep_slopes_peaked(causal):
    """Slopes in [0.5, 2]: each row's weight sits on one or two keys, so the
    output is nearly one value row and the rounding of the dominant P to bf16
    is not averaged away.  Rows span many key tiles and ragged ends."""
    q_lens = [1, 7, 130, 513, 64]
    kv_lens = [3000, 7, 1000, 513, 2]
    case = W.make_varlen_kv(q_lens, kv_lens, 32, 8, 128, 16, BF16, seed=130 + int(causal),
                            sink="randn", causal=causal, alibi="steep")
    _check(case)


def test_alibi_contiguous():
    case = W.make_varlen_kv([5, 127, 300], [5, 1000, 300], 32, 8, 128, 16, BF16, seed=120,
                            sink="randn", alibi="geometric", causal=False)
    _check_contig(case, pad_rows=64)


def test_alibi_decode_equals_prefill_with_one_query():
    dec = W.make_decode([1, 300, 1024, 4097], 32, 8, 128, 16, BF16, seed=121, sink="randn",
                        window_left=700, alibi="uniform")
    B = dec.batch
    var = W.VarlenCase("as-prefill", dec.q, dec.k_cache, dec.v_cache, dec.block_table,
                       W.cumsum0(torch.ones(B, dtype=torch.int32)),
                       W.cumsum0(dec.cache_seqlens), dec.sink, dec.window_left, dec.sm_scale,
                       True, dec.alibi)
    a = gpu_decode(dec)
    b = gpu_prefill(var)
    assert np.abs(a - b).max() <= 2e-2
    assert max_abs(b, oracle_decode(dec)) <= TOL[BF16]


# ---------------------------------------------------------------------------
# head sizes 64 / 80 / 96 / 112 (tiles padded to 128 with zeros)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 80, 96, 112])
@pytest.mark.parametrize("G,Hkv", [(4, 8), (1, 4), (16, 1)])
def test_head_sizes(D, G, Hkv):
    q_lens = [1, 33, 129, 300]
    kv_lens = [1, 333, 1000, 300]
    case = W.make_varlen_kv(q_lens, kv_lens, G * Hkv, Hkv, D, 16, BF16, seed=D + G,
                            sink="randn", window_left=200 if G == 1 else -1,
                            alibi="geometric" if G == 16 else "none")
    _check(case)


@pytest.mark.parametrize("D", [80, 112])
def test_head_sizes_contiguous_non_causal(D):
    case = W.make_varlen_kv([5, 127, 300], [5, 1000, 300], 32, 8, D, 16, BF16, seed=D + 3,
                            sink="randn", causal=False)
    _check_contig(case, pad_rows=32)


# ---------------------------------------------------------------------------
# head size 256 (its own kernel: query tiles in sequence, 64-key tiles)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("G,Hkv,bs", [(4, 4, 16), (1, 8, 32), (16, 1, 16), (2, 2, 32)])
@pytest.mark.parametrize("causal", [True, False])
def test_head_size_256(G, Hkv, bs, causal):
    q_lens = [1, 7, 64, 130, 300, 5]
    kv_lens = [1, 900, 64, 130, 700, 0]
    case = W.make_varlen_kv(q_lens, kv_lens, G * Hkv, Hkv, 256, bs, BF16, seed=G * 5 + bs,
                            sink="randn", causal=causal)
    _check(case)


@pytest.mark.parametrize("window,alibi", [(0, "none"), (100, "uniform"), (-1, "steep")])
def test_head_size_256_windows_alibi(window, alibi):
    case = W.make_varlen([1, 33, 129, 250], [0, 300, 128, 1000], 16, 4, 256, 16, BF16,
                         seed=window + 7, sink="randn", window_left=window, alibi=alibi)
    _check(case)


def test_head_size_256_q_longer_than_kv():
    """Rows at negative positions in the first query tile attend nothing while
    the second tile has keys: the tiles of an item run with their own ranges."""
    case = W.make_varlen_kv([200, 3], [70, 1], 8, 2, 256, 16, BF16, seed=141, sink="randn")
    _check(case)


def test_head_size_256_contiguous_and_hnd():
    case = W.make_varlen_kv([5, 127, 300], [5, 1000, 300], 16, 4, 256, 16, BF16, seed=142,
                            sink="randn", alibi="geometric")
    _check_contig(case, pad_rows=64)
    got = gpu_prefill(case, layout="HND")
    assert max_abs(got, oracle_prefill(case)) <= TOL[BF16]
    assert np.array_equal(got, gpu_prefill(case))


def test_head_size_256_decode_equals_prefill():
    dec = W.make_decode([1, 300, 1024, 2049], 16, 4, 256, 16, BF16, seed=143, sink="randn",
                        window_left=700)
    B = dec.batch
    var = W.VarlenCase("as-prefill", dec.q, dec.k_cache, dec.v_cache, dec.block_table,
                       W.cumsum0(torch.ones(B, dtype=torch.int32)),
                       W.cumsum0(dec.cache_seqlens), dec.sink, dec.window_left, dec.sm_scale)
    a = gpu_decode(dec)
    b = gpu_prefill(var)
    assert np.abs(a - b).max() <= 2e-2
    assert max_abs(b, oracle_decode(dec)) <= TOL[BF16]


def test_decode_equals_prefill_with_one_query():
    """Cross-op: paged_decode == varlen_prefill with q_len = 1 per request."""
    dec = W.make_decode([1, 300, 1024, 4097], 32, 8, 128, 16, BF16, seed=23, sink="randn",
                        window_left=500)
    B = dec.batch
    var = W.VarlenCase("as-prefill", dec.q, dec.k_cache, dec.v_cache, dec.block_table,
                       W.cumsum0(torch.ones(B, dtype=torch.int32)),
                       W.cumsum0(dec.cache_seqlens), dec.sink, dec.window_left, dec.sm_scale)
    a = gpu_decode(dec)
    b = gpu_prefill(var)
    assert np.abs(a - b).max() <= 2e-2
    assert max_abs(b, oracle_decode(dec)) <= TOL[BF16]


def test_chunk_is_suffix_of_longer_chunk():
    """A chunk of the last 40 queries equals the last 40 rows of a 300-query
    chunk over the same keys (mask aligned to the end of kv)."""
    long_ = W.make_varlen([300], [700], 32, 8, 128, 16, BF16, seed=24, sink="randn")
    short = W.VarlenCase("short", long_.q[-40:].contiguous(), long_.k_cache, long_.v_cache,
                         long_.block_table, W.cumsum0(torch.tensor([40], dtype=torch.int32)),
                         long_.cu_seq_lens_k, long_.sink, -1, long_.sm_scale)
    a = gpu_prefill(long_)
    b = gpu_prefill(short)
    assert np.abs(a[-40:] - b).max() <= 2e-2


def test_block_relabelling_invariance():
    case = W.make_varlen([150, 40], [500, 9], 32, 8, 128, 16, BF16, seed=25)
    a = gpu_prefill(case)
    perm = torch.randperm(case.k_cache.shape[0], generator=torch.Generator().manual_seed(4))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    case.k_cache = case.k_cache[perm].contiguous()
    case.v_cache = case.v_cache[perm].contiguous()
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    case.block_table = bt
    b = gpu_prefill(case)
    assert np.array_equal(a, b)


def test_bad_block_id_is_flagged():
    case = W.make_varlen([40, 40], [100, 100], 8, 2, 128, 16, BF16, seed=26)
    case.block_table[1, 3] = -7
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    got = gpu_prefill(case, err=err)
    assert int(err.item()) & pkv.DEVERR_BLOCK_ID
    assert np.isfinite(got).all()
    ref = oracle_prefill(case, rows=list(range(40)))
    assert max_abs(got[:40], ref) <= TOL[BF16]


@pytest.mark.parametrize("G", [2, 4])
def test_work_list_is_each_item_once_in_request_order(G):
    """The work list the prefill builds on the device holds every (request,
    query block, kv head) exactly once; the requests come heaviest first by
    the key-tile count of their heaviest query block, and each request's
    items are contiguous: its query blocks heaviest first (for causal
    attention the later ones), each with its kv heads side by side.  The
    output is still the attention (checked against the oracle)."""
    Hkv = 4
    q_lens, pre = [1, 300, 129, 700, 64, 40], [0, 5000, 100, 0, 3000, 200]
    case = W.make_varlen(q_lens, pre, G * Hkv, Hkv, 128, 16, BF16, seed=31)
    ws = torch.zeros(pkv.varlen_prefill_workspace_size(case.batch, G * Hkv, Hkv, case.total_q,
                                                       case.max_seqlen_q),
                     dtype=torch.uint8, device=dev())
    kc, vc = to_dev(case.k_cache), to_dev(case.v_cache)
    out = pkv.varlen_prefill(to_dev(case.q), kc, vc, to_dev(case.block_table),
                             to_dev(case.cu_seq_lens_q), to_dev(case.cu_seq_lens_k),
                             case.max_seqlen_q, case.max_seqlen_k, sink=to_dev(case.sink),
                             sm_scale=case.sm_scale, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle_prefill(case)
    assert max_abs(out.float().cpu().numpy(), ref) <= TOL[BF16]

    w = ws.view(torch.int32).cpu().numpy()
    n = int(w[0])
    items = w[64:64 + 4 * n].reshape(n, 4)  # (request, first query token, kv head, cost)
    tokens = 2 * (128 // G)
    kv_lens = case.kv_lens.tolist()

    def cost(r, t0):  # key tiles of a causal query block, from the definition
        t_end = min(t0 + tokens, q_lens[r])
        hi = min(kv_lens[r], kv_lens[r] - q_lens[r] + t_end)
        return (hi - 1) // 128 + 1 if hi > 0 else 0

    want = {(r, t0, g) for r in range(case.batch) for t0 in range(0, q_lens[r], tokens)
            for g in range(Hkv)}
    got = [tuple(int(v) for v in it[:3]) for it in items]
    assert len(got) == len(want) and set(got) == want
    assert all(int(it[3]) == cost(int(it[0]), int(it[1])) for it in items)
    # each request's items contiguous, blocks from the heaviest down, heads
    # side by side
    order = [int(it[0]) for it in items]
    firsts = [order.index(r) for r in range(case.batch)]
    for r in range(case.batch):
        nb = (q_lens[r] + tokens - 1) // tokens
        mine = [tuple(int(v) for v in it[:3]) for it in items[firsts[r]:firsts[r] + nb * Hkv]]
        assert mine == [(r, t0, g) for t0 in reversed(range(0, q_lens[r], tokens))
                        for g in range(Hkv)]
    # requests by their heaviest block, heaviest first
    heaviest = [max(cost(r, t0) for t0 in range(0, q_lens[r], tokens)) for r in range(case.batch)]
    seq = [heaviest[r] for r in sorted(range(case.batch), key=lambda r: firsts[r])]
    assert seq == sorted(seq, reverse=True)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("cu_q", [[0, 40, 80], [0, 70, 80], [0, 50, 30]])
def test_query_offsets_past_total_q_are_clipped_and_flagged(D, cu_q):
    """cu_seq_lens_q lives on the device: offsets past total_q (the rows of q
    the caller declared), a request running past them, or a decreasing pair
    must be clipped to the declared rows and flagged, and nothing past the
    output and lse rows may be written (sentinel tail)."""
    Hq, Hkv, T = 8, 2, 60
    case = W.make_varlen([40, 40], [100, 100], Hq, Hkv, D, 16, BF16, seed=27)
    d = dev()
    q_full = case.q.to(d)                  # 80 rows; the call sees the first 60
    out_buf = torch.full((80, Hq, D), 7.0, dtype=BF16, device=d)
    lse_buf = torch.full((80, Hq), 7.0, dtype=torch.float32, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    cuq = torch.tensor(cu_q, dtype=torch.int32, device=d)
    pkv.varlen_prefill(q_full[:T], case.k_cache.to(d), case.v_cache.to(d),
                       case.block_table.to(d), cuq, case.cu_seq_lens_k.to(d), 80,
                       case.max_seqlen_k, sm_scale=case.sm_scale, out=out_buf[:T],
                       lse=lse_buf[:T], dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_SEQLEN
    assert torch.all(out_buf[T:] == 7.0) and torch.all(lse_buf[T:] == 7.0)
    got = out_buf[:T].float().cpu().numpy()
    assert np.isfinite(got).all()
    if cu_q[1] == 40:  # request 0 is intact: its rows match the oracle
        ref = oracle_prefill(case, rows=list(range(40)))
        assert max_abs(got[:40], ref) <= TOL[BF16]


def _sample_rows(case, n_per_req=4):
    rows = []
    cu = case.cu_seq_lens_q.tolist()
    for r in range(case.batch):
        a, b = cu[r], cu[r + 1]
        if b > a:
            rows += sorted({a, b - 1, (a + b) // 2, a + (b - a) // 3})[:n_per_req]
    return rows


def _every_nth_row(case, n):
    """Every n-th query row of the batch, plus each request's first and last
    row (the rows at the ends of the causal ranges)."""
    rows = set(range(0, case.total_q, n))
    cu = case.cu_seq_lens_q.tolist()
    for r in range(case.batch):
        if cu[r + 1] > cu[r]:
            rows |= {cu[r], cu[r + 1] - 1}
    return sorted(rows)


def test_config4_prefill_full_size():
    """The B16 varlen batch at full size: every query row of every request
    (16 requests, prefixes up to 8K keys) against the oracle, with lse."""
    case = W.config4_prefill()
    _check(case)


def test_config4_prefill_alibi_full_size():
    # the B16 batch with geometric slopes: prefixes up to ~10K keys, so the
    # per-tile ALiBi constant slope * (tile start - position) reaches its
    # largest magnitudes; every fourth row and each request's ends
    case = W.config4_prefill()
    case.alibi = W.alibi_slopes("geometric", case.q.shape[1], None)
    _check(case, rows=_every_nth_row(case, 4))


def test_config4_prefill_head_size_256_full_size():
    case = W.config4_prefill(16, 8, 256)
    _check(case, rows=_every_nth_row(case, 4))


def test_config5_prefill_half_after_cache_write():
    case = W.config5_mixed()
    d = dev()
    kc, vc = case.k_cache.to(d), case.v_cache.to(d)
    pkv.reshape_and_cache(case.key.to(d), case.value.to(d), kc, vc, case.slot_mapping.to(d))
    torch.cuda.synchronize()
    pre = case.prefill
    pre.k_cache, pre.v_cache = kc.cpu(), vc.cpu()
    _check(pre)  # all 8192 query rows, with lse


def test_many_requests_work_list():
    """1500 requests: more than the work-list kernel takes in one pass of its
    1024 threads, with lengths spread over many cost buckets; every 7th
    request has no queries.  Sampled rows of every request against the
    oracle."""
    g = np.random.default_rng(31)
    n = 1500
    q_lens = g.integers(1, 48, n)
    q_lens[::7] = 0
    prefix = g.integers(0, 600, n)
    case = W.make_varlen(q_lens.tolist(), prefix.tolist(), 8, 2, 128, 16, BF16, seed=32,
                         sink="randn")
    _check(case, rows=_sample_rows(case, 2))
