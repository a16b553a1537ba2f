"""The seeded input generators (CPU): the recipe the tests and the benchmark
share holds what it promises -- reproducible draws, a shuffled pool with
exactly the owned pages plus NaN-poisoned spares, block tables padded with -1,
exclusive prefix sums for cu_seq_lens, and new-token slots of the mixed step
that land at each sequence's next position in its own pages."""
import math

import numpy as np
import torch

from paged_kv_cache_attention_gb300 import workloads as W

BF16 = torch.bfloat16


def _bits(t):
    return t.view(torch.int16) if t.dtype == BF16 else t


def test_same_seed_same_inputs_other_seed_other_inputs():
    a = W.make_decode([33, 70, 5], 8, 2, 64, 16, BF16, seed=7, sink="randn")
    b = W.make_decode([33, 70, 5], 8, 2, 64, 16, BF16, seed=7, sink="randn")
    c = W.make_decode([33, 70, 5], 8, 2, 64, 16, BF16, seed=8, sink="randn")
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache)):
        assert torch.equal(_bits(x), _bits(y))
    assert torch.equal(a.block_table, b.block_table) and torch.equal(a.sink, b.sink)
    assert not torch.equal(_bits(a.q), _bits(c.q))
    assert not torch.equal(a.block_table, c.block_table)


def _check_pool(k_cache, v_cache, tables_and_lens, bs, spare=64):
    """Owned pages: distinct, finite; every other page NaN; tables -1 padded."""
    owned = []
    for bt, lens in tables_and_lens:
        for i, L in enumerate(lens):
            n = (int(L) + bs - 1) // bs
            row = bt[i].tolist()
            assert all(p >= 0 for p in row[:n]) and all(p == -1 for p in row[n:])
            owned += row[:n]
    nb = k_cache.shape[0]
    assert len(owned) == len(set(owned)) and nb == len(owned) + spare
    mask = torch.zeros(nb, dtype=torch.bool)
    mask[torch.tensor(owned, dtype=torch.int64)] = True
    for pool in (k_cache, v_cache):
        flat = pool.float().reshape(nb, -1)
        assert torch.isfinite(flat[mask]).all()
        assert torch.isnan(flat[~mask]).all()
    # the pages are shuffled, not handed out in order
    assert owned != sorted(owned)


def test_decode_pool_holds_the_owned_pages_plus_poisoned_spares():
    lens = [1, 16, 17, 300, 0, 1024]
    case = W.make_decode(lens, 8, 2, 64, 16, BF16, seed=11)
    _check_pool(case.k_cache, case.v_cache, [(case.block_table, lens)], 16)
    assert case.cache_seqlens.tolist() == lens and case.max_seqlen == 1024
    assert case.block_table.dtype == torch.int32 and case.cache_seqlens.dtype == torch.int32


def test_varlen_offsets_are_exclusive_prefix_sums():
    q_lens, prefix = [5, 0, 130, 1], [0, 40, 2000, 31]
    case = W.make_varlen(q_lens, prefix, 8, 2, 64, 32, BF16, seed=12)
    kv = [q + p for q, p in zip(q_lens, prefix)]
    assert case.cu_seq_lens_q.tolist() == list(np.cumsum([0] + q_lens))
    assert case.cu_seq_lens_k.tolist() == list(np.cumsum([0] + kv))
    assert case.q.shape[0] == sum(q_lens) == case.total_q
    assert case.max_seqlen_q == 130 and case.max_seqlen_k == 2130
    _check_pool(case.k_cache, case.v_cache, [(case.block_table, kv)], 32)


def test_mixed_step_slots_are_each_sequences_next_positions():
    dec_lens, cq, cp, nch, bs = [15, 16, 31, 200, 1], 40, 70, 3, 16
    case = W.make_mixed(dec_lens, cq, cp, nch, 8, 2, 64, bs, BF16, seed=13)
    dec, pre = case.decode, case.prefill
    assert case.num_new_tokens == len(dec_lens) + nch * cq
    assert dec.cache_seqlens.tolist() == [L + 1 for L in dec_lens]
    assert pre.cu_seq_lens_k.tolist() == [r * (cp + cq) for r in range(nch + 1)]
    _check_pool(case.k_cache, case.v_cache,
                [(dec.block_table, [L + 1 for L in dec_lens]),
                 (pre.block_table, [cp + cq] * nch)], bs)
    # where each new token must go: (table, row, position)
    want = [(dec.block_table, b, L) for b, L in enumerate(dec_lens)]
    want += [(pre.block_table, r, p) for r in range(nch) for p in range(cp, cp + cq)]
    slots = case.slot_mapping.tolist()
    assert len(set(slots)) == len(slots)
    for s, (bt, row, pos) in zip(slots, want):
        page, off = divmod(s, bs)
        assert page == int(bt[row, pos // bs]) and off == pos % bs
    assert case.positions.tolist() == [pos for _, _, pos in want]


def test_integer_draws_cover_their_inclusive_ranges():
    g = W._gen(5)
    u = W.uniform_int(3, 9, 20000, g)
    assert int(u.min()) == 3 and int(u.max()) == 9
    lu = W.log_uniform_int(128, 16384, 20000, g)
    assert int(lu.min()) >= 128 and int(lu.max()) <= 16384
    # log-uniform: the median sits near the geometric mean of the bounds, and
    # each factor-of-two band holds about the same share of the draws
    med = float(lu.double().median())
    assert abs(math.log(med) - 0.5 * (math.log(128) + math.log(16384))) < 0.05
    bands = torch.histc(torch.log2(lu.double()), bins=7, min=7, max=14)
    assert float(bands.min()) > 0.8 * 20000 / 7


def test_input_values_are_standard_normal_rounded_to_the_dtype():
    g = W._gen(6)
    x = W.randn((256, 1024), BF16, g)
    assert x.dtype == BF16
    f = x.float()
    assert abs(float(f.mean())) < 0.01 and abs(float(f.std()) - 1.0) < 0.01
    # drawn in fp32, then rounded once: the same draw in fp32 rounds to it
    y = W.randn((256, 1024), torch.float32, W._gen(6))
    assert torch.equal(y.to(BF16).view(torch.int16), x.view(torch.int16))


def test_alibi_slopes():
    g = W._gen(7)
    geo = W.alibi_slopes("geometric", 8, g)
    assert geo.tolist() == [2.0 ** -(i + 1) for i in range(8)]  # 2^(-8 (i+1) / 8)
    uni = W.alibi_slopes("uniform", 1000, g)
    assert float(uni.min()) >= 0.01 and float(uni.max()) <= 1.0
    assert W.alibi_slopes("none", 8, g) is None
