"""Pins of the fp64 CPU oracle to things other than itself (CPU only).

Each test checks the oracle against a fact the pages or the mathematics fix:
  * the worked examples of the transformers docs "paged_attention" page
    (token -> request by cu_seq_lens; pages and new-token slots by block_table),
    stored under tests/golden/ with their citation;
  * a library routine: torch's scaled_dot_product_attention in fp64, for the
    plain softmax (no sink), and for the sink read as one more softmax column
    with a zero value row (sink_attention_reference.py, sink_softmax);
  * closed forms: window_left = 0 leaves one key, o = v * sigmoid(s - sink);
  * invariances: physical page relabelling, page size, window >= kv_len,
    decode == last prefill row, chunk == suffix of a longer chunk;
  * an independent dense brute force in numpy on tiny inputs (with and
    without ALiBi);
  * ALiBi: the page's own prompt bias (arange(L)[None, :] - arange(L)[:, None]
    times the head's slope, under the causal mask) handed to torch SDPA;
  * the rotary step: RoFormer's complex-multiplication statement of the
    rotation, composition of rotations, relative-position invariance of the
    rotated dot product, linear position scaling and the neox / GPT-J pairing
    relation.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests._dense import brute_force, cu, paginate, random_dense

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# worked examples of the page (exact)
# ---------------------------------------------------------------------------

def test_varlen_example_token_to_request():
    g = _golden("varlen_example.json")
    assert list(np.cumsum([0] + g["q_lens"])) == g["cu_seq_lens_q"]
    assert list(np.cumsum([0] + g["k_lens"])) == g["cu_seq_lens_k"]
    assert max(g["q_lens"]) == g["max_length_q"] and max(g["k_lens"]) == g["max_length_k"]
    q_map = oracle.token_to_request(g["cu_seq_lens_q"], g["total_q"])
    k_map = oracle.token_to_request(g["cu_seq_lens_k"], g["total_k"])
    assert q_map.tolist() == g["q_request_index"]
    assert k_map.tolist() == g["k_request_index"]  # r0 has no key token


def test_decode_example_pages_and_new_token_slots():
    g = _golden("decode_example.json")
    bt, bs = g["block_table"], g["block_size"]
    for b, L in enumerate(g["cache_seqlens"]):
        # positions 0..L (cached tokens and the new one) live in the blocks
        # the page lists for the sequence
        blocks = {oracle.slot(bt, b, p, bs) // bs for p in range(L + 1)}
        assert blocks == set(g["blocks_listed_for_seq"][b])
        assert not blocks & set(g["blocks_never_owned"])
        # the new token (position L) lands where the page says
        s = oracle.slot(bt, b, L, bs)
        assert s // bs == g["new_token_block"][b]
        assert s % bs == g["new_token_offset_in_block"][b]
        assert s == g["new_token_slot"][b]


def test_decode_example_unallocated_entry_is_not_a_slot():
    g = _golden("decode_example.json")
    # position 32 of sequence 0 would need block_table[0][1] == -1
    assert oracle.slot(g["block_table"], 0, 32, g["block_size"]) == -1


def test_decode_example_never_reads_unowned_pages():
    """Pool blocks 4 and 7 (never owned in the example) hold NaN; the oracle's
    outputs stay finite, so it never reads them or a -1 entry."""
    from paged_kv_cache_attention_gb300 import workloads as W
    case = W.config1_tiny()
    out = oracle.paged_decode(W.to_oracle(case.q), W.to_oracle(case.k_cache),
                              W.to_oracle(case.v_cache), case.block_table.numpy(),
                              case.cache_seqlens.numpy(), sink=case.sink.numpy(),
                              sm_scale=case.sm_scale)
    assert np.isfinite(out).all()


# ---------------------------------------------------------------------------
# library routine: scaled_dot_product_attention in fp64
# ---------------------------------------------------------------------------

def _sdpa(q, k, v, scale, sink=None):
    """Causal prefill (q_len == kv_len) through torch SDPA in fp64.  With a
    sink, one extra key is appended whose value row is 0 and whose logit is
    sink[h] (given as an additive mask column): the sink column joins the
    softmax and contributes nothing to the output."""
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]  # [1,Hq,L,D]
    G = q.shape[1] // k.shape[1]
    kt = torch.from_numpy(k.astype(np.float64)).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    if sink is None:
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                             scale=scale)
    else:
        L, Hq = q.shape[0], q.shape[1]
        causal = torch.triu(torch.full((L, L), float("-inf"), dtype=torch.float64), 1)
        bias = torch.cat([causal[None].expand(Hq, L, L),
                          torch.from_numpy(sink.astype(np.float64))[:, None, None].expand(Hq, L, 1)],
                         dim=-1)[None]
        zk = torch.zeros(1, Hq, 1, q.shape[2], dtype=torch.float64)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, torch.cat([kt, zk], 2), torch.cat([vt, zk], 2), attn_mask=bias, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("Hq,Hkv,D,bs,lens", [
    (4, 4, 16, 4, [5, 9]),
    (4, 2, 32, 8, [17, 1, 33]),
    (8, 2, 64, 16, [40, 7]),
    (8, 1, 16, 16, [3, 50]),
])
@pytest.mark.parametrize("with_sink", [False, True])
def test_prefill_matches_sdpa(Hq, Hkv, D, bs, lens, with_sink):
    rng = np.random.default_rng(7 + Hq + D + len(lens))
    qd, kd, vd = random_dense(rng, lens, lens, Hq, Hkv, D)
    kp, vp, bt = paginate(kd, vd, bs, rng)
    sink = rng.standard_normal(Hq).astype(np.float32) * 2 if with_sink else None
    scale = 1.0 / math.sqrt(D)
    out = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(lens), np.array(lens, np.int32),
                           sink=sink, causal=True, sm_scale=scale)
    ref = np.concatenate([_sdpa(qd[r], kd[r], vd[r], scale, sink) for r in range(len(lens))])
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv,D,bs,q_lens,kv_lens", [
    (4, 4, 16, 4, [5, 9], [12, 3]),
    (8, 2, 64, 16, [40, 1], [7, 70]),
    (8, 1, 32, 8, [3, 20], [50, 20]),
])
def test_non_causal_prefill_matches_sdpa(Hq, Hkv, D, bs, q_lens, kv_lens):
    """Non-causal, no window: every query row attends to all of its request's
    keys whatever its position, which is SDPA with no mask (q_len may exceed
    kv_len or fall short of it)."""
    rng = np.random.default_rng(11 + Hq + D)
    qd, kd, vd = random_dense(rng, q_lens, kv_lens, Hq, Hkv, D)
    kp, vp, bt = paginate(kd, vd, bs, rng)
    scale = 1.0 / math.sqrt(D)
    out = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(q_lens),
                           np.array(kv_lens, np.int32), causal=False, sm_scale=scale)
    G = Hq // Hkv
    ref = []
    for r in range(len(q_lens)):
        qt = torch.from_numpy(qd[r].astype(np.float64)).permute(1, 0, 2)[None]
        kt = torch.from_numpy(kd[r].astype(np.float64)).repeat_interleave(G, 1).permute(1, 0, 2)[None]
        vt = torch.from_numpy(vd[r].astype(np.float64)).repeat_interleave(G, 1).permute(1, 0, 2)[None]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        ref.append(o[0].permute(1, 0, 2).numpy())
    np.testing.assert_allclose(out, np.concatenate(ref), rtol=0, atol=1e-12)


def test_sink_only_rescales():
    """With a sink the output is the plain output times one per-row factor in
    (0, 1): the sink adds to the denominator only."""
    rng = np.random.default_rng(3)
    qd, kd, vd = random_dense(rng, [6], [6], 4, 2, 32)
    kp, vp, bt = paginate(kd, vd, 8, rng)
    sink = np.array([0.5, -1.0, 2.0, 3.0], np.float32)
    args = (qd[0], kp, vp, bt, cu([6]), np.array([6], np.int32))
    plain = oracle.attention(*args, sink=None, sm_scale=0.2)
    with_s = oracle.attention(*args, sink=sink, sm_scale=0.2)
    ratio = with_s / plain
    assert np.all(ratio > 0) and np.all(ratio < 1)
    np.testing.assert_allclose(ratio, ratio[..., :1].repeat(32, -1), rtol=1e-12)


# ---------------------------------------------------------------------------
# closed forms and invariances
# ---------------------------------------------------------------------------

def test_window_zero_keeps_only_own_key():
    """window_left = 0: the query at position p keeps key p alone, so
    o = v_p * e^{s_p} / (e^{s_p} + e^{sink}) = v_p * sigmoid(s_p - sink)."""
    rng = np.random.default_rng(11)
    q_lens, kv_lens = [3, 1], [7, 5]
    qd, kd, vd = random_dense(rng, q_lens, kv_lens, 4, 2, 16)
    kp, vp, bt = paginate(kd, vd, 4, rng)
    sink = rng.standard_normal(4).astype(np.float32)
    scale = 0.3
    out = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(q_lens),
                           np.array(kv_lens, np.int32), sink=sink, window_left=0,
                           sm_scale=scale)
    row = 0
    for r in range(2):
        for i in range(q_lens[r]):
            p = kv_lens[r] - q_lens[r] + i
            for h in range(4):
                g = h // 2
                s = scale * float(np.dot(qd[r][i, h].astype(np.float64),
                                         kd[r][p, g].astype(np.float64)))
                w = 1.0 / (1.0 + math.exp(float(sink[h]) - s))
                np.testing.assert_allclose(out[row, h], w * vd[r][p, g].astype(np.float64),
                                           rtol=1e-13, atol=1e-14)
            row += 1


def test_window_at_least_kv_len_is_no_window():
    rng = np.random.default_rng(12)
    lens = [9, 20]
    qd, kd, vd = random_dense(rng, lens, lens, 4, 4, 16)
    kp, vp, bt = paginate(kd, vd, 4, rng)
    args = (np.concatenate(qd), kp, vp, bt, cu(lens), np.array(lens, np.int32))
    a = oracle.attention(*args, window_left=-1, sm_scale=0.25)
    b = oracle.attention(*args, window_left=20, sm_scale=0.25)
    c = oracle.attention(*args, window_left=1000, sm_scale=0.25)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_physical_relabelling_is_invisible():
    """Moving pages (and their block-table entries) leaves outputs bit-identical."""
    rng = np.random.default_rng(13)
    lens = [33, 17, 64]
    qd, kd, vd = random_dense(rng, [4, 1, 5], lens, 8, 2, 32)
    sink = rng.standard_normal(8).astype(np.float32)
    outs = []
    for seed in (1, 2, 3):
        kp, vp, bt = paginate(kd, vd, 16, np.random.default_rng(seed), spare=5)
        outs.append(oracle.attention(np.concatenate(qd), kp, vp, bt, cu([4, 1, 5]),
                                     np.array(lens, np.int32), sink=sink, window_left=9,
                                     sm_scale=0.17))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_page_size_is_invisible():
    rng = np.random.default_rng(14)
    lens = [70, 31]
    qd, kd, vd = random_dense(rng, [2, 3], lens, 4, 2, 16)
    res = []
    for bs in (16, 32, 1, 7):
        kp, vp, bt = paginate(kd, vd, bs, rng)
        res.append(oracle.attention(np.concatenate(qd), kp, vp, bt, cu([2, 3]),
                                    np.array(lens, np.int32), sm_scale=0.2))
    for r in res[1:]:
        assert np.array_equal(res[0], r)


def test_decode_is_last_row_of_prefill():
    rng = np.random.default_rng(15)
    lens = [12, 30]
    qd, kd, vd = random_dense(rng, lens, lens, 4, 2, 16)
    kp, vp, bt = paginate(kd, vd, 8, rng)
    sink = rng.standard_normal(4).astype(np.float32)
    full = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(lens), np.array(lens, np.int32),
                            sink=sink, window_left=5, sm_scale=0.3)
    last_q = np.stack([qd[0][-1], qd[1][-1]])
    dec = oracle.paged_decode(last_q, kp, vp, bt, np.array(lens, np.int32), sink=sink,
                              window_left=5, sm_scale=0.3)
    np.testing.assert_array_equal(dec[0], full[lens[0] - 1])
    np.testing.assert_array_equal(dec[1], full[sum(lens) - 1])


def test_chunk_is_suffix_of_longer_chunk():
    """A chunk of the last c queries over kv_len keys equals the last c rows of
    a longer chunk over the same keys (the causal mask is aligned to the end)."""
    rng = np.random.default_rng(16)
    kv = 40
    qd, kd, vd = random_dense(rng, [25], [kv], 4, 1, 16)
    kp, vp, bt = paginate(kd, vd, 16, rng)
    long_ = oracle.attention(qd[0], kp, vp, bt, cu([25]), np.array([kv], np.int32),
                             sm_scale=0.25, window_left=8)
    short = oracle.attention(qd[0][-6:], kp, vp, bt, cu([6]), np.array([kv], np.int32),
                             sm_scale=0.25, window_left=8)
    np.testing.assert_array_equal(short, long_[-6:])


# ---------------------------------------------------------------------------
# independent brute force on tiny inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_matches_bruteforce(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 5))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([8, 16, 64]))
    bs = int(rng.choice([1, 4, 16, 32]))
    kv_lens = [int(x) for x in rng.integers(0, 45, n)]
    q_lens = [int(rng.integers(0, 8)) for _ in range(n)]
    q_lens[0] = max(q_lens[0], 1)
    causal = bool(seed % 3 != 2)
    window = int(rng.choice([-1, 0, 3, 17]))
    sink = None if seed % 4 == 0 else (rng.standard_normal(Hkv * G) * 3).astype(np.float32)
    qd, kd, vd = random_dense(rng, q_lens, kv_lens, Hkv * G, Hkv, D)
    kp, vp, bt = paginate(kd, vd, bs, rng)
    alibi = (rng.uniform(0.01, 0.6, Hkv * G).astype(np.float32) if seed % 2 else None)
    out, lse = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(q_lens),
                                np.array(kv_lens, np.int32), sink=sink, causal=causal,
                                window_left=window, sm_scale=0.21, with_lse=True,
                                alibi_slopes=alibi)
    ref, ref_lse = brute_force(qd, kd, vd, sink, causal, window, 0.21, alibi=alibi)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse))
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)


def test_rows_with_no_key_are_zero():
    """kv_len = 0 (r0 of the varlen example), and rows whose position is
    negative because q_len > kv_len, attend to nothing: output 0."""
    rng = np.random.default_rng(17)
    q_lens, kv_lens = [3, 4], [0, 2]
    qd, kd, vd = random_dense(rng, q_lens, kv_lens, 2, 1, 8)
    kp, vp, bt = paginate([np.zeros((1, 1, 8), np.float32) if k.shape[0] == 0 else k for k in kd],
                          [np.zeros((1, 1, 8), np.float32) if v.shape[0] == 0 else v for v in vd],
                          4, rng)
    sink = np.array([0.3, -0.2], np.float32)
    out, lse = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(q_lens),
                                np.array(kv_lens, np.int32), sink=sink, sm_scale=0.5,
                                with_lse=True)
    assert np.all(out[:3] == 0)        # request 0: no keys at all
    assert np.all(out[3:5] == 0)       # request 1 rows 0,1: positions -2, -1
    assert np.all(out[5:] != 0)
    np.testing.assert_array_equal(lse[:5], np.broadcast_to(sink.astype(np.float64), (5, 2)))


# ---------------------------------------------------------------------------
# the cache write
# ---------------------------------------------------------------------------

def test_reshape_and_cache_places_rows_bit_exactly():
    g = _golden("decode_example.json")
    rng = np.random.default_rng(18)
    nb, bs, Hkv, D = 8, g["block_size"], 2, 64
    kc = np.full((nb, bs, Hkv, D), np.nan, np.float32)
    vc = np.full((nb, bs, Hkv, D), np.nan, np.float32)
    key = rng.standard_normal((4, Hkv, D)).astype(np.float32)
    val = rng.standard_normal((4, Hkv, D)).astype(np.float32)
    slots = np.array(g["new_token_slot"] + [-1], np.int64)  # last token is not cached
    oracle.reshape_and_cache(key, val, kc, vc, slots)
    flat_k = kc.reshape(nb * bs, Hkv, D)
    flat_v = vc.reshape(nb * bs, Hkv, D)
    for t, s in enumerate(g["new_token_slot"]):
        assert flat_k[s].tobytes() == key[t].tobytes()
        assert flat_v[s].tobytes() == val[t].tobytes()
    untouched = np.setdiff1d(np.arange(nb * bs), g["new_token_slot"])
    assert np.isnan(flat_k[untouched]).all() and np.isnan(flat_v[untouched]).all()


# ---------------------------------------------------------------------------
# rotary position embedding
# ---------------------------------------------------------------------------

def _rope_complex(x, pos, rd, base, scale, neox):
    """RoFormer's statement: the pair of frequency i, read as the complex
    number x_a + i x_b, is multiplied by exp(i * (m / scale) * base^(-2i/rd))."""
    x = x.astype(np.float64)
    out = x.copy()
    half = rd // 2
    idx = np.arange(half)
    a, b = (idx, idx + half) if neox else (2 * idx, 2 * idx + 1)
    z = x[..., a] + 1j * x[..., b]
    freq = np.power(float(base), -(2.0 * idx) / rd)
    rot = np.exp(1j * (np.asarray(pos, np.float64)[:, None] / scale) * freq[None, :])
    z = z * rot[:, None, :]
    out[..., a], out[..., b] = z.real, z.imag
    return out


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("D,rd,base,scale", [(64, 64, 10000.0, 1.0), (128, 64, 10000.0, 1.0),
                                             (80, 80, 500000.0, 4.0), (16, 8, 10.0, 2.0)])
def test_rope_matches_complex_rotation(neox, D, rd, base, scale):
    rng = np.random.default_rng(D + rd)
    x = rng.standard_normal((7, 3, D)).astype(np.float32)
    pos = np.array([0, 1, 2, 17, 1000, 32767, 131071], np.int64)
    got = oracle.rope(x, pos, rd, base=base, position_scale=scale, neox=neox)
    np.testing.assert_allclose(got, _rope_complex(x, pos, rd, base, scale, neox), rtol=0,
                               atol=1e-9)
    np.testing.assert_array_equal(got[..., rd:], x[..., rd:].astype(np.float64))
    np.testing.assert_array_equal(got[0], x[0].astype(np.float64))  # position 0: identity


def test_rope_bf16_input_widened_exactly():
    rng = np.random.default_rng(3)
    xf = rng.standard_normal((4, 2, 32)).astype(np.float32)
    bits = (xf.view(np.uint32) >> 16).astype(np.uint16)           # truncate to bf16
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    pos = np.array([3, 9, 27, 81])
    np.testing.assert_array_equal(oracle.rope(bits, pos, 32), oracle.rope(widened, pos, 32))


@pytest.mark.parametrize("neox", [True, False])
def test_rope_composes_and_is_relative(neox):
    """Rotations compose (rotating by a then by b is rotating by a+b) and the
    rotated dot product depends only on the distance of the two positions."""
    rng = np.random.default_rng(4)
    D = 32
    q32 = rng.standard_normal((1, 1, D)).astype(np.float32)
    k32 = rng.standard_normal((1, 1, D)).astype(np.float32)
    once = oracle.rope(oracle.rope(q32, [300], D, neox=neox).astype(np.float32), [45], D,
                       neox=neox)
    np.testing.assert_allclose(once, oracle.rope(q32, [345], D, neox=neox),
                               atol=1e-6)  # the intermediate was rounded to fp32
    dots = [float(np.sum(oracle.rope(q32, [m], D, neox=neox) *
                         oracle.rope(k32, [m - 13], D, neox=neox))) for m in (13, 50, 4000)]
    np.testing.assert_allclose(dots, dots[0], rtol=0, atol=1e-9)
    norms = np.linalg.norm(oracle.rope(q32, [777], D, neox=neox))
    assert abs(norms - np.linalg.norm(q32.astype(np.float64))) < 1e-12


def test_rope_linear_scaling_divides_the_position():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 2, 64)).astype(np.float32)
    a = oracle.rope(x, [10, 400, 9000], 64, position_scale=2.0)
    b = oracle.rope(x, [5, 200, 4500], 64, position_scale=1.0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("rd,alpha", [(64, 4.0), (128, 2.5), (16, 8.0)])
def test_rope_ntk_scaling_divides_the_lowest_frequency(rd, alpha):
    """NTK-aware scaling (the page's "dynamic" rope_scaling) raises the base so
    that the lowest frequency, i = rd/2 - 1, is divided by exactly alpha (its
    wavelength stretched alpha times) while the highest, i = 0, is kept.  The
    angle of each frequency is read back from the rotation of a unit vector
    (neox pair (i, i + rd/2)): x_a = 1, x_b = 0 turns into (cos, sin) of
    position * theta_i."""
    half = rd // 2
    x = np.zeros((half, 1, rd), np.float32)
    for i in range(half):
        x[i, 0, i] = 1.0

    def angles(m, a):
        out = oracle.rope(x, [m] * half, rd, ntk_alpha=a)
        return np.array([np.arctan2(out[i, 0, i + half], out[i, 0, i]) for i in range(half)])

    lo = half - 1
    m_lo = 2000  # position * theta_lo stays below pi for both bases
    assert abs(angles(m_lo, alpha)[lo] * alpha - angles(m_lo, 1.0)[lo]) < 1e-12
    assert abs(angles(3, alpha)[0] - 3.0) < 1e-12 and abs(angles(3, 1.0)[0] - 3.0) < 1e-12
    # every frequency in between is lowered, monotonically in i (position 3
    # keeps every angle below pi)
    r = angles(3, alpha)[1:] / angles(3, 1.0)[1:]
    assert np.all(r < 1.0) and np.all(np.diff(r) < 0)


def test_rope_neox_is_gptj_on_interleaved_dims():
    """neox pairs (i, i + rd/2); GPT-J pairs (2i, 2i+1): moving dim i to 2i and
    dim i + rd/2 to 2i + 1 turns one into the other."""
    rng = np.random.default_rng(6)
    D, rd = 48, 32
    x = rng.standard_normal((5, 2, D)).astype(np.float32)
    perm = np.arange(D)
    perm[:rd:2] = np.arange(rd // 2)
    perm[1:rd:2] = np.arange(rd // 2) + rd // 2
    pos = [1, 2, 3, 100, 12345]
    neox = oracle.rope(x, pos, rd, neox=True)
    gptj = oracle.rope(np.ascontiguousarray(x[..., perm]), pos, rd, neox=False)
    np.testing.assert_allclose(gptj, neox[..., perm], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# ALiBi
# ---------------------------------------------------------------------------

def _alibi_slopes(n):
    """The geometric slopes of the ALiBi paper for n heads: 2^(-8 i / n)."""
    return np.array([2.0 ** (-8.0 * (i + 1) / n) for i in range(n)], np.float32)


@pytest.mark.parametrize("Hq,Hkv,D,bs,lens", [(4, 4, 16, 4, [9, 30]), (8, 2, 32, 16, [40, 3]),
                                              (8, 1, 64, 8, [65])])
@pytest.mark.parametrize("with_sink", [False, True])
def test_alibi_prefill_matches_the_pages_bias_through_sdpa(Hq, Hkv, D, bs, lens, with_sink):
    """vLLM attention.py, PagedAttentionWithALiBi.set_attn_bias: for a prompt of
    length L the bias is (arange(L)[None, :] - arange(L)[:, None]) times each
    head's slope, added to the scaled scores under the lower-triangular mask.
    With a sink, one more key with a zero value row and logit sink[h]."""
    rng = np.random.default_rng(19 + Hq + D)
    qd, kd, vd = random_dense(rng, lens, lens, Hq, Hkv, D)
    kp, vp, bt = paginate(kd, vd, bs, rng)
    slopes = _alibi_slopes(Hq) * np.float32(3.0)  # steeper than the paper's, to matter
    sink = rng.standard_normal(Hq).astype(np.float32) if with_sink else None
    scale = 1.0 / math.sqrt(D)
    out = oracle.attention(np.concatenate(qd), kp, vp, bt, cu(lens), np.array(lens, np.int32),
                           sink=sink, causal=True, sm_scale=scale, alibi_slopes=slopes)
    G = Hq // Hkv
    ref = []
    for r, L in enumerate(lens):
        b = torch.arange(L, dtype=torch.float64)
        bias = (b[None, :] - b[:, None])[None] * torch.from_numpy(slopes.astype(np.float64))[:, None, None]
        bias = bias.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1)[None], float("-inf"))
        qt = torch.from_numpy(qd[r].astype(np.float64)).permute(1, 0, 2)[None]
        kt = torch.from_numpy(kd[r].astype(np.float64)).repeat_interleave(G, 1).permute(1, 0, 2)[None]
        vt = torch.from_numpy(vd[r].astype(np.float64)).repeat_interleave(G, 1).permute(1, 0, 2)[None]
        if sink is not None:
            col = torch.from_numpy(sink.astype(np.float64))[:, None, None].expand(Hq, L, 1)
            bias = torch.cat([bias, col], -1)
            z = torch.zeros(1, Hq, 1, D, dtype=torch.float64)
            kt, vt = torch.cat([kt, z], 2), torch.cat([vt, z], 2)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=bias[None],
                                                             scale=scale)
        ref.append(o[0].permute(1, 0, 2).numpy())
    np.testing.assert_allclose(out, np.concatenate(ref), rtol=0, atol=1e-12)


def test_alibi_zero_slopes_is_no_alibi():
    rng = np.random.default_rng(20)
    qd, kd, vd = random_dense(rng, [5, 20], [30, 20], 4, 2, 16)
    kp, vp, bt = paginate(kd, vd, 4, rng)
    args = (np.concatenate(qd), kp, vp, bt, cu([5, 20]), np.array([30, 20], np.int32))
    a = oracle.attention(*args, sm_scale=0.3)
    b = oracle.attention(*args, sm_scale=0.3, alibi_slopes=np.zeros(4, np.float32))
    np.testing.assert_array_equal(a, b)


def test_alibi_decode_is_the_last_prompt_row():
    """The decode query at position L-1 sees bias slope * (j - (L-1)): the
    last row of the prompt's bias matrix."""
    rng = np.random.default_rng(21)
    L, Hq, Hkv, D = 37, 8, 2, 32
    qd, kd, vd = random_dense(rng, [L], [L], Hq, Hkv, D)
    kp, vp, bt = paginate(kd, vd, 8, rng)
    slopes = _alibi_slopes(Hq)
    full = oracle.attention(qd[0], kp, vp, bt, cu([L]), np.array([L], np.int32),
                            sm_scale=0.2, alibi_slopes=slopes)
    dec = oracle.paged_decode(np.ascontiguousarray(qd[0][-1:]), kp, vp, bt,
                              np.array([L], np.int32), sm_scale=0.2, alibi_slopes=slopes)
    np.testing.assert_allclose(dec[0], full[-1], rtol=0, atol=1e-13)


def test_alibi_identical_keys_give_geometric_weights():
    """All keys equal: the softmax weights of a decode query are proportional
    to exp(slope * j), so with value rows e_j the output is that geometric
    distribution (closed form)."""
    L, D = 6, 8
    q = np.ones((1, 1, D), np.float32)
    k = np.tile(np.full((1, 1, D), 0.5, np.float32), (L, 1, 1))
    v = np.zeros((L, 1, D), np.float32)
    v[np.arange(L), 0, np.arange(L)] = 1.0
    kp, vp, bt = paginate([k], [v], 4, np.random.default_rng(22))
    slope = 0.7
    out = oracle.paged_decode(q, kp, vp, bt, np.array([L], np.int32), sm_scale=0.3,
                              alibi_slopes=np.array([slope], np.float32))
    w = np.exp(np.float64(np.float32(slope)) * np.arange(L))
    np.testing.assert_allclose(out[0, 0, :L], w / w.sum(), rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# MInference vertical + slash sparse prefill
# ---------------------------------------------------------------------------

def _numpy_pattern_scores(q, k, last_q, scale):
    """Independent dense statement: softmax rows of the last queries (causal),
    summed per key column and per diagonal pos - j."""
    S, Hq, D = q.shape
    G = Hq // k.shape[1]
    kk = np.repeat(k.astype(np.float64), G, axis=1)
    lq = min(last_q, S)
    pos = np.arange(S - lq, S)
    qk = np.einsum("qhd,khd->hqk", q[S - lq:].astype(np.float64), kk) * scale
    col = np.arange(S)[None, :]
    qk = np.where((col <= pos[:, None])[None], qk, -np.inf)
    p = np.exp(qk - qk.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    vert = p.sum(1)
    slash = np.zeros((Hq, S))
    diag = np.broadcast_to(pos[:, None] - col, (lq, S))
    for h in range(Hq):
        ok = col.repeat(lq, 0) <= pos[:, None]
        np.add.at(slash[h], diag[ok], p[h][ok])
    return vert, slash


@pytest.mark.parametrize("S,Hq,Hkv,D", [(200, 4, 2, 16), (64, 2, 1, 32), (37, 4, 4, 8),
                                        (130, 8, 2, 16)])
def test_minference_scores_match_numpy(S, Hq, Hkv, D):
    rng = np.random.default_rng(S + Hq)
    q = rng.standard_normal((S, Hq, D)).astype(np.float32)
    k = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    scale = 1.0 / math.sqrt(D)
    vert, slash = oracle.minference_scores(q, k, 64, scale)
    rv, rs = _numpy_pattern_scores(q, k, 64, scale)
    np.testing.assert_allclose(vert, rv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(slash, rs, rtol=0, atol=1e-12)
    # each softmax row sums to one: both score vectors sum to the number of
    # estimating queries
    np.testing.assert_allclose(vert.sum(1), min(64, S), rtol=1e-12)
    np.testing.assert_allclose(slash.sum(1), min(64, S), rtol=1e-12)


def test_minference_sizes_follow_the_budget():
    # S = 1000, budget 0.3: b = 300, vertical max(31, 60), slash max(101, 240)
    assert oracle.minference_sizes(1000) == (60, 240)
    # S = 100: b = 30; the floors 31 and 101, the latter capped at S
    assert oracle.minference_sizes(100) == (31, 100)
    # no adaptive budget: the fixed sizes, capped at S
    assert oracle.minference_sizes(5000, adaptive_budget=None) == (1000, 5000)
    assert oracle.minference_sizes(20000, adaptive_budget=None) == (1000, 6096)


def test_minference_selection_keeps_sinks_and_recent_diagonals():
    rng = np.random.default_rng(23)
    S = 500
    q = rng.standard_normal((S, 4, 16)).astype(np.float32)
    k = rng.standard_normal((S, 2, 16)).astype(np.float32)
    vi, si, vs, ss = oracle.minference_pattern(q, k)
    nv, ns = oracle.minference_sizes(S)
    assert vi.shape == (4, nv) and si.shape == (4, ns)
    for h in range(4):
        assert np.all(np.diff(vi[h]) > 0) and np.all(np.diff(si[h]) > 0)  # sorted, unique
        assert set(range(30)) <= set(vi[h].tolist())
        assert set(range(100)) <= set(si[h].tolist())
        # every kept (unforced) index scores at least as much as every dropped one
        free_v = [j for j in vi[h] if j >= 30]
        drop_v = np.setdiff1d(np.arange(30, S), vi[h])
        assert vs[h][free_v].min() >= vs[h][drop_v].max()
        free_s = [d for d in si[h] if d >= 100]
        drop_s = np.setdiff1d(np.arange(100, S), si[h])
        assert ss[h][free_s].min() >= ss[h][drop_s].max()


def test_sparse_attention_with_every_key_vertical_is_dense_causal():
    rng = np.random.default_rng(24)
    S, Hq, Hkv, D = 90, 4, 2, 16
    q = rng.standard_normal((S, Hq, D)).astype(np.float32)
    k = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    allv = np.tile(np.arange(S, dtype=np.int32), (Hq, 1))
    none_s = np.zeros((Hq, 0), np.int32)
    out = oracle.sparse_attention(q, k, v, allv, none_s, scale=0.25)
    kp, vp, bt = paginate([k], [v], 8, rng)
    ref = oracle.attention(q, kp, vp, bt, cu([S]), np.array([S], np.int32), causal=True,
                           sm_scale=0.25)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # every diagonal as a slash line is the same mask
    alls = np.tile(np.arange(S, dtype=np.int32), (Hq, 1))
    out2 = oracle.sparse_attention(q, k, v, np.zeros((Hq, 0), np.int32), alls, scale=0.25)
    np.testing.assert_allclose(out2, ref, rtol=0, atol=1e-12)


def test_sparse_attention_main_diagonal_only_returns_own_value():
    rng = np.random.default_rng(25)
    S, Hq, Hkv, D = 40, 4, 2, 8
    q = rng.standard_normal((S, Hq, D)).astype(np.float32)
    k = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    out = oracle.sparse_attention(q, k, v, np.zeros((Hq, 0), np.int32),
                                  np.zeros((Hq, 1), np.int32))
    np.testing.assert_array_equal(out, np.repeat(v.astype(np.float64), 2, axis=1))


@pytest.mark.parametrize("seed", range(4))
def test_sparse_attention_matches_numpy_bruteforce(seed):
    rng = np.random.default_rng(30 + seed)
    S, Hq, Hkv, D = 70, 4, 2, 16
    q = rng.standard_normal((S, Hq, D)).astype(np.float32)
    k = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((S, Hkv, D)).astype(np.float32)
    vi = np.sort(np.stack([rng.choice(S, 9, replace=False) for _ in range(Hq)]), 1).astype(np.int32)
    si = np.sort(np.stack([rng.choice(S, 13, replace=False) for _ in range(Hq)]), 1).astype(np.int32)
    out = oracle.sparse_attention(q, k, v, vi, si, scale=0.3)
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    kk = np.repeat(k.astype(np.float64), 2, axis=1)
    vv = np.repeat(v.astype(np.float64), 2, axis=1)
    for h in range(Hq):
        keep = (j <= i) & (np.isin(j, vi[h]) | np.isin(i - j, si[h]))
        s = np.where(keep, q[:, h].astype(np.float64) @ kk[:, h].T * 0.3, -np.inf)
        m = s.max(1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m)
        z = e.sum(1, keepdims=True)
        ref = np.where(z > 0, (e @ vv[:, h]) / np.where(z > 0, z, 1), 0.0)
        np.testing.assert_allclose(out[:, h], ref, rtol=0, atol=1e-12)
