"""rope_reshape_and_cache on the GPU against the fp64 oracle.

The rotated query and key are floating point: each GPU value must lie within
one unit in the last place of the dtype of the exactly rotated value (fp32
arithmetic, rounded once), and inside the spec bars (2e-2 bf16, 1e-5
fp32).  Everything else is index and copy work and must be bit-exact: the
dimensions past rotary_dim, the value rows, which slots are written, and every
slot that is not.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import TOL, dev, gpu_decode, max_abs, oracle_decode

pytestmark = pytest.mark.gpu
ULP_REL = {torch.bfloat16: 2.0 ** -7, torch.float32: 2.0 ** -23}


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()


def _run(case, err=None):
    d = dev()
    q, k, v = case.query.to(d), case.key.to(d), case.value.to(d)
    kc, vc = case.k_cache.to(d), case.v_cache.to(d)
    tab = pkv.rope_cos_sin_table(case.max_position, case.rotary_dim, case.base,
                                 case.position_scale, ntk_alpha=case.ntk_alpha)
    pkv.rope_reshape_and_cache(q, k, v, kc, vc, case.positions.to(d), case.slot_mapping.to(d),
                               tab, case.rotary_dim, case.neox, dev_error=err)
    torch.cuda.synchronize()
    return q.cpu(), k.cpu(), kc.cpu(), vc.cpu()


def _oracle_rot(case, x):
    return oracle.rope(W.to_oracle(x), case.positions.numpy(), case.rotary_dim, base=case.base,
                       position_scale=case.position_scale, neox=case.neox,
                       ntk_alpha=case.ntk_alpha)


def _assert_rotated(case, got, x, ref):
    """got: GPU result [T, H, D]; x: input; ref: oracle fp64 rotation of x.
    Bound: one unit in the last place of the dtype, plus the fp32 rounding of
    the products when the two terms nearly cancel."""
    rd = case.rotary_dim
    g = got.float().numpy().astype(np.float64)
    err = np.abs(g[..., :rd] - ref[..., :rd])
    bound = ULP_REL[x.dtype] * np.abs(ref[..., :rd]) + 4e-6
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"
    assert err.max() <= TOL[x.dtype]
    assert np.array_equal(_bits(got)[..., rd:], _bits(x)[..., rd:])  # untouched dims


def _check_case(case):
    q, k, kc, vc = _run(case)
    ref_q, ref_k = _oracle_rot(case, case.query), _oracle_rot(case, case.key)
    _assert_rotated(case, q, case.query, ref_q)
    _assert_rotated(case, k, case.key, ref_k)
    slots = case.slot_mapping.numpy()
    cached = np.nonzero(slots >= 0)[0]
    H, D = case.key.shape[1:]
    kflat = kc.reshape(-1, H, D)
    # key rows in the cache: the oracle's rotation (to one ulp) and the very
    # bits of the in-place rotated key
    _assert_rotated(case, kflat[slots[cached]], case.key[cached], ref_k[cached])
    assert np.array_equal(_bits(kflat[slots[cached]]), _bits(k[cached]))
    # slots nobody writes keep their bits (NaN)
    untouched = np.setdiff1d(np.arange(kflat.shape[0]), slots[cached])
    assert np.array_equal(_bits(kflat[untouched]),
                          _bits(case.k_cache.reshape(-1, H, D)[untouched]))
    # value rows: the oracle's bit copy of the input values
    ok = W.to_oracle(case.k_cache).copy()
    ov = W.to_oracle(case.v_cache).copy()
    oracle.reshape_and_cache(W.to_oracle(case.key), W.to_oracle(case.value), ok, ov, slots)
    assert np.array_equal(_bits(vc).reshape(-1), ov.view(_bits(vc).dtype).reshape(-1))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("Hq,Hkv,D,rd", [(32, 8, 128, 128), (8, 2, 64, 32), (16, 4, 80, 80),
                                         (4, 1, 256, 64), (12, 4, 96, 48)])
def test_rope_cache_matches_oracle(dtype, neox, Hq, Hkv, D, rd):
    if dtype == torch.bfloat16 and rd % 16:
        pytest.skip("bf16 rotary_dim must be a multiple of 16")
    case = W.make_rope(300, Hq, Hkv, D, rd, 16, dtype, seed=D + rd + int(neox), neox=neox)
    _check_case(case)


@pytest.mark.parametrize("base,scale,ntk,max_pos", [(10000.0, 1.0, 1.0, 131072),
                                                    (500000.0, 8.0, 1.0, 32768),
                                                    (10000.0, 1.0, 4.0, 16384),
                                                    (10000.0, 2.0, 2.5, 65536)])
def test_rope_long_positions_and_scaling(base, scale, ntk, max_pos):
    """Angles up to ~1.3e5 rad: the fp64-built table keeps the rotation exact
    to fp32 rounding even there; linear and NTK-aware scaling (the table's
    ntk_alpha against the oracle's own NTK base) included."""
    case = W.make_rope(512, 8, 2, 128, 128, 32, torch.bfloat16, seed=int(scale + ntk) + 7,
                       max_position=max_pos, base=base, position_scale=scale, ntk_alpha=ntk)
    _check_case(case)


def test_rope_table_is_fp64_rounded_once():
    tab = pkv.rope_cos_sin_table(131072, 64, 10000.0, 2.0).cpu().numpy().astype(np.float64)
    pos = np.arange(131072, dtype=np.float64)[:, None] / 2.0
    ang = pos * np.power(10000.0, -2.0 * np.arange(32) / 64)[None, :]
    # fp32 rounding of cos/sin in [-1, 1]: at most 2^-25, plus the fp64 error
    # of angles up to 6.6e4 rad (~1e-11)
    assert np.abs(tab[..., 0] - np.cos(ang)).max() <= 2.0 ** -25 + 1e-10
    assert np.abs(tab[..., 1] - np.sin(ang)).max() <= 2.0 ** -25 + 1e-10


def test_rope_bad_positions_and_slots_are_flagged():
    case = W.make_rope(64, 8, 2, 64, 64, 16, torch.bfloat16, seed=3, max_position=1000,
                       skip_every=0)
    case.positions[5] = -1
    case.positions[9] = 1000
    capacity = case.k_cache.shape[0] * case.k_cache.shape[1]
    case.slot_mapping[20] = capacity + 3
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    q, k, kc, vc = _run(case, err)
    e = int(err.item())
    assert e & pkv.DEVERR_POSITION and e & pkv.DEVERR_SLOT
    for t in (5, 9):  # untouched: query, key and their slots
        assert torch.equal(q[t], case.query[t]) and torch.equal(k[t], case.key[t])
        s = int(case.slot_mapping[t])
        assert torch.isnan(kc.view(-1, 2, 64)[s].float()).all()
        assert torch.isnan(vc.view(-1, 2, 64)[s].float()).all()
    # token 20 is rotated but not cached
    ref = _oracle_rot(case, case.query)
    assert np.abs(q[20].float().numpy() - ref[20]).max() <= TOL[torch.bfloat16]
    good = [t for t in range(64) if t not in (5, 9, 20)]
    assert np.abs(q[good].float().numpy() - ref[good]).max() <= TOL[torch.bfloat16]


def test_rope_without_query():
    case = W.make_rope(50, 4, 2, 128, 64, 16, torch.bfloat16, seed=4)
    d = dev()
    k, v = case.key.to(d), case.value.to(d)
    kc, vc = case.k_cache.to(d), case.v_cache.to(d)
    tab = pkv.rope_cos_sin_table(case.max_position, 64)
    pkv.rope_reshape_and_cache(None, k, v, kc, vc, case.positions.to(d),
                               case.slot_mapping.to(d), tab)
    torch.cuda.synchronize()
    _assert_rotated(case, k.cpu(), case.key, _oracle_rot(case, case.key))


def test_rope_then_decode_matches_oracle():
    """Cross-op: rotate and write each sequence's new token, then decode with
    the rotated queries; the oracle rotates the same inputs in fp64, stores the
    key rounded to bf16 and attends."""
    dec = W.make_decode([37, 600, 1029, 4096], 32, 8, 128, 16, torch.bfloat16, seed=31,
                        sink="randn")
    B = dec.batch
    gen = torch.Generator().manual_seed(32)
    key = torch.randn(B, 8, 128, generator=gen).to(torch.bfloat16)
    val = torch.randn(B, 8, 128, generator=gen).to(torch.bfloat16)
    pos = (dec.cache_seqlens - 1).to(torch.int64)  # the new token is the last attended one
    bs = 16
    slots = torch.tensor([int(dec.block_table[b, int(pos[b]) // bs]) * bs + int(pos[b]) % bs
                          for b in range(B)], dtype=torch.int64)
    d = dev()
    q, k, v = dec.q.to(d), key.to(d), val.to(d)
    kc, vc = dec.k_cache.to(d), dec.v_cache.to(d)
    tab = pkv.rope_cos_sin_table(8192, 128)
    pkv.rope_reshape_and_cache(q, k, v, kc, vc, pos.to(d), slots.to(d), tab)
    torch.cuda.synchronize()
    gpu_case = W.DecodeCase(dec.name, q.cpu(), kc.cpu(), vc.cpu(), dec.block_table,
                            dec.cache_seqlens, dec.sink, dec.window_left, dec.sm_scale)
    got = gpu_decode(gpu_case)
    # oracle side, from the original inputs
    q_rot = oracle.rope(W.to_oracle(dec.q), pos.numpy(), 128)
    k_rot = oracle.rope(W.to_oracle(key), pos.numpy(), 128)
    ref_case = W.DecodeCase(dec.name, torch.from_numpy(q_rot).to(torch.bfloat16),
                            dec.k_cache.clone(), dec.v_cache.clone(), dec.block_table,
                            dec.cache_seqlens, dec.sink, dec.window_left, dec.sm_scale)
    kflat = ref_case.k_cache.view(-1, 8, 128)
    vflat = ref_case.v_cache.view(-1, 8, 128)
    kflat[slots] = torch.from_numpy(k_rot).to(torch.bfloat16)
    vflat[slots] = val
    ref = oracle_decode(ref_case)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]


def test_mixed_step_tokens_full_size():
    """All 8448 new tokens of the mixed continuous batch (decode tokens at
    their cache length, prefill chunks at prefix + i)."""
    mc = W.config5_mixed()
    case = W.RopeCase("mixed", W.randn((mc.num_new_tokens, 32, 128), torch.bfloat16,
                                       torch.Generator().manual_seed(33)),
                      mc.key, mc.value, mc.k_cache, mc.v_cache, mc.positions, mc.slot_mapping,
                      128, 10000.0, 1.0, True, 32768)
    _check_case(case)
