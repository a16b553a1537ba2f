"""The HND pool layout ([num_blocks, Hkv, block_size, D]) on the GPU.

Each case is built in the NHD layout, its pools re-indexed to HND, and the
GPU result compared with the fp64 oracle on the NHD original (the layout is
addressing only), and with the NHD GPU path bit for bit (same tiles, same
arithmetic order).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import (LSE_TOL, TOL, dev, from_hnd, gpu_decode, gpu_prefill, lse_err,
                        max_abs, oracle_decode, oracle_prefill, to_hnd)

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()


@pytest.mark.parametrize("dtype", [torch.float32, BF16])
def test_cache_write_hnd_is_bit_exact(dtype):
    case = W.make_mixed([100, 513, 2000], 64, 128, 2, 32, 8, 128, 16, dtype, seed=5)
    d = dev()
    kc, vc = to_hnd(case.k_cache).to(d), to_hnd(case.v_cache).to(d)
    slots = case.slot_mapping.clone()
    slots[::5] = -1  # some tokens are not cached
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.reshape_and_cache(case.key.to(d), case.value.to(d), kc, vc, slots.to(d), dev_error=err,
                          layout="HND")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ok, ov = W.to_oracle(case.k_cache).copy(), W.to_oracle(case.v_cache).copy()
    oracle.reshape_and_cache(W.to_oracle(case.key), W.to_oracle(case.value), ok, ov,
                             slots.numpy())
    g_k, g_v = _bits(from_hnd(kc.cpu())), _bits(from_hnd(vc.cpu()))
    assert np.array_equal(g_k, ok.view(g_k.dtype).reshape(g_k.shape))
    assert np.array_equal(g_v, ov.view(g_v.dtype).reshape(g_v.shape))


@pytest.mark.parametrize("Hq,Hkv,D,bs,window,alibi", [(32, 8, 128, 16, -1, "none"),
                                                      (16, 2, 64, 32, 300, "uniform"),
                                                      (8, 8, 256, 16, -1, "geometric"),
                                                      (32, 2, 96, 32, 1000, "none")])
def test_decode_hnd(Hq, Hkv, D, bs, window, alibi):
    lens = [1, 16, 17, 511, 513, 3000]
    case = W.make_decode(lens, Hq, Hkv, D, bs, BF16, seed=Hq + D + bs, sink="randn",
                         window_left=window, alibi=alibi)
    got, glse = gpu_decode(case, with_lse=True, layout="HND")
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[BF16]
    assert lse_err(glse, rlse) <= LSE_TOL[BF16]
    assert np.array_equal(got, gpu_decode(case, layout="NHD"))


def test_decode_hnd_fp32():
    case = W.make_decode([1, 31, 70, 300], 4, 2, 64, 32, torch.float32, seed=7, sink="randn")
    got = gpu_decode(case, layout="HND")
    assert max_abs(got, oracle_decode(case)) <= TOL[torch.float32]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("G,Hkv,bs,D", [(4, 8, 16, 128), (1, 4, 32, 80), (16, 1, 16, 128)])
def test_prefill_hnd(causal, G, Hkv, bs, D):
    q_lens = [1, 33, 129, 300]
    kv_lens = [1, 333, 1000, 300]
    case = W.make_varlen_kv(q_lens, kv_lens, G * Hkv, Hkv, D, bs, BF16, seed=G + bs + D,
                            sink="randn", causal=causal,
                            alibi="geometric" if G == 16 else "none")
    got, glse = gpu_prefill(case, with_lse=True, layout="HND")
    ref, rlse = oracle_prefill(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[BF16]
    assert lse_err(glse, rlse) <= LSE_TOL[BF16]
    assert np.array_equal(got, gpu_prefill(case, layout="NHD"))


def test_rope_hnd_writes_the_same_pages():
    case = W.make_rope(300, 16, 4, 128, 64, 16, BF16, seed=8)
    d = dev()
    tab = pkv.rope_cos_sin_table(case.max_position, 64)
    outs = {}
    for layout in ("NHD", "HND"):
        q, k, v = case.query.to(d), case.key.to(d), case.value.to(d)
        kc = (to_hnd(case.k_cache) if layout == "HND" else case.k_cache).to(d)
        vc = (to_hnd(case.v_cache) if layout == "HND" else case.v_cache).to(d)
        pkv.rope_reshape_and_cache(q, k, v, kc, vc, case.positions.to(d),
                                   case.slot_mapping.to(d), tab, layout=layout)
        torch.cuda.synchronize()
        if layout == "HND":
            kc, vc = from_hnd(kc.cpu()), from_hnd(vc.cpu())
        outs[layout] = (_bits(q), _bits(k), _bits(kc), _bits(vc))
    for a, b in zip(outs["NHD"], outs["HND"]):
        assert np.array_equal(a, b)
    # and the NHD result is the oracle's rotation (checked in test_gpu_rope);
    # here its value rows are the oracle's bit copy
    ok, ov = W.to_oracle(case.k_cache).copy(), W.to_oracle(case.v_cache).copy()
    oracle.reshape_and_cache(W.to_oracle(case.key), W.to_oracle(case.value), ok, ov,
                             case.slot_mapping.numpy())
    assert np.array_equal(outs["HND"][3].reshape(-1), ov.view(np.int16).reshape(-1))
