"""reshape_and_cache on the GPU: bit-exact against the oracle's row copy."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import dev

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().copy() if t.dtype == torch.bfloat16 \
        else t.view(torch.int32).numpy().copy()


def _run_both(key, value, kc, vc, slots):
    d = dev()
    gk, gv = kc.to(d), vc.to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.reshape_and_cache(key.to(d), value.to(d), gk, gv, slots.to(d), dev_error=err)
    torch.cuda.synchronize()
    ok, ov = W.to_oracle(kc).copy(), W.to_oracle(vc).copy()
    oracle.reshape_and_cache(W.to_oracle(key), W.to_oracle(value), ok, ov, slots.numpy())
    return gk, gv, ok, ov, int(err.item())


def _same_bits(gpu_t, oracle_arr):
    g = _bits(gpu_t)
    o = oracle_arr.view(np.int16 if oracle_arr.dtype == np.uint16 else np.int32)
    return np.array_equal(g, o.reshape(g.shape))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_example_new_token_slots(dtype):
    """The transformers-docs decode example: the three new tokens land at
    slots 94, 32 and 198 of an 8-page pool with pages 4 and 7 unowned."""
    g = json.load(open(os.path.join(GOLDEN, "decode_example.json")))
    gen = torch.Generator().manual_seed(1)
    shape = (8, g["block_size"], 2, 64)
    kc = torch.full(shape, float("nan"), dtype=dtype)
    vc = torch.full(shape, float("nan"), dtype=dtype)
    key = torch.randn(3, 2, 64, generator=gen).to(dtype)
    val = torch.randn(3, 2, 64, generator=gen).to(dtype)
    slots = torch.tensor(g["new_token_slot"], dtype=torch.int64)
    gk, gv, ok, ov, err = _run_both(key, val, kc, vc, slots)
    assert err == 0
    assert _same_bits(gk, ok) and _same_bits(gv, ov)
    flat = gk.view(-1, 2, 64).cpu()
    for t, s in enumerate(g["new_token_slot"]):
        assert torch.equal(flat[s], key[t])


def test_mixed_step_write_is_bit_exact():
    """All 8448 new tokens of the mixed continuous batch (2 KB rows)."""
    case = W.config5_mixed()
    gk, gv, ok, ov, err = _run_both(case.key, case.value, case.k_cache, case.v_cache,
                                    case.slot_mapping)
    assert err == 0
    assert _same_bits(gk, ok) and _same_bits(gv, ov)


def test_negative_slots_skip_and_out_of_pool_flags():
    gen = torch.Generator().manual_seed(2)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    key = torch.randn(5, 2, 64, generator=gen).to(torch.bfloat16)
    val = torch.randn(5, 2, 64, generator=gen).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 63, 64, 10_000], dtype=torch.int64)
    d = dev()
    gk, gv = kc.to(d), vc.to(d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.reshape_and_cache(key.to(d), val.to(d), gk, gv, slots.to(d), dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_SLOT
    # the oracle receives only the in-pool part
    ok, ov = W.to_oracle(kc).copy(), W.to_oracle(vc).copy()
    oracle.reshape_and_cache(W.to_oracle(key), W.to_oracle(val), ok, ov,
                             np.array([3, -1, 63, -1, -1], np.int64))
    assert _same_bits(gk, ok) and _same_bits(gv, ov)


def test_zero_tokens_is_a_no_op():
    d = dev()
    kc = torch.zeros(2, 16, 1, 64, dtype=torch.bfloat16, device=d)
    e = torch.empty(0, 1, 64, dtype=torch.bfloat16, device=d)
    pkv.reshape_and_cache(e, e, kc, kc.clone(), torch.empty(0, dtype=torch.int64, device=d))
    torch.cuda.synchronize()
    assert int(kc.abs().sum()) == 0
