"""paged_decode on the GPU against the fp64 oracle on the same seeded inputs.

Bars: max-abs error 1e-5 (fp32) / 2e-2 (bf16) on outputs; lse within 1e-5 /
2e-3.  Pool pages no sequence owns hold NaN, so a stray read fails the test.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import (LSE_TOL, TOL, dev, gpu_decode, lse_err, max_abs, oracle_decode,
                        to_dev)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------------------
# the tiny fp32 worked example
# ---------------------------------------------------------------------------

def test_tiny_fp32_example_attend():
    case = W.config1_tiny()
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.float32]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.float32]


def test_tiny_fp32_example_append_then_attend():
    """Write each sequence's new token (slots 94, 32, 198) with
    reshape_and_cache, then attend over [31, 33, 71]."""
    case = W.config1_tiny()
    d = dev()
    kc, vc = case.k_cache.to(d), case.v_cache.to(d)
    slots = torch.tensor([94, 32, 198], dtype=torch.int64, device=d)
    pkv.reshape_and_cache(case.new_k.to(d), case.new_v.to(d), kc, vc, slots)
    torch.cuda.synchronize()
    case.k_cache, case.v_cache = kc.cpu(), vc.cpu()
    case.cache_seqlens = case.cache_seqlens + 1
    got = gpu_decode(case)
    ref = oracle_decode(case)
    assert max_abs(got, ref) <= TOL[torch.float32]


# ---------------------------------------------------------------------------
# bf16 tensor-core path: shapes, ragged tails, windows, sinks, partitions
# ---------------------------------------------------------------------------

SHAPES = [
    # (Hq, Hkv, D, bs)
    (32, 8, 128, 16),
    (64, 8, 64, 16),
    (8, 8, 128, 32),
    (16, 2, 64, 32),
    (32, 2, 128, 16),   # G = 16
    (6, 2, 64, 16),     # G = 3
]


@pytest.mark.parametrize("Hq,Hkv,D,bs", SHAPES)
@pytest.mark.parametrize("sink", ["none", "randn"])
def test_bf16_shapes(Hq, Hkv, D, bs, sink):
    lens = [1, 15, 16, 17, 511, 512, 513, 1500]
    case = W.make_decode(lens, Hq, Hkv, D, bs, torch.bfloat16, seed=Hq * 7 + D + bs, sink=sink)
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.bfloat16]


@pytest.mark.parametrize("window", [0, 1, 5, 127, 511, 512, 1000, 5000])
def test_bf16_windows(window):
    lens = [1, 40, 512, 700, 2049, 3000]
    case = W.make_decode(lens, 16, 4, 64, 16, torch.bfloat16, seed=window + 3, sink="randn",
                         window_left=window)
    got = gpu_decode(case)
    ref = oracle_decode(case)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("part", [16, 32, 64, 512, 1024, 16384])
def test_bf16_partition_sizes(part):
    lens = [3, 100, 1000, 4000]
    case = W.make_decode(lens, 32, 8, 128, 16, torch.bfloat16, seed=part, sink="randn")
    got = gpu_decode(case, partition_size=part)
    ref = oracle_decode(case)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("D,window,sink", [(128, -1, "randn"), (64, 300, "randn"), (128, 0, "none")])
def test_many_heads_batch(D, window, sink):
    """A batch with many (sequence, head) pairs and few partitions each takes
    the warp-per-head merge; it must agree with the oracle like the
    CTA-per-head merge, including empty and one-token sequences."""
    gen = torch.Generator().manual_seed(D + window)
    lens = torch.randint(0, 3000, (64,), generator=gen).tolist()
    lens[:4] = [0, 1, 512, 513]
    case = W.make_decode(lens, 32, 8, D, 16, torch.bfloat16, seed=D * 3 + window, sink=sink,
                         window_left=window)
    got, glse = gpu_decode(case, with_lse=True)
    rows = list(range(0, 64, 3)) + [0, 1, 2, 3]
    ref, rlse = oracle_decode(case, rows=rows, with_lse=True)
    assert max_abs(got[rows], ref) <= TOL[torch.bfloat16]
    assert lse_err(glse[rows], rlse) <= LSE_TOL[torch.bfloat16]


def test_partition_size_invariance():
    """Split-KV is exact up to fp32 rounding: 512-token partitions and one
    partition for the whole sequence agree far inside the bf16 bar."""
    case = W.make_decode([5000, 333, 4096], 32, 8, 128, 16, torch.bfloat16, seed=9,
                         sink="randn")
    a = gpu_decode(case, partition_size=512)
    b = gpu_decode(case, partition_size=16384)
    assert np.abs(a - b).max() <= 1.6e-2  # at most a couple of bf16 ulps apart


def test_block_relabelling_invariance():
    case = W.make_decode([700, 33, 2000], 32, 8, 128, 16, torch.bfloat16, seed=10)
    a = gpu_decode(case)
    perm = torch.randperm(case.k_cache.shape[0], generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    case.k_cache = case.k_cache[perm].contiguous()
    case.v_cache = case.v_cache[perm].contiguous()
    bt = case.block_table.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    case.block_table = bt
    b = gpu_decode(case)
    assert np.array_equal(a, b)  # same arithmetic in the same order


def test_zero_length_sequences():
    case = W.make_decode([0, 10, 0], 8, 2, 64, 16, torch.bfloat16, seed=11, sink="randn")
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    np.testing.assert_allclose(glse[0], case.sink.numpy(), rtol=0, atol=1e-6)


def test_bad_block_id_is_flagged_not_read():
    case = W.make_decode([64, 64], 8, 2, 64, 16, torch.bfloat16, seed=12)
    case.block_table[1, 2] = case.k_cache.shape[0] + 5  # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    got = gpu_decode(case, err=err)
    assert int(err.item()) & pkv.DEVERR_BLOCK_ID
    assert np.isfinite(got).all()
    ref = oracle_decode(case, rows=[0])
    assert max_abs(got[:1], ref) <= TOL[torch.bfloat16]


def test_device_error_status_through_the_abi():
    """pkv_get_device_error turns the word the kernels OR their checks into
    into a status: an out-of-pool block id gives PKV_ERR_OUT_OF_RANGE with
    the block-id bit, and the clear flag resets the word."""
    case = W.make_decode([64, 64], 8, 2, 64, 16, torch.bfloat16, seed=12)
    case.block_table[1, 2] = case.k_cache.shape[0] + 5  # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    gpu_decode(case, err=err)
    lib = pkv.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    bits = ctypes.c_int32(0)
    st = lib.pkv_get_device_error(err.data_ptr(), ctypes.addressof(bits), 1, stream)
    assert lib.pkv_status_string(st) == b"PKV_ERR_OUT_OF_RANGE"
    assert bits.value & pkv.DEVERR_BLOCK_ID and not bits.value & pkv.DEVERR_TIMEOUT
    torch.cuda.synchronize()
    assert int(err.item()) == 0  # cleared on the stream
    assert lib.pkv_get_device_error(err.data_ptr(), None, 0, stream) == 0
    # the binding: bits back, or an exception on request
    gpu_decode(case, err=err)
    assert pkv.get_device_error(err) & pkv.DEVERR_BLOCK_ID
    with pytest.raises(pkv.PkvError) as e:
        pkv.get_device_error(err, raise_on_error=True)
    assert e.value.status_name == "PKV_ERR_OUT_OF_RANGE"


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """A pipeline wait that nothing completes gives up by itself (no trap, no
    hang): the library's self-test runs one on a barrier nothing arrives on,
    the timeout bit lands in the error word, pkv_get_device_error reports
    PKV_ERR_TIMEOUT, and the next calls on the same context still compute
    the attention."""
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    pkv.selftest_bounded_wait(err)
    lib = pkv.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    bits = ctypes.c_int32(0)
    st = lib.pkv_get_device_error(err.data_ptr(), ctypes.addressof(bits), 1, stream)
    assert lib.pkv_status_string(st) == b"PKV_ERR_TIMEOUT"
    assert bits.value == pkv.DEVERR_TIMEOUT
    with pytest.raises(pkv.PkvError) as e:
        pkv.selftest_bounded_wait(err)
        pkv.get_device_error(err, clear=True, raise_on_error=True)
    assert e.value.status_name == "PKV_ERR_TIMEOUT"
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    case = W.make_decode([37, 300], 8, 2, 64, 16, torch.bfloat16, seed=14)
    got = gpu_decode(case, err=err)
    assert max_abs(got, oracle_decode(case)) <= TOL[torch.bfloat16]
    assert int(err.item()) == 0


def test_seqlen_above_declared_max_is_flagged():
    case = W.make_decode([100, 40], 8, 2, 64, 16, torch.bfloat16, seed=13)
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    gpu_decode(case, err=err, max_seqlen=64)
    assert int(err.item()) & pkv.DEVERR_SEQLEN


# ---------------------------------------------------------------------------
# the serving configurations at full size
# ---------------------------------------------------------------------------

def test_config2_decode_full():
    case = W.config2_decode()
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.bfloat16]


@pytest.mark.parametrize("layer", [0, 1])
def test_config3_long_context(layer):
    """Long-context split-KV decode, every sequence of both layers against the
    oracle: layer 0 (window 127) and layer 1 (full 32K-128K context, up to
    256 partitions merged per head), outputs and lse."""
    case = W.config3_long(layer)
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.bfloat16]


def test_config5_decode_half_after_cache_write():
    """The decode half of the mixed step: write the new tokens, then attend
    over cache length + 1; all 256 sequences against the oracle."""
    case = W.config5_mixed()
    d = dev()
    kc, vc = case.k_cache.to(d), case.v_cache.to(d)
    pkv.reshape_and_cache(case.key.to(d), case.value.to(d), kc, vc, case.slot_mapping.to(d))
    torch.cuda.synchronize()
    dec = case.decode
    dec.k_cache, dec.v_cache = kc.cpu(), vc.cpu()
    got, glse = gpu_decode(dec, with_lse=True)
    ref, rlse = oracle_decode(dec, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.bfloat16]


# ---------------------------------------------------------------------------
# ALiBi
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Hq,Hkv,D,bs", [(32, 8, 128, 16), (16, 16, 64, 32), (32, 2, 128, 16),
                                         (6, 2, 64, 16)])
@pytest.mark.parametrize("alibi", ["geometric", "uniform"])
def test_alibi_bf16(Hq, Hkv, D, bs, alibi):
    lens = [1, 17, 511, 513, 1500, 4096]
    case = W.make_decode(lens, Hq, Hkv, D, bs, torch.bfloat16, seed=Hq + D + bs + 5,
                         sink="randn", alibi=alibi)
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.bfloat16]


@pytest.mark.parametrize("window,part", [(-1, 64), (100, 512), (1000, 16384)])
def test_alibi_windows_and_partitions(window, part):
    case = W.make_decode([3, 700, 2049, 5000], 32, 8, 128, 16, torch.bfloat16, seed=window + 41,
                         sink="randn", window_left=window, alibi="uniform")
    got = gpu_decode(case, partition_size=part)
    assert max_abs(got, oracle_decode(case)) <= TOL[torch.bfloat16]


def test_alibi_fp32_path():
    case = W.make_decode([1, 31, 70, 300], 4, 2, 64, 32, torch.float32, seed=42, sink="randn",
                         alibi="uniform")
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.float32]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.float32]


def test_alibi_long_context_sampled():
    """Slopes as shallow as 2^-8 over 32K-128K keys: the bias spans hundreds of
    log2 units and the fp32 distance arithmetic must stay exact enough."""
    gen = torch.Generator().manual_seed(43)
    lens = torch.randint(32768, 131072, (4,), generator=gen).tolist()
    case = W.make_decode(lens, 64, 8, 64, 16, torch.bfloat16, seed=43, sink="randn",
                         alibi="geometric")
    got = gpu_decode(case)
    ref = oracle_decode(case, rows=[0, 3])
    assert max_abs(got[[0, 3]], ref) <= TOL[torch.bfloat16]


# ---------------------------------------------------------------------------
# head sizes 80 / 96 / 112 / 256
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D", [80, 96, 112, 256])
@pytest.mark.parametrize("Hq,Hkv,bs", [(32, 8, 16), (16, 1, 32), (8, 8, 16)])
def test_head_sizes_bf16(D, Hq, Hkv, bs):
    lens = [1, 17, 511, 513, 2000]
    case = W.make_decode(lens, Hq, Hkv, D, bs, torch.bfloat16, seed=D + Hq + bs, sink="randn",
                         window_left=700 if bs == 32 else -1)
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.bfloat16]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.bfloat16]


@pytest.mark.parametrize("D", [80, 112])
def test_head_sizes_fp32(D):
    case = W.make_decode([1, 31, 70, 300], 4, 2, D, 32, torch.float32, seed=D, sink="randn")
    got, glse = gpu_decode(case, with_lse=True)
    ref, rlse = oracle_decode(case, with_lse=True)
    assert max_abs(got, ref) <= TOL[torch.float32]
    assert lse_err(glse, rlse) <= LSE_TOL[torch.float32]


@pytest.mark.parametrize("D", [96, 256])
def test_head_sizes_many_heads_warp_merge(D):
    """Many (sequence, head) pairs with few partitions: the warp-per-head
    merge for 256, the CTA merge for 96."""
    gen = torch.Generator().manual_seed(D)
    lens = torch.randint(1, 1500, (64,), generator=gen).tolist()
    case = W.make_decode(lens, 32, 8, D, 16, torch.bfloat16, seed=D + 1, sink="randn",
                         alibi="geometric")
    got = gpu_decode(case)
    rows = list(range(0, 64, 5))
    assert max_abs(got[rows], oracle_decode(case, rows=rows)) <= TOL[torch.bfloat16]
