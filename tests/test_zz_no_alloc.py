"""The no-allocation decode entry point (GPU).

pkv_paged_decode_noalloc serves callers that cannot allocate device memory at
the call site (a plug-in whose host framework owns all device memory, a
serving loop that must not allocate once running): its split-KV scratch is a
fixed 32 MiB device array inside the library instead of a caller workspace.
This file is collected last, so a run that stops at its first failure has
already run every other test.  It checks, through the C ABI, that two calls
in a row (the second one reusing the array the first one left behind) match
the workspace entry point (the same kernels with the same arithmetic, so the
outputs must be bit-identical), and that a problem needing more scratch than
the array holds is rejected before any launch.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import TOL, dev, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20  # PKV_NOALLOC_DECODE_SCRATCH_BYTES in include/pkv.h
PKV_ERR_WORKSPACE = 3


def _abi():
    lib = pkv.load_library()
    fn = lib.pkv_paged_decode_noalloc
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, pkv.CacheDesc, P, i32, P, i32, P, i32, i32, i32, f32, i32, P, P, P]
    fn.restype = i32
    return fn


def _tensors(case):
    return dict(q=to_dev(case.q), kc=to_dev(case.k_cache), vc=to_dev(case.v_cache),
                bt=to_dev(case.block_table), sl=to_dev(case.cache_seqlens),
                sink=to_dev(case.sink))


def _call_noalloc(fn, case, t, out, lse, err):
    desc = pkv.CacheDesc(*t["kc"].shape[:4], 0 if t["kc"].dtype == torch.float32 else 1)
    return fn(out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(), desc,
              t["bt"].data_ptr(), t["bt"].shape[1], t["sl"].data_ptr(), case.max_seqlen,
              None if t["sink"] is None else t["sink"].data_ptr(), case.batch,
              case.num_qo_heads, case.window_left, case.sm_scale, case.partition_size,
              lse.data_ptr(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_decode_matches_workspace_decode_on_two_calls_in_a_row():
    fn = _abi()
    cases = [
        W.make_decode([700, 1, 2500, 512, 4097], 32, 8, 128, 16, torch.bfloat16, seed=41,
                      sink="randn", window_left=1500),
        W.config1_tiny(),
    ]
    for case in cases:
        need = pkv.paged_decode_workspace_size(case.batch, case.num_qo_heads, case.q.shape[2],
                                               case.max_seqlen, case.partition_size,
                                               case.window_left)
        assert need <= SCRATCH_BYTES
    for case in cases:  # call 2 reuses the array call 1 left behind
        t = _tensors(case)
        ref_lse = torch.empty(case.batch, case.num_qo_heads, dtype=torch.float32, device=dev())
        ref = pkv.paged_decode(t["q"], t["kc"], t["vc"], t["bt"], t["sl"], case.max_seqlen,
                               sink=t["sink"], window_left=case.window_left,
                               sm_scale=case.sm_scale, partition_size=case.partition_size,
                               lse=ref_lse)
        out = torch.full_like(t["q"], float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=dev())
        st = _call_noalloc(fn, case, t, out, lse, err)
        torch.cuda.synchronize()
        assert st == 0, pkv.load_library().pkv_status_string(st)
        assert int(err.item()) == 0
        o, r = out.float().cpu().numpy(), ref.float().cpu().numpy()
        assert np.isfinite(o).all()
        assert np.abs(o - r).max() <= TOL[case.q.dtype]  # the suite's bar ...
        assert torch.equal(out, ref)                      # ... and in fact bit-identical
        assert torch.equal(lse, ref_lse)


def test_noalloc_rejects_problems_beyond_the_scratch():
    fn = _abi()
    case = W.make_decode([64, 64, 64, 64], 32, 8, 128, 16, torch.bfloat16, seed=42)
    t = _tensors(case)
    huge = 1 << 20  # declared max length: 2048 partitions of 512 -> ~135 MB of partials
    need = pkv.paged_decode_workspace_size(case.batch, case.num_qo_heads, 128, huge, 512, -1)
    assert need > SCRATCH_BYTES
    out = torch.zeros_like(t["q"])
    lse = torch.zeros(case.batch, case.num_qo_heads, dtype=torch.float32, device=dev())
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    desc = pkv.CacheDesc(*t["kc"].shape[:4], 1)
    st = fn(out.data_ptr(), t["q"].data_ptr(), t["kc"].data_ptr(), t["vc"].data_ptr(), desc,
            t["bt"].data_ptr(), t["bt"].shape[1], t["sl"].data_ptr(), huge, None, case.batch,
            case.num_qo_heads, -1, case.sm_scale, 512, lse.data_ptr(), err.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == PKV_ERR_WORKSPACE
    assert int(out.abs().sum()) == 0  # nothing ran


def test_binding_noalloc_matches_paged_decode():
    """The Python binding of the entry point (argument marshalling only) gives
    what the workspace entry point gives on the same inputs."""
    case = W.make_decode([300, 17, 1024, 4096], 32, 8, 128, 16, torch.bfloat16, seed=43,
                         sink="randn")
    t = _tensors(case)
    ref_lse = torch.empty(case.batch, case.num_qo_heads, dtype=torch.float32, device=dev())
    ref = pkv.paged_decode(t["q"], t["kc"], t["vc"], t["bt"], t["sl"], case.max_seqlen,
                           sink=t["sink"], sm_scale=case.sm_scale,
                           partition_size=case.partition_size, lse=ref_lse)
    lse = torch.full_like(ref_lse, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=dev())
    out = pkv.paged_decode_noalloc(t["q"], t["kc"], t["vc"], t["bt"], t["sl"], case.max_seqlen,
                                   sink=t["sink"], sm_scale=case.sm_scale,
                                   partition_size=case.partition_size, lse=lse, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o, r = out.float().cpu().numpy(), ref.float().cpu().numpy()
    assert np.isfinite(o).all()
    assert np.abs(o - r).max() <= TOL[case.q.dtype]
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
