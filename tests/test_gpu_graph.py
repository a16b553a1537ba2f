"""The calls are stream-ordered kernel launches with host-side set-up only, so
a serving loop can capture a whole step in a CUDA graph and replay it: the
replayed step must give exactly the eager results."""
import pytest
import torch

import paged_kv_cache_attention_gb300 as pkv
from paged_kv_cache_attention_gb300 import workloads as W
from tests._gpu import dev

pytestmark = pytest.mark.gpu


def test_mixed_step_replays_from_a_cuda_graph():
    d = dev()
    case = W.make_mixed([300, 1000, 17, 4096, 511], 256, 512, 2, 32, 8, 128, 16,
                        torch.bfloat16, seed=77)
    dc, pc = case.decode, case.prefill
    key, value, slots = case.key.to(d), case.value.to(d), case.slot_mapping.to(d)
    q_dec, bt_dec, sl_dec = dc.q.to(d), dc.block_table.to(d), dc.cache_seqlens.to(d)
    q_pre, bt_pre = pc.q.to(d), pc.block_table.to(d)
    cuq, cuk = pc.cu_seq_lens_q.to(d), pc.cu_seq_lens_k.to(d)
    ws_dec = torch.empty(pkv.paged_decode_workspace_size(
        dc.batch, dc.num_qo_heads, 128, dc.max_seqlen), dtype=torch.uint8, device=d)
    ws_pre = torch.empty(pkv.varlen_prefill_workspace_size(
        pc.batch, 32, 8, pc.total_q, pc.max_seqlen_q), dtype=torch.uint8, device=d)

    def step(kc, vc, out_dec, out_pre):
        pkv.reshape_and_cache(key, value, kc, vc, slots)
        pkv.paged_decode(q_dec, kc, vc, bt_dec, sl_dec, dc.max_seqlen, sm_scale=dc.sm_scale,
                         out=out_dec, workspace=ws_dec)
        pkv.varlen_prefill(q_pre, kc, vc, bt_pre, cuq, cuk, pc.max_seqlen_q, pc.max_seqlen_k,
                           sm_scale=pc.sm_scale, out=out_pre, workspace=ws_pre)

    # eager
    kc_e, vc_e = case.k_cache.to(d), case.v_cache.to(d)
    dec_e, pre_e = torch.empty_like(q_dec), torch.empty_like(q_pre)
    step(kc_e, vc_e, dec_e, pre_e)
    torch.cuda.synchronize()

    # captured on a side stream, then replayed on a fresh copy of the pool
    kc_g, vc_g = case.k_cache.to(d), case.v_cache.to(d)
    dec_g, pre_g = torch.zeros_like(q_dec), torch.zeros_like(q_pre)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(kc_g, vc_g, dec_g, pre_g)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    kc_g.copy_(case.k_cache.to(d))
    vc_g.copy_(case.v_cache.to(d))
    dec_g.zero_()
    pre_g.zero_()
    with torch.cuda.graph(graph):
        step(kc_g, vc_g, dec_g, pre_g)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(dec_g, dec_e)
    assert torch.equal(pre_g, pre_e)
    # the pools hold NaN-poisoned spare pages: compare their bits
    assert torch.equal(kc_g.view(torch.int16), kc_e.view(torch.int16))
    assert torch.equal(vc_g.view(torch.int16), vc_e.view(torch.int16))
