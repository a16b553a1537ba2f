#!/usr/bin/env python3
"""Throughput benchmark of the paged KV-cache attention hot path on GB300.

One step = one continuous-batching step of the mixed serving workload, which
exercises every operation of the hot path in the order vLLM's
PagedAttention.forward runs them: reshape_and_cache writes the K/V of all
8448 new tokens into the page pool, then paged_decode attends 256 decode
sequences over their cache (+ the new token), then varlen_prefill attends 4
prefill chunks of 2048 tokens over 4096 cached tokens each.  32 query / 8 kv
heads, head_dim 128, block_size 16, bf16, synthetic seeded inputs.

The decode and prefill calls of a step both follow the cache write and are
independent of each other, so the step runs the prefill on a high-priority
stream beside the decode, with the prefill's persistent CTAs capped at 104 of
the 152 SMs (varlen_prefill's max_ctas) and the HBM-bound decode on the rest;
every call is a plain C-ABI call on a caller stream.

Printed: ONE JSON line (rank 0).  value = query tokens per second of the whole
job; `e2e` repeats the measurement through host (pinned) buffers with the
per-step inputs copied in and the outputs copied out inside the timed region;
`roofline` rates the dominant call against the measured HBM / bf16 peak, each
call timed alone in a second pass of the same steps run one call after the
other (`serial_ms_per_step`); `step_roofline` rates the whole step against
max(HBM bytes / HBM peak, flops / bf16 peak); `cpu_baseline` times the fp64
oracle on a bounded sample of the same step.

--impl reference runs the reference arm: the fp64 CPU oracle, on a bounded
sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s (% HBM peak); varlen prefill TFLOP/s; tokens/s"
WORKLOAD = ("mixed continuous batch bf16: 256 decode sequences (cache lengths log-uniform in "
            "[128,16384]) + 4 prefill chunks of 2048 tokens over prefixes of 4096, 32 qo / 8 kv "
            "heads, head_dim 128, block_size 16; reshape_and_cache of all 8448 new tokens, then "
            "paged_decode, then varlen_prefill")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of the same launch as the bench step's call, valid
# only while the kernel's code is unchanged (sha256 prefix of the files it is
# compiled from, comments and layout aside).
NCU_TRAFFIC = {
    # decode call of the mixed step (split-KV kernel + merge): 3157.8 MB read
    # and 7.6 MB of partials written by the partition kernel, 27.8 MB of
    # partials read back by the merge (cold caches under ncu; live they are
    # L2 hits); mean of three calls
    "decode": {"bytes": 3193203285, "sha": "f65c0ecb16b8e406"},
    # prefill launch of the mixed step: 172.3 MB read + 48.4 MB written
    # (mean of three launches)
    "prefill": {"bytes": 220608427, "sha": "3b1493568a2ab8b6"},
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-configuration decode / prefill lines")
    ap.add_argument("--profile", choices=["decode", "decode_long", "decode_mixed", "prefill",
                                          "prefill_d256", "prefill_mixed", "write", "rope"],
                    default=None,
                    help="run a few launches of one call on a mid-size case (for ncu)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; the step shards by request)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        import torch
        import torch.distributed as td
        self.td = td
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.on = self.world > 1
        if self.on:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            td.init_process_group(backend=backend)
        if torch.cuda.is_available():
            torch.cuda.set_device(self.local_rank)

    def barrier(self):
        if self.on:
            self.td.barrier()

    def max(self, x: float) -> float:
        if not self.on:
            return x
        import torch
        dev = torch.device("cuda", self.local_rank) if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.td.all_reduce(t, op=self.td.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.on:
            self.td.destroy_process_group()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        # median over samples taken while the SMs were clocked up (under load)
        hi = sorted(sm)
        under = hi[len(hi) // 2:] if hi else []
        return {"sm_mhz": statistics.median(under) if under else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# workload accounting
# ---------------------------------------------------------------------------

def kv_bytes_decode(case):
    L = case.cache_seqlens.long()
    if case.window_left >= 0:
        L = L.clamp(max=case.window_left + 1)
    Hkv, D = case.k_cache.shape[2], case.k_cache.shape[3]
    return int(L.sum()) * Hkv * D * case.k_cache.element_size() * 2


def attended_pairs(q_len, kv_len, window_left=-1):
    """Number of (query, key) pairs the causal (+window) mask keeps."""
    tot = 0
    for i in range(q_len):
        qpos = kv_len - q_len + i
        if qpos < 0:
            continue
        lo = 0 if window_left < 0 else max(0, qpos - window_left)
        tot += min(qpos, kv_len - 1) - lo + 1
    return tot


def prefill_flops(case):
    Hq, D = case.q.shape[1], case.q.shape[2]
    pairs = sum(attended_pairs(int(q), int(k), case.window_left)
                for q, k in zip(case.q_lens.tolist(), case.kv_lens.tolist()))
    return 4 * Hq * D * pairs


def rope_bytes(num_tokens, Hq, Hkv, D, rotary_dim, elem_bytes):
    """Algorithmic HBM bytes of rope_reshape_and_cache: per token the rotated
    part of every q head is read and written back; every k head is read,
    its rotated part written back and the whole row written to the cache;
    every v head is read and written to the cache; plus the int64 position
    and slot.  The cos/sin table (L2 resident, shared by tokens at one
    position) is not counted."""
    per_token = elem_bytes * (2 * Hq * rotary_dim + Hkv * (2 * D + rotary_dim) + 2 * Hkv * D)
    return num_tokens * (per_token + 16)


def sparse_kept_pairs(seq_len, vertical, slash):
    """Causal (query, key) pairs the vertical + slash pattern keeps, summed
    over heads: per row i, |V <= i| + |S <= i| - |{j in V: i - j in S}|, the
    last term a convolution of the two indicator vectors (FFT, rounded)."""
    S = int(seq_len)
    total = 0
    n = 1 << (2 * S - 1).bit_length()
    for vh, sh in zip(vertical, slash):
        v = np.zeros(S)
        v[np.asarray(vh)] = 1.0
        d = np.zeros(S)
        d[np.asarray(sh)] = 1.0
        both = np.rint(np.fft.irfft(np.fft.rfft(v, n) * np.fft.rfft(d, n), n)[:S])
        total += int(np.cumsum(v).sum() + np.cumsum(d).sum() - both.sum())
    return total


def sparse_tile_fraction(seq_len, vertical, slash, num_kv_heads, rows=128, keys=128,
                         tiles_per_item=2):
    """(key tiles the sparse prefill must process, key tiles of dense causal
    attention) at the kernel's granularity: one work item takes
    tiles_per_item * rows / G query tokens of the G query heads of a kv head,
    and a 128-key tile is needed iff it holds a kept (query, key) pair for
    one of them: a kept column in the tile, or a kept diagonal between the
    item's and the tile's positions."""
    S = int(seq_len)
    Hq = vertical.shape[0]
    G = Hq // num_kv_heads
    tok = tiles_per_item * rows // G
    nkt = (S + keys - 1) // keys
    need = dense = 0
    for g in range(num_kv_heads):
        vb = np.zeros(nkt * keys, bool)
        sb = np.zeros(S, bool)
        for h in range(g * G, (g + 1) * G):
            vb[np.asarray(vertical[h])] = True
            sb[np.asarray(slash[h])] = True
        vcol = vb.reshape(nkt, keys).any(axis=1)
        scum = np.concatenate([[0], np.cumsum(sb)])
        for p0 in range(0, S, tok):
            p1 = min(p0 + tok, S) - 1
            nk = p1 // keys + 1
            k0 = np.arange(nk) * keys
            k1 = np.minimum(k0 + keys - 1, p1)
            anys = (scum[p1 - k0 + 1] - scum[np.maximum(p0 - k1, 0)]) > 0
            need += int((vcol[:nk] | anys).sum())
            dense += nk
    return need, dense


def time_flushed(fn, K, flush):
    """Mean device time of fn over K launches, each timed alone with CUDA
    events after a write of a buffer larger than L2 (so no launch reads what
    the previous one left in L2)."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(K):
        flush.add_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


# the files the dense prefill and the bf16 decode kernels are compiled from
PREFILL_SOURCES = ("prefill.cu", "prefill_common.cuh", "pkv_tcgen05.cuh", "pkv_device.cuh",
                   "pkv_internal.h")
DECODE_SOURCES = ("decode.cu", "pkv_device.cuh", "pkv_internal.h")


def strip_c_comments(text: str) -> str:
    """C/C++ source with its comments removed and each line's whitespace
    collapsed, string and character literals kept: what the compiler sees."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (" ".join(line.split()) for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def source_sha(*names):
    """sha256 prefix of the code (comments and layout aside) of csrc files."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_attention_gb300", "csrc", n)) as f:
            h.update(strip_c_comments(f.read()).encode())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class MixedStep:
    """Device-resident inputs and the three C-ABI calls of one step."""

    # the high-priority stream the prefill of an overlapped step runs on
    _side = None
    # In an overlapped step the prefill's persistent attention CTAs are capped
    # at this fraction of the SMs, leaving the rest to the decode beside it:
    # measured on GB300 over caps of 88-136 of 152 SMs, 104 gave the shortest
    # step (1.039 ms against 1.086 ms uncapped and 1.118 ms serial).
    PREFILL_SM_FRACTION = 104 / 152

    def __init__(self, case, dev, pool=None):
        import torch
        import paged_kv_cache_attention_gb300 as pkv
        self.pkv = pkv
        self.case = case
        self.dev = dev
        d, p = case.decode, case.prefill
        # the KV pool is the serving state: a second stepper may share it
        self.kc, self.vc = pool if pool is not None else (case.k_cache.to(dev),
                                                          case.v_cache.to(dev))
        self.key = case.key.to(dev)
        self.value = case.value.to(dev)
        self.slots = case.slot_mapping.to(dev)
        self.q_dec = d.q.to(dev)
        self.bt_dec = d.block_table.to(dev)
        self.sl_dec = d.cache_seqlens.to(dev)
        self.q_pre = p.q.to(dev)
        self.bt_pre = p.block_table.to(dev)
        self.cuq = p.cu_seq_lens_q.to(dev)
        self.cuk = p.cu_seq_lens_k.to(dev)
        self.out_dec = torch.empty_like(self.q_dec)
        self.out_pre = torch.empty_like(self.q_pre)
        self.ws_dec = torch.empty(pkv.paged_decode_workspace_size(
            d.batch, d.num_qo_heads, d.q.shape[2], d.max_seqlen, 512, -1), dtype=torch.uint8,
            device=dev)
        self.ws_pre = torch.empty(pkv.varlen_prefill_workspace_size(
            p.batch, p.q.shape[1], p.k_cache.shape[2], p.total_q, p.max_seqlen_q),
            dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_dec = d.max_seqlen
        self.tokens = case.num_new_tokens

    def write(self):
        self.pkv.reshape_and_cache(self.key, self.value, self.kc, self.vc, self.slots,
                                   dev_error=self.err)

    def decode(self):
        d = self.case.decode
        self.pkv.paged_decode(self.q_dec, self.kc, self.vc, self.bt_dec, self.sl_dec,
                              self.max_dec, sink=None, window_left=-1, sm_scale=d.sm_scale,
                              out=self.out_dec, workspace=self.ws_dec, dev_error=self.err)

    def prefill(self, max_ctas=0):
        p = self.case.prefill
        self.pkv.varlen_prefill(self.q_pre, self.kc, self.vc, self.bt_pre, self.cuq, self.cuk,
                                p.max_seqlen_q, p.max_seqlen_k, sink=None, window_left=-1,
                                sm_scale=p.sm_scale, out=self.out_pre, workspace=self.ws_pre,
                                dev_error=self.err, max_ctas=max_ctas)

    def step(self):
        self.write()
        self.decode()
        self.prefill()

    def prefill_ctas(self):
        import torch
        sms = torch.cuda.get_device_properties(self.dev).multi_processor_count
        return max(1, round(self.PREFILL_SM_FRACTION * sms))

    def side_stream(self):
        import torch
        if MixedStep._side is None:
            lo, hi = torch.cuda.Stream.priority_range()
            MixedStep._side = torch.cuda.Stream(device=self.dev, priority=min(lo, hi))
        return MixedStep._side

    def step_overlapped(self, events=None):
        """The same three calls: the cache write, then the prefill on the
        high-priority side stream and the decode on the caller's stream, both
        after the write; the caller's stream then waits for the prefill.
        events: optional [write end, decode end, prefill start, prefill end]
        CUDA events to record."""
        import torch
        main = torch.cuda.current_stream()
        side = self.side_stream()
        self.write()
        written = events[0] if events else torch.cuda.Event()
        written.record(main)
        side.wait_event(written)
        with torch.cuda.stream(side):
            if events:
                events[2].record(side)
            self.prefill(max_ctas=self.prefill_ctas())
            if events:
                events[3].record(side)
        self.decode()
        if events:
            events[1].record(main)
        done = torch.cuda.Event()
        done.record(side)
        main.wait_event(done)


def time_overlapped(stepper, K, W, dist):
    """K timed overlapped steps bracketed by barrier + synchronize.  Returns
    the total time and how long the decode (caller's stream) and the prefill
    (side stream) took inside them, each from the end of the write."""
    import torch
    for _ in range(W):
        stepper.step_overlapped()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    start.record()
    for k in range(K):
        stepper.step_overlapped(events=ev[k])
    end.record()
    torch.cuda.synchronize()
    dist.barrier()
    total_ms = start.elapsed_time(end)
    inside = {"paged_decode": statistics.mean(ev[k][0].elapsed_time(ev[k][1]) for k in range(K)),
              "varlen_prefill": statistics.mean(ev[k][0].elapsed_time(ev[k][3])
                                                for k in range(K))}
    return total_ms, inside


def time_device(stepper, K, W, dist):
    """K timed steps run one call after the other, bracketed by barrier +
    synchronize, with per-call events (each call's own duration)."""
    import torch
    for _ in range(W):
        stepper.step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    start.record()
    for k in range(K):
        ev[k][0].record()
        stepper.write()
        ev[k][1].record()
        stepper.decode()
        ev[k][2].record()
        stepper.prefill()
        ev[k][3].record()
    end.record()
    torch.cuda.synchronize()
    dist.barrier()
    total_ms = start.elapsed_time(end)
    calls = {name: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K))
             for i, name in enumerate(["reshape_and_cache", "paged_decode", "varlen_prefill"])}
    return total_ms, calls


def time_e2e(stepper, K, W, dist, overlapped=True):
    """The same step through pinned host buffers: every step's inputs (queries,
    new K/V, slot mapping, block tables, lengths) are copied in from pinned
    host memory and its outputs copied out, all inside the timed region; the
    page pool stays resident (it is the cache).  The copies are pipelined the
    way a serving loop would run them: two device buffer sets, an upload
    stream bringing in step k+1's inputs and a download stream taking out step
    k-1's outputs while the compute stream runs step k (the steps themselves
    stay in order on the compute stream, so every step sees the cache writes
    of the ones before); uploads and downloads use separate streams so that
    neither queues behind the other."""
    import torch
    dev = stepper.dev
    other = MixedStep(stepper.case, dev, pool=(stepper.kc, stepper.vc))
    sets = [stepper, other]

    def ins(st):
        return [st.q_dec, st.q_pre, st.key, st.value, st.slots, st.bt_dec, st.sl_dec,
                st.bt_pre, st.cuq, st.cuk]

    def outs(st):
        return [st.out_dec, st.out_pre]

    host_in = [t.cpu().pin_memory() for t in ins(stepper)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs(stepper)]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])

    def step(st):
        if overlapped:
            st.step_overlapped()
        else:
            st.step()
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def run(n):
        h2d_start = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        h2d_done = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        done = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        d2h_done = [torch.cuda.Event(enable_timing=True) for _ in range(n)]

        def upload(k):
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(done[k - 2])  # step k-2 no longer reads set k % 2
                h2d_start[k].record(up)
                for h, d in zip(host_in, ins(sets[k % 2])):
                    d.copy_(h, non_blocking=True)
                h2d_done[k].record(up)

        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            compute.wait_event(h2d_done[k])
            if k >= 2:
                compute.wait_event(d2h_done[k - 2])  # set k % 2's outputs are out
            step(sets[k % 2])
            done[k].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(done[k])
                for h, d in zip(host_out[k % 2], outs(sets[k % 2])):
                    h.copy_(d, non_blocking=True)
                d2h_done[k].record(down)
        torch.cuda.synchronize()
        # per-step copy durations on their streams (diagnostics)
        return (statistics.mean(h2d_start[k].elapsed_time(h2d_done[k]) for k in range(n)),
                statistics.mean(done[k].elapsed_time(d2h_done[k]) for k in range(n)))

    run(W)
    dist.barrier()
    t0 = time.perf_counter()
    up_ms, down_ms = run(K)
    dist.barrier()
    ms = (time.perf_counter() - t0) * 1e3
    del other
    return ms, h2d, d2h, up_ms, down_ms


def time_back_to_back(fn, n, reps=3):
    """Median over reps of the mean device time of n back-to-back launches of
    fn (CUDA events on the current stream, after 3 warm-up launches)."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    means = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        means.append(a.elapsed_time(b) / n)
    return statistics.median(means)


def extra_configs(dev, K, peaks):
    """Per-configuration lines for the other serving shapes (decode GB/s and
    prefill TFLOP/s), each input set larger than L2: the median of three
    means of back-to-back launches (50 for decode, 20 for prefill)."""
    import torch
    import paged_kv_cache_attention_gb300 as pkv
    from paged_kv_cache_attention_gb300 import workloads as W
    out = {}

    def run_decode(name, cases):
        tens = []
        byts = 0
        for c in cases:
            tens.append(dict(q=c.q.to(dev), kc=c.k_cache.to(dev), vc=c.v_cache.to(dev),
                             bt=c.block_table.to(dev), sl=c.cache_seqlens.to(dev),
                             sink=None if c.sink is None else c.sink.to(dev), c=c,
                             alibi=None if c.alibi is None else c.alibi.to(dev),
                             ws=torch.empty(pkv.paged_decode_workspace_size(
                                 c.batch, c.num_qo_heads, c.q.shape[2], c.max_seqlen,
                                 c.partition_size, c.window_left), dtype=torch.uint8,
                                 device=dev)))
            byts += kv_bytes_decode(c)

        def go():
            for t in tens:
                c = t["c"]
                pkv.paged_decode(t["q"], t["kc"], t["vc"], t["bt"], t["sl"], c.max_seqlen,
                                 sink=t["sink"], window_left=c.window_left,
                                 sm_scale=c.sm_scale, partition_size=c.partition_size,
                                 workspace=t["ws"], alibi_slopes=t["alibi"])
        ms = time_back_to_back(go, max(K, 50))
        gbs = byts / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 4), "kv_bytes": byts, "GB/s": round(gbs, 1),
                     "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 3),
                     "frac_hbm_8TBs": round(gbs / 8000.0, 3)}
        del tens
        torch.cuda.empty_cache()

    run_decode("config2_decode_B64_L512-4096", [W.config2_decode()])
    c2a = W.config2_decode()
    c2a.alibi = W.alibi_slopes("geometric", c2a.num_qo_heads, None)
    run_decode("config2_decode_B64_alibi", [c2a])
    del c2a
    run_decode("config3_decode_B8_L32K-128K_2layers", [W.config3_long(0), W.config3_long(1)])
    c4 = W.config4_prefill()
    q, kc, vc = c4.q.to(dev), c4.k_cache.to(dev), c4.v_cache.to(dev)
    bt, cq, ck, sink = (c4.block_table.to(dev), c4.cu_seq_lens_q.to(dev),
                        c4.cu_seq_lens_k.to(dev), c4.sink.to(dev))
    ws = torch.empty(pkv.varlen_prefill_workspace_size(c4.batch, q.shape[1], kc.shape[2],
                                                       c4.total_q, c4.max_seqlen_q),
                     dtype=torch.uint8, device=dev)
    outp = torch.empty_like(q)

    fl = prefill_flops(c4)
    geo = W.alibi_slopes("geometric", q.shape[1], None).to(dev)
    for name, al in (("config4_prefill_B16", None), ("config4_prefill_B16_alibi", geo)):
        def go4():
            pkv.varlen_prefill(q, kc, vc, bt, cq, ck, c4.max_seqlen_q, c4.max_seqlen_k,
                               sink=sink, sm_scale=c4.sm_scale, out=outp, workspace=ws,
                               alibi_slopes=al)
        ms = time_back_to_back(go4, max(K, 20))
        tf = fl / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "flops": fl, "TFLOP/s": round(tf, 1),
                     "frac_bf16_measured_burst": round(tf / peaks["bf16_tflops"], 3)}
    del q, kc, vc, outp, ws
    torch.cuda.empty_cache()

    # the same lengths with head_dim 256 (16 query / 8 kv heads: the same
    # flops), on the head_dim-256 prefill kernel
    c4w = W.config4_prefill(16, 8, 256)
    qw, kcw, vcw = c4w.q.to(dev), c4w.k_cache.to(dev), c4w.v_cache.to(dev)
    btw, cqw, ckw, sinkw = (c4w.block_table.to(dev), c4w.cu_seq_lens_q.to(dev),
                            c4w.cu_seq_lens_k.to(dev), c4w.sink.to(dev))
    wsw = torch.empty(pkv.varlen_prefill_workspace_size(c4w.batch, 16, 8, c4w.total_q,
                                                        c4w.max_seqlen_q),
                      dtype=torch.uint8, device=dev)
    outw = torch.empty_like(qw)

    def gow():
        pkv.varlen_prefill(qw, kcw, vcw, btw, cqw, ckw, c4w.max_seqlen_q, c4w.max_seqlen_k,
                           sink=sinkw, sm_scale=c4w.sm_scale, out=outw, workspace=wsw)
    ms = time_back_to_back(gow, max(K, 20))
    flw = prefill_flops(c4w)
    tf = flw / (ms * 1e-3) / 1e12
    out["config4_prefill_B16_D256"] = {"ms": round(ms, 4), "flops": flw, "TFLOP/s": round(tf, 1),
                                       "frac_bf16_measured_burst": round(tf / peaks["bf16_tflops"], 3)}
    del qw, kcw, vcw, outw, wsw
    torch.cuda.empty_cache()

    # MInference vertical + slash sparse prefill of one 32K-token sequence
    # whose attention has local (slash) and stripe (vertical) structure
    # (default budget 0.3), against the dense causal prefill of the same one
    S = 32768
    qm, km, vm = (t.to(dev) for t in W.make_long_sequence(S, 32, 8, 128, W.seed_for(6)))
    outm = torch.empty_like(qm)
    wsm = torch.empty(pkv.lib_minference_workspace(S, 32, 8), dtype=torch.uint8, device=dev)
    _, vim, sim = pkv.minference_prefill(qm, km, vm, out=outm, workspace=wsm,
                                         return_pattern=True)
    cum = torch.tensor([0, S], dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ms_sparse = time_flushed(lambda: pkv.minference_prefill(qm, km, vm, out=outm, workspace=wsm),
                             max(3, K // 10), flush)
    ms_dense = time_flushed(lambda: pkv.varlen_prefill_contiguous(qm, km, vm, cum, cum, S, S,
                                                                  out=outm),
                            max(3, K // 10), flush)
    kept = sparse_kept_pairs(S, vim.cpu().numpy(), sim.cpu().numpy())
    t_need, t_dense = sparse_tile_fraction(S, vim.cpu().numpy(), sim.cpu().numpy(), 8)
    fl_kept = 4 * 128 * kept  # per kept (query, key) pair of a head: QK^T and PV
    fl_dense = 4 * 128 * 32 * (S * (S + 1) // 2)
    out["minference_prefill_S32K_Hq32_D128"] = {
        "ms": round(ms_sparse, 4), "dense_ms": round(ms_dense, 4),
        "speedup_vs_dense": round(ms_dense / ms_sparse, 3),
        "kept_pair_fraction": round(kept / (32 * S * (S + 1) // 2), 4),
        "key_tiles_needed_fraction": round(t_need / t_dense, 4),
        "TFLOP/s_on_kept_pairs": round(fl_kept / (ms_sparse * 1e-3) / 1e12, 1),
        "dense_TFLOP/s": round(fl_dense / (ms_dense * 1e-3) / 1e12, 1),
        "l2": "256 MB buffer written before each timed launch"}
    del qm, km, vm, outm, wsm, flush
    torch.cuda.empty_cache()

    # rotary embedding fused with the cache write, on the mixed step's 8448 new
    # tokens (their queries are the decode and prefill queries of the step)
    c5 = W.config5_mixed()
    qr = torch.cat([c5.decode.q, c5.prefill.q]).to(dev)
    kr, vr = c5.key.to(dev), c5.value.to(dev)
    kc5, vc5 = c5.k_cache.to(dev), c5.v_cache.to(dev)
    pos, sm = c5.positions.to(dev), c5.slot_mapping.to(dev)
    tab = pkv.rope_cos_sin_table(32768, 128)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ms = time_flushed(lambda: pkv.rope_reshape_and_cache(qr, kr, vr, kc5, vc5, pos, sm, tab),
                      K, flush)
    byts = rope_bytes(c5.num_new_tokens, qr.shape[1], kr.shape[1], kr.shape[2], 128, 2)
    gbs = byts / (ms * 1e-3) / 1e9
    out["rope_reshape_and_cache_mixed_8448tok"] = {
        "ms": round(ms, 4), "bytes": byts, "GB/s": round(gbs, 1),
        "frac_hbm_measured": round(gbs / peaks["hbm_gbs"], 3),
        "l2": "256 MB buffer written before each timed launch"}
    return out


def cpu_baseline(case, n_dec_every=2, n_pre_every=2, threads=0):
    """The fp64 oracle, as it stands, on a bounded sample of the mixed step:
    the full cache write, every n-th decode sequence and every n-th prefill
    row.  Returns (tokens/s on the sample, threads, description)."""
    import numpy as np
    import oracle
    from paged_kv_cache_attention_gb300 import workloads as W
    d, p = case.decode, case.prefill
    kc = W.to_oracle(case.k_cache).copy()
    vc = W.to_oracle(case.v_cache).copy()
    dec_rows = list(range(0, d.batch, n_dec_every))
    pre_rows = list(range(0, p.total_q, n_pre_every))
    t0 = time.perf_counter()
    oracle.reshape_and_cache(W.to_oracle(case.key), W.to_oracle(case.value), kc, vc,
                             case.slot_mapping.numpy())
    oracle.paged_decode(W.to_oracle(d.q), kc, vc, d.block_table.numpy(),
                        d.cache_seqlens.numpy(), sm_scale=d.sm_scale, rows=dec_rows,
                        threads=threads)
    oracle.attention(W.to_oracle(p.q), kc, vc, p.block_table.numpy(),
                     p.cu_seq_lens_q.numpy(), p.kv_lens.numpy(), sm_scale=p.sm_scale,
                     rows=pre_rows, threads=threads)
    dt = time.perf_counter() - t0
    tokens = len(dec_rows) + len(pre_rows)
    cores = threads if threads > 0 else oracle.online_cores()

    def every(n):
        return "every" if n == 1 else f"one in {n} of the"

    desc = (f"full cache write of {case.num_new_tokens} tokens + {every(n_dec_every)} decode "
            f"sequences ({len(dec_rows)}) + {every(n_pre_every)} prefill rows ({len(pre_rows)}); "
            f"value = sampled query tokens / wall time")
    return tokens / dt, cores, desc, dt


def run_ours(args, dist):
    import torch
    import paged_kv_cache_attention_gb300 as pkv
    from paged_kv_cache_attention_gb300 import workloads as W

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", torch.cuda.current_device())
    pkv.load_library()
    peaks, peak_src = load_peaks()
    case = W.config5_mixed()
    stepper = MixedStep(case, dev)
    K, Wm = args.steps, max(args.warmup, 3)

    clocks = ClockSampler(dist.local_rank)
    clocks.start()
    total_ms, inside = time_overlapped(stepper, K, Wm, dist)
    # the same steps with the calls one after the other: each call's own time
    serial_ms, calls = time_device(stepper, K, Wm, dist)
    clk = clocks.stop()
    err = int(stepper.err.item())
    if err:
        raise RuntimeError(f"device error flags {err} during the benchmark")
    ms_step = dist.max(total_ms / K)
    ms_serial = dist.max(serial_ms / K)
    tokens = stepper.tokens * dist.world
    value = tokens / (ms_step * 1e-3)

    dec_bytes = kv_bytes_decode(case.decode)
    pre_flops = prefill_flops(case.prefill)
    write_bytes = 2 * 2 * case.num_new_tokens * case.key[0].numel() * case.key.element_size()
    dec_gbs = dec_bytes / (calls["paged_decode"] * 1e-3) / 1e9
    pre_tf = pre_flops / (calls["varlen_prefill"] * 1e-3) / 1e12
    wr_gbs = write_bytes / (calls["reshape_and_cache"] * 1e-3) / 1e9
    hbm = peaks["hbm_gbs"]
    # the burst peak for a kernel timed in a region well under a second, the
    # sustained (power-capped) one once the timed region lasts seconds
    long_region = min(total_ms, serial_ms) >= 2000.0
    bf16_key = "bf16_tflops_sustained" if long_region and "bf16_tflops_sustained" in peaks \
        else "bf16_tflops"
    bf16 = peaks[bf16_key]
    rl_dec = {"call": "paged_decode (split-KV partition kernel + merge kernel)", "bound": "hbm",
              "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s",
              "frac": round(dec_gbs / hbm, 4),
              "traffic": NCU_TRAFFIC.get("decode", {}).get("bytes")
              if NCU_TRAFFIC.get("decode", {}).get("sha") == source_sha(*DECODE_SOURCES) else None,
              "algorithmic_bytes": dec_bytes, "ms": round(calls["paged_decode"], 4),
              "peak_source": f"{peak_src} hbm_gbs"}
    rl_pre = {"call": "varlen_prefill (work-list kernel + tcgen05 attention kernel)",
              "bound": "tensor", "achieved": round(pre_tf, 1), "peak": bf16, "unit": "TFLOP/s",
              "frac": round(pre_tf / bf16, 4),
              "traffic": NCU_TRAFFIC.get("prefill", {}).get("bytes")
              if NCU_TRAFFIC.get("prefill", {}).get("sha") == source_sha(*PREFILL_SOURCES) else None,
              "algorithmic_flops": pre_flops, "ms": round(calls["varlen_prefill"], 4),
              "peak_source": f"{peak_src} {bf16_key} (timed region {serial_ms:.0f} ms)"}
    dominant = rl_dec if calls["paged_decode"] >= calls["varlen_prefill"] else rl_pre
    other = rl_pre if dominant is rl_dec else rl_dec
    # the whole step against its own roofline: the HBM time of every byte it
    # must move (decode KV, cache write) or the tensor time of its flops,
    # whichever is longer
    bound_ms = max((dec_bytes + write_bytes) / (hbm * 1e9), pre_flops / (bf16 * 1e12)) * 1e3
    step_rl = {"bound_ms": round(bound_ms, 4), "ms_per_step": round(ms_step, 4),
               "frac": round(bound_ms / ms_step, 4),
               "bound": "max(HBM bytes of decode KV + cache write / hbm peak, "
                        "prefill flops / bf16 peak)",
               "serial_sum_bound_ms": round((dec_bytes + write_bytes) / (hbm * 1e9) * 1e3
                                            + pre_flops / (bf16 * 1e12) * 1e3, 4)}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world,
        "steps": K, "warmup": Wm, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, shuffled page pool; no dataset)",
        "config": {"workload": WORKLOAD, "decode_seqs": case.decode.batch,
                   "prefill_chunks": case.prefill.batch, "new_tokens": case.num_new_tokens,
                   "l2": "inputs larger than L2: each step reads ~3.2 GB of decode KV",
                   "parallelism": f"replicas x{dist.world} (independent steps per GPU)",
                   "prefill_ctas_in_step": stepper.prefill_ctas()},
        "gpu_launches": 5 * K,
        "roofline": dominant, "roofline_other": other, "step_roofline": step_rl,
        "serial_ms_per_step": round(ms_serial, 4),
        "calls_ms": {k: round(v, 4) for k, v in calls.items()},
        "overlapped_ms_from_write": {k: round(v, 4) for k, v in inside.items()},
        "reshape_and_cache_GBs": round(wr_gbs, 1),
        "clocks": clk,
    }
    if not args.no_e2e:
        # a serving loop's steady state: a run of steps long enough that
        # filling and draining the copy pipeline (the first upload, ~0.6 ms,
        # and the last download, ~0.4 ms) is a small part of it (~2 % at 60)
        K_e2e = max(60, K)
        e2e_ms, h2d, d2h, up_ms, down_ms = time_e2e(stepper, K_e2e, 3, dist)
        e2e_step = dist.max(e2e_ms / K_e2e)
        line["e2e"] = {"value": round(tokens / (e2e_step * 1e-3), 1), "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_step, 4), "steps": K_e2e,
                       "h2d_ms_per_step": round(up_ms, 4), "d2h_ms_per_step": round(down_ms, 4),
                       "timing": "host wall clock around all steps, copies included"}
    del stepper
    torch.cuda.empty_cache()
    if not args.no_extra:
        line["configs"] = extra_configs(dev, max(5, K // 2), peaks)
    if dist.rank == 0 and not args.no_cpu_baseline:
        v, cores, desc, secs = cpu_baseline(case)
        # the same oracle on one core, on a thirty-second of that sample
        v1, _, desc1, secs1 = cpu_baseline(case, n_dec_every=64, n_pre_every=64, threads=1)
        line["cpu_baseline"] = {"value": round(v, 2), "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": desc,
                                "seconds": round(secs, 2),
                                "single_core": {"value": round(v1, 2), "unit": "tokens/s",
                                                "cores": 1, "sample": desc1,
                                                "seconds": round(secs1, 2)}}
    return line


def run_reference(args, dist):
    """Reference arm: the fp64 oracle on the host cores, a bounded sample of
    the same workload per step."""
    from paged_kv_cache_attention_gb300 import workloads as W
    import oracle
    oracle.build()
    case = W.config5_mixed()
    K, Wm = args.steps, max(args.warmup, 3)
    for _ in range(Wm):
        cpu_baseline(case, n_dec_every=64, n_pre_every=64)
    t0 = time.perf_counter()
    toks = 0
    desc = cores = None
    for _ in range(K):
        _, cores, desc, dt = cpu_baseline(case, n_dec_every=64, n_pre_every=64)
        toks += len(range(0, case.decode.batch, 64)) + len(range(0, case.prefill.total_q, 64))
    secs = time.perf_counter() - t0
    value = toks / secs
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": dist.world, "steps": K, "warmup": Wm,
        "ms_per_step": round(secs / K * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; same inputs as ours)",
        "config": {"workload": WORKLOAD, "parallelism": "host cores of rank 0"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_profile(which: str):
    """A few launches of one call on a case larger than L2 but a few GB at
    most: decode = the B64 / L512-4096 decode batch (~0.6 GB of KV),
    decode_mixed = the mixed step's decode call (256 sequences, ~3.2 GB of KV),
    prefill = the B16 varlen prefill batch (prefill_d256: with head_dim 256), write = the mixed step's cache
    write, rope = the rotary step fused with the write for 8448 tokens."""
    import torch
    import paged_kv_cache_attention_gb300 as pkv
    from paged_kv_cache_attention_gb300 import workloads as W
    dev = torch.device("cuda", torch.cuda.current_device())
    pkv.load_library()
    if which in ("decode", "decode_long", "decode_mixed"):
        c = (W.config2_decode() if which == "decode" else
             W.config3_long(1) if which == "decode_long" else W.config5_mixed().decode)
        q, kc, vc = c.q.to(dev), c.k_cache.to(dev), c.v_cache.to(dev)
        bt, sl = c.block_table.to(dev), c.cache_seqlens.to(dev)
        ws = torch.empty(pkv.paged_decode_workspace_size(c.batch, c.num_qo_heads, q.shape[2],
                                                         c.max_seqlen, c.partition_size,
                                                         c.window_left), dtype=torch.uint8,
                         device=dev)
        sink = None if c.sink is None else c.sink.to(dev)
        go = lambda: pkv.paged_decode(q, kc, vc, bt, sl, c.max_seqlen, sink=sink,
                                      window_left=c.window_left, sm_scale=c.sm_scale,
                                      partition_size=c.partition_size, workspace=ws)
    elif which in ("prefill", "prefill_d256", "prefill_mixed"):
        # prefill_mixed: the prefill launch of the mixed step (4 chunks of 2048
        # over 4096-token prefixes), on a pool holding only those pages;
        # prefill_d256: the B16 batch with head_dim 256 (16 query / 8 kv heads)
        c = (W.config4_prefill() if which == "prefill" else
             W.config4_prefill(16, 8, 256) if which == "prefill_d256" else W.make_mixed(
                 [], 2048, 4096, 4, 32, 8, 128, 16, torch.bfloat16,
                 seed=W.seed_for(5) + 100).prefill)
        q, kc, vc = c.q.to(dev), c.k_cache.to(dev), c.v_cache.to(dev)
        bt, cq, ck = c.block_table.to(dev), c.cu_seq_lens_q.to(dev), c.cu_seq_lens_k.to(dev)
        sink = None if c.sink is None else c.sink.to(dev)
        go = lambda: pkv.varlen_prefill(q, kc, vc, bt, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                        sink=sink, sm_scale=c.sm_scale)
    elif which == "rope":
        # 8448 tokens shaped like the mixed step's new tokens, on a pool just
        # large enough for them (~0.2 GB on the device in all)
        c = W.make_rope(8448, 32, 8, 128, 128, 16, torch.bfloat16, seed=W.seed_for(5) + 7,
                        max_position=32768, skip_every=0)
        qr, key, val = c.query.to(dev), c.key.to(dev), c.value.to(dev)
        kc, vc = c.k_cache.to(dev), c.v_cache.to(dev)
        pos, sm = c.positions.to(dev), c.slot_mapping.to(dev)
        tab = pkv.rope_cos_sin_table(c.max_position, 128)
        go = lambda: pkv.rope_reshape_and_cache(qr, key, val, kc, vc, pos, sm, tab)
    else:
        c = W.config5_mixed()
        kc, vc = c.k_cache.to(dev), c.v_cache.to(dev)
        key, val, sm = c.key.to(dev), c.value.to(dev), c.slot_mapping.to(dev)
        go = lambda: pkv.reshape_and_cache(key, val, kc, vc, sm)
    for _ in range(3):
        go()
    torch.cuda.synchronize()
    print(json.dumps({"profile": which, "launched": 3}), flush=True)
    return 0


def main():
    args = parse_args()
    if args.profile:
        return run_profile(args.profile)
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        line = run_reference(args, type("D", (), {"world": int(os.environ.get("WORLD_SIZE", "1"))})())
        print(json.dumps(line), flush=True)
        return 0
    dist = Dist()
    try:
        line = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
