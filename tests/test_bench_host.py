"""Host-side logic of bench.py on CPU: the work accounting, and the
max-over-ranks timing of the replica run on 2 gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from paged_kv_cache_attention_gb300 import workloads as W


def test_attended_pairs_matches_a_mask_count():
    rng = np.random.default_rng(0)
    for _ in range(50):
        q = int(rng.integers(0, 40))
        k = int(rng.integers(0, 60))
        w = int(rng.choice([-1, 0, 3, 10]))
        pos = (k - q + np.arange(q))[:, None]
        col = np.arange(k)[None, :]
        m = col <= pos
        if w >= 0:
            m &= col >= pos - w
        assert bench.attended_pairs(q, k, w) == int(m.sum())


def test_prefill_flops_of_the_mixed_step():
    case = W.make_mixed([100, 200], 64, 128, 2, 32, 8, 128, 16, torch.bfloat16, seed=1)
    # each chunk: 64 queries over 128 + 64 keys, causal at the end
    pairs = sum(128 + i + 1 for i in range(64))
    assert bench.prefill_flops(case.prefill) == 4 * 32 * 128 * 2 * pairs


def test_decode_bytes_count_window():
    case = W.make_decode([10, 1000], 8, 2, 64, 16, torch.bfloat16, seed=2, window_left=99)
    assert bench.kv_bytes_decode(case) == (10 + 100) * 2 * 64 * 2 * 2


def test_rope_bytes_by_hand():
    """2 q heads, 1 kv head, head_dim 8, rotary_dim 4, bf16: q reads and writes
    4 dims of 2 heads (32 B), k is read (16 B), its 4 rotated dims written
    back (8 B) and its row cached (16 B), v read and cached (32 B), plus 16 B
    of position and slot: 120 B a token."""
    assert bench.rope_bytes(3, 2, 1, 8, 4, 2) == 360


def test_sparse_kept_pairs_by_brute_force():
    rng = np.random.default_rng(3)
    S = 97
    vert = [np.sort(rng.choice(S, 11, replace=False)) for _ in range(3)]
    slash = [np.sort(rng.choice(S, 17, replace=False)) for _ in range(3)]
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    want = sum(int(((j <= i) & (np.isin(j, v) | np.isin(i - j, d))).sum())
               for v, d in zip(vert, slash))
    assert bench.sparse_kept_pairs(S, vert, slash) == want


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.Dist()
    try:
        assert d.on and d.world == world and d.rank == rank
        d.barrier()
        m = d.max(1.5 + rank)  # per-rank step times: the slowest one wins
        q.put((rank, m))
    finally:
        d.close()


@pytest.mark.skipif(torch.cuda.is_available(), reason="gloo replica test runs on CPU hosts")
def test_max_over_ranks_with_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 2.5, 1: 2.5}


def test_traffic_key_ignores_comments_only():
    # the stored ncu traffic stays valid across comment edits and is dropped
    # on any code change
    code = 'int a = 1;  // one\n/* block\n   comment */ const char *s = "x // kept";\n'
    assert bench.strip_c_comments(code) == 'int a = 1;\nconst char *s = "x // kept";'
    assert bench.strip_c_comments(code.replace("// one", "// uno")) == \
        bench.strip_c_comments(code)
    assert bench.strip_c_comments(code.replace("a = 1", "a = 2")) != \
        bench.strip_c_comments(code)
    assert bench.strip_c_comments("x = '\\'' ; /* c */ y") == "x = '\\'' ; y"


def test_clock_sampler_reads_the_nvidia_smi_csv(tmp_path):
    """The clocks record of the bench line from sampled nvidia-smi rows: the
    median SM clock of the loaded half of the samples, the maximum clock, and
    every throttle reason seen Active in any sample."""
    rows = ["0, 1200, 2070, 350.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1965, 2070, 990.5, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1010.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2040, 2070, 1005.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, [N/A], 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")

    class _Done:  # a sampler process that has already exited
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = bench.ClockSampler(0)
    s.proc, s.path = _Done(), str(path)
    clk = s.stop()
    assert clk["samples"] == 5
    assert clk["sm_max_mhz"] == 2070.0
    assert clk["sm_mhz"] == 2055.0  # median of the upper half (2040, 2070) of the four clocks
    assert clk["reasons"] == ["sw_power_cap"]
    assert not path.exists()

    s2 = bench.ClockSampler(0)
    s2.proc = None
    assert s2.stop()["reasons"] == ["nvidia-smi unavailable"]
