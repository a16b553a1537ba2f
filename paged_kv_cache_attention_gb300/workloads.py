"""Seeded synthetic inputs for paged KV-cache attention.

This module only *builds inputs*: sequence lengths, a shuffled page pool, block
tables, slot mappings and random q/k/v/sink values.  It holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle may be fed from
it.  Everything is generated on the CPU with a seeded ``torch.Generator``; the
caller moves tensors to the device.

Pool layout (NHD pages): ``k_cache``/``v_cache`` are
``[num_blocks, block_size, num_kv_heads, head_dim]``.  Pages are handed out in
the order of a seeded random permutation of the pool; pages no sequence owns
are filled with NaN so that any stray read turns an output into NaN.

Workload shapes follow the serving scenarios on the source pages: the decode
worked example of the transformers docs "paged_attention" page (block size 32,
``cache_seqlens = [30, 32, 70]``, its block table), vLLM's 512-token
split-KV decode, and FlashInfer's sink-attention reference modes (incremental,
chunk and varlen prefill, GQA, sliding window, per-head sink).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

NEG_INF = float("-inf")

# The decode worked example of the transformers docs "paged_attention" page
# ("Decode path", example): three sequences, block size 32, 4 blocks per row.
EXAMPLE_CACHE_SEQLENS = [30, 32, 70]
EXAMPLE_BLOCK_TABLE = [[2, -1, -1, -1], [0, 1, -1, -1], [3, 5, 6, -1]]
EXAMPLE_BLOCK_SIZE = 32
EXAMPLE_NUM_BLOCKS = 8

CONFIG_NAMES = {
    1: "tiny paged decode fp32 (B3, seqlens [30,32,70], bs32, Hq4/Hkv2, D64)",
    2: "paged decode bf16 (B64, L~U[512,4096], bs16, Hq32/Hkv8, D128)",
    3: "long-context split-KV decode bf16 (B8, L~U[32768,131072], bs16, Hq64/Hkv8, D64, "
       "sink, 2 layers: window 127 / none)",
    4: "varlen causal chunk prefill bf16 (B16, q~U[1,2048], prefix~U[0,8192], bs16, "
       "Hq32/Hkv8, D128, sink)",
    5: "mixed continuous batch bf16 (256 decode L~logU[128,16384] + 4x2048 prefill over "
       "4096 prefix, Hq32/Hkv8, D128, bs16)",
}


def seed_for(config: int) -> int:
    return 1000 + config


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def randn(shape, dtype, gen) -> torch.Tensor:
    """N(0,1) samples drawn in fp32 and rounded to ``dtype``."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def uniform_int(lo: int, hi: int, n: int, gen) -> torch.Tensor:
    """n integers uniform in [lo, hi], inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64)


def log_uniform_int(lo: int, hi: int, n: int, gen) -> torch.Tensor:
    """floor(exp(U(ln lo, ln hi))), clamped to [lo, hi]."""
    u = torch.rand(n, generator=gen, dtype=torch.float64)
    x = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return x.clamp(lo, hi).to(torch.int64)


@dataclass
class PagedPool:
    """A shuffled page pool and the block tables of the sequences that own pages."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: List[torch.Tensor]   # one int32 [n_seq, max_blocks] per group
    num_blocks: int
    block_size: int
    spare_blocks: List[int] = field(default_factory=list)


def build_pool(page_counts: List[List[int]], block_size: int, num_kv_heads: int,
               head_dim: int, dtype, gen, spare: int = 64, fill: bool = True,
               max_blocks: Optional[List[int]] = None) -> PagedPool:
    """Allocate pages for groups of sequences from one seeded, shuffled pool.

    page_counts[g][i] is the number of pages sequence i of group g needs.
    Returns a pool of sum(pages) + spare blocks; unowned pages hold NaN.
    """
    total = sum(sum(pc) for pc in page_counts)
    nb = total + spare
    perm = torch.randperm(nb, generator=gen).to(torch.int32)
    tables = []
    cursor = 0
    for gi, pc in enumerate(page_counts):
        mb = max(pc) if pc else 1
        if max_blocks is not None:
            mb = max(mb, max_blocks[gi])
        mb = max(mb, 1)
        bt = torch.full((len(pc), mb), -1, dtype=torch.int32)
        for i, n in enumerate(pc):
            bt[i, :n] = perm[cursor:cursor + n]
            cursor += n
        tables.append(bt)
    spare_ids = perm[cursor:].tolist()
    shape = (nb, block_size, num_kv_heads, head_dim)
    if fill:
        k = randn(shape, dtype, gen)
        v = randn(shape, dtype, gen)
    else:
        k = torch.zeros(shape, dtype=dtype)
        v = torch.zeros(shape, dtype=dtype)
    if spare_ids:
        idx = torch.tensor(spare_ids, dtype=torch.int64)
        k[idx] = float("nan")
        v[idx] = float("nan")
    return PagedPool(k, v, tables, nb, block_size, spare_ids)


def pages_for(length: int, block_size: int) -> int:
    return (length + block_size - 1) // block_size


@dataclass
class DecodeCase:
    name: str
    q: torch.Tensor              # [B, Hq, D]
    k_cache: torch.Tensor        # [num_blocks, bs, Hkv, D]
    v_cache: torch.Tensor
    block_table: torch.Tensor    # int32 [B, max_blocks]
    cache_seqlens: torch.Tensor  # int32 [B]
    sink: Optional[torch.Tensor] # float32 [Hq] or None
    window_left: int
    sm_scale: float
    partition_size: int = 512
    alibi: Optional[torch.Tensor] = None  # float32 [Hq] ALiBi slopes or None

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def num_qo_heads(self):
        return self.q.shape[1]

    @property
    def max_seqlen(self):
        return int(self.cache_seqlens.max()) if self.batch else 0


@dataclass
class VarlenCase:
    name: str
    q: torch.Tensor              # [total_q, Hq, D]
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor    # int32 [B, max_blocks]
    cu_seq_lens_q: torch.Tensor  # int32 [B+1]
    cu_seq_lens_k: torch.Tensor  # int32 [B+1]
    sink: Optional[torch.Tensor]
    window_left: int
    sm_scale: float
    causal: bool = True
    alibi: Optional[torch.Tensor] = None  # float32 [Hq] ALiBi slopes or None

    @property
    def batch(self):
        return self.cu_seq_lens_q.numel() - 1

    @property
    def q_lens(self):
        return (self.cu_seq_lens_q[1:] - self.cu_seq_lens_q[:-1])

    @property
    def kv_lens(self):
        return (self.cu_seq_lens_k[1:] - self.cu_seq_lens_k[:-1])

    @property
    def max_seqlen_q(self):
        return int(self.q_lens.max()) if self.batch else 0

    @property
    def max_seqlen_k(self):
        return int(self.kv_lens.max()) if self.batch else 0

    @property
    def total_q(self):
        return int(self.cu_seq_lens_q[-1])


def cumsum0(lens: torch.Tensor) -> torch.Tensor:
    out = torch.zeros(lens.numel() + 1, dtype=torch.int32)
    out[1:] = torch.cumsum(lens.to(torch.int64), 0).to(torch.int32)
    return out


def make_decode(lens, num_qo_heads, num_kv_heads, head_dim, block_size, dtype, seed,
                sink: str = "none", window_left: int = -1, sm_scale: Optional[float] = None,
                spare: int = 64, partition_size: int = 512, name: str = "decode",
                extra_blocks_per_seq: int = 0, alibi: str = "none") -> DecodeCase:
    """A decode batch over a shuffled pool.  sink: 'none' | 'randn' | 'zero';
    alibi: 'none' | 'geometric' | 'uniform' (see alibi_slopes)."""
    gen = _gen(seed)
    lens = [int(x) for x in lens]
    pc = [pages_for(L, block_size) + extra_blocks_per_seq for L in lens]
    pool = build_pool([pc], block_size, num_kv_heads, head_dim, dtype, gen, spare=spare)
    q = randn((len(lens), num_qo_heads, head_dim), dtype, gen)
    sk = _make_sink(sink, num_qo_heads, gen)
    scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim)
    return DecodeCase(name, q, pool.k_cache, pool.v_cache, pool.block_tables[0],
                      torch.tensor(lens, dtype=torch.int32), sk, window_left, scale,
                      partition_size, alibi_slopes(alibi, num_qo_heads, gen))


def alibi_slopes(kind: str, n: int, gen) -> Optional[torch.Tensor]:
    """ALiBi slopes for n query heads: 'geometric' = the ALiBi paper's
    2^(-8 (i+1) / n); 'uniform' = seeded U[0.01, 1] (steep and shallow heads
    mixed); 'steep' = seeded U[0.5, 2] (one key dominates each row); 'none' =
    no bias."""
    if kind == "none":
        return None
    if kind == "steep":
        return torch.rand(n, generator=gen, dtype=torch.float32) * 1.5 + 0.5
    if kind == "geometric":
        return torch.tensor([2.0 ** (-8.0 * (i + 1) / n) for i in range(n)], dtype=torch.float32)
    if kind == "uniform":
        return (torch.rand(n, generator=gen, dtype=torch.float32) * 0.99 + 0.01)
    raise ValueError(kind)


def _make_sink(kind: str, n: int, gen) -> Optional[torch.Tensor]:
    if kind == "none":
        return None
    if kind == "randn":
        return torch.randn(n, generator=gen, dtype=torch.float32)
    if kind == "zero":
        return torch.zeros(n, dtype=torch.float32)
    raise ValueError(kind)


def make_varlen(q_lens, prefix_lens, num_qo_heads, num_kv_heads, head_dim, block_size,
                dtype, seed, sink: str = "randn", window_left: int = -1,
                sm_scale: Optional[float] = None, spare: int = 64, causal: bool = True,
                name: str = "varlen", alibi: str = "none") -> VarlenCase:
    """A varlen chunk-prefill batch: request r has q_lens[r] new queries over
    prefix_lens[r] cached tokens plus the new tokens themselves (kv_len =
    prefix + q_len), all already in the pool."""
    gen = _gen(seed)
    ql = torch.tensor([int(x) for x in q_lens], dtype=torch.int32)
    pl = torch.tensor([int(x) for x in prefix_lens], dtype=torch.int32)
    kvl = ql + pl
    pc = [pages_for(int(L), block_size) for L in kvl]
    pool = build_pool([pc], block_size, num_kv_heads, head_dim, dtype, gen, spare=spare)
    q = randn((int(ql.sum()), num_qo_heads, head_dim), dtype, gen)
    sk = _make_sink(sink, num_qo_heads, gen)
    scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim)
    return VarlenCase(name, q, pool.k_cache, pool.v_cache, pool.block_tables[0],
                      cumsum0(ql), cumsum0(kvl), sk, window_left, scale, causal,
                      alibi_slopes(alibi, num_qo_heads, gen))


def make_varlen_kv(q_lens, kv_lens, num_qo_heads, num_kv_heads, head_dim, block_size, dtype,
                   seed, sink: str = "randn", window_left: int = -1,
                   sm_scale: Optional[float] = None, spare: int = 64, causal: bool = True,
                   name: str = "varlen", alibi: str = "none") -> VarlenCase:
    """A varlen batch with explicit per-request kv lengths (q_len may exceed
    kv_len; such rows sit at negative positions and attend to nothing)."""
    gen = _gen(seed)
    ql = torch.tensor([int(x) for x in q_lens], dtype=torch.int32)
    kvl = torch.tensor([int(x) for x in kv_lens], dtype=torch.int32)
    pc = [pages_for(int(L), block_size) for L in kvl]
    pool = build_pool([pc], block_size, num_kv_heads, head_dim, dtype, gen, spare=spare)
    q = randn((int(ql.sum()), num_qo_heads, head_dim), dtype, gen)
    sk = _make_sink(sink, num_qo_heads, gen)
    scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim)
    return VarlenCase(name, q, pool.k_cache, pool.v_cache, pool.block_tables[0],
                      cumsum0(ql), cumsum0(kvl), sk, window_left, scale, causal,
                      alibi_slopes(alibi, num_qo_heads, gen))


@dataclass
class RopeCase:
    """New tokens for the rotary step fused with the cache write."""
    name: str
    query: torch.Tensor           # [T, Hq, D]
    key: torch.Tensor             # [T, Hkv, D]
    value: torch.Tensor
    k_cache: torch.Tensor         # [num_blocks, bs, Hkv, D], NaN before the write
    v_cache: torch.Tensor
    positions: torch.Tensor       # int64 [T]
    slot_mapping: torch.Tensor    # int64 [T], distinct; some -1 (not cached)
    rotary_dim: int
    base: float
    position_scale: float
    neox: bool
    max_position: int
    ntk_alpha: float = 1.0        # NTK-aware context stretch of the rotary base (1: none)


def make_rope(num_tokens: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
              rotary_dim: int, block_size: int, dtype, seed: int, max_position: int = 8192,
              base: float = 10000.0, position_scale: float = 1.0, neox: bool = True,
              skip_every: int = 7, name: str = "rope", ntk_alpha: float = 1.0) -> RopeCase:
    """num_tokens tokens at uniform positions in [0, max_position) (the first
    two at 0 and max_position - 1), written to distinct random slots of a NaN
    pool with a quarter of spare room; every skip_every-th token has slot -1."""
    gen = _gen(seed)
    T = int(num_tokens)
    nb = max(1, pages_for(T + T // 4, block_size))
    q = randn((T, num_qo_heads, head_dim), dtype, gen)
    k = randn((T, num_kv_heads, head_dim), dtype, gen)
    v = randn((T, num_kv_heads, head_dim), dtype, gen)
    pos = torch.randint(0, max_position, (T,), generator=gen, dtype=torch.int64)
    if T > 0:
        pos[0] = 0
    if T > 1:
        pos[1] = max_position - 1
    slots = torch.randperm(nb * block_size, generator=gen)[:T].to(torch.int64)
    if skip_every > 0:
        slots[skip_every - 1::skip_every] = -1
    shape = (nb, block_size, num_kv_heads, head_dim)
    kc = torch.full(shape, float("nan"), dtype=dtype)
    vc = torch.full(shape, float("nan"), dtype=dtype)
    return RopeCase(name, q, k, v, kc, vc, pos, slots, int(rotary_dim), float(base),
                    float(position_scale), bool(neox), int(max_position), float(ntk_alpha))


def make_long_sequence(seq_len: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                       seed: int, n_stripes: int = 32, n_sinks: int = 4, dtype=torch.bfloat16):
    """One long sequence whose attention has the structure MInference's
    vertical + slash pattern targets (long-context LLM prefill): q and k share
    a component rotated by position (RoFormer rotation of the first half of
    the dims, frequencies 10000^(-2f/half)), so q_i . k_j peaks near i = j and
    decays with the distance (slash lines); the unrotated half of the query
    is a common direction that a few keys (the first n_sinks and n_stripes
    seeded columns) carry strongly (vertical lines); plus N(0, 1) noise.
    Returns q [S, Hq, D], k, v [S, Hkv, D] in dtype."""
    gen = _gen(seed)
    S, D = int(seq_len), int(head_dim)
    half = D // 2
    pos = torch.arange(S, dtype=torch.float64)[:, None]
    freq = torch.pow(10000.0, -2.0 * torch.arange(half // 2, dtype=torch.float64) / half)
    ang = pos * freq[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)  # [S, half/2]

    def rotate(x):  # x [S, H, half]: pairs (f, f + half/2) turned by pos * freq_f
        a, b = x[..., : half // 2], x[..., half // 2:]
        c, s_ = cos[:, None, :], sin[:, None, :]
        return torch.cat([a * c - b * s_, b * c + a * s_], dim=-1)

    base = torch.randn(num_kv_heads, half, generator=gen, dtype=torch.float64) * 1.5
    qdir = torch.randn(num_kv_heads, D - half, generator=gen, dtype=torch.float64)
    qdir = qdir / qdir.norm(dim=-1, keepdim=True) * 3.0
    G = num_qo_heads // num_kv_heads
    qr = base.repeat_interleave(G, 0)[None] + 0.5 * torch.randn(S, num_qo_heads, half,
                                                                 generator=gen,
                                                                 dtype=torch.float64)
    kr = base[None] + 0.5 * torch.randn(S, num_kv_heads, half, generator=gen,
                                        dtype=torch.float64)
    qu = qdir.repeat_interleave(G, 0)[None].expand(S, -1, -1) + 0.5 * torch.randn(
        S, num_qo_heads, D - half, generator=gen, dtype=torch.float64)
    ku = 0.5 * torch.randn(S, num_kv_heads, D - half, generator=gen, dtype=torch.float64)
    cols = torch.cat([torch.arange(min(n_sinks, S)),
                      torch.randperm(S, generator=gen)[:n_stripes]]).unique()
    ku[cols] += qdir[None] * 12.0
    q = torch.cat([rotate(qr), qu], dim=-1)
    k = torch.cat([rotate(kr), ku], dim=-1)
    v = torch.randn(S, num_kv_heads, D, generator=gen, dtype=torch.float64)
    return q.to(dtype), k.to(dtype), v.to(dtype)


# ---------------------------------------------------------------------------
# the five serving configurations
# ---------------------------------------------------------------------------

def config1_tiny(variant: str = "attend") -> DecodeCase:
    """The decode worked example as a tiny fp32 problem: 8-block pool with
    blocks 4 and 7 unowned (NaN), 4 query / 2 kv heads, head_dim 64,
    sm_scale 1/8, sink ~ N(0,1), no window.

    variant 'attend': attend over cache_seqlens [30, 32, 70].
    variant 'append': also returns the new token's K/V, to be written first,
    after which the batch attends over [31, 33, 71].
    """
    gen = _gen(seed_for(1))
    Hq, Hkv, D, bs = 4, 2, 64, EXAMPLE_BLOCK_SIZE
    shape = (EXAMPLE_NUM_BLOCKS, bs, Hkv, D)
    k = randn(shape, torch.float32, gen)
    v = randn(shape, torch.float32, gen)
    for b in (4, 7):
        k[b] = float("nan")
        v[b] = float("nan")
    q = randn((3, Hq, D), torch.float32, gen)
    sink = torch.randn(Hq, generator=gen, dtype=torch.float32)
    new_k = randn((3, Hkv, D), torch.float32, gen)
    new_v = randn((3, Hkv, D), torch.float32, gen)
    lens = list(EXAMPLE_CACHE_SEQLENS)
    case = DecodeCase("config1-" + variant, q, k, v,
                      torch.tensor(EXAMPLE_BLOCK_TABLE, dtype=torch.int32),
                      torch.tensor(lens, dtype=torch.int32), sink, -1, 1.0 / 8.0)
    case.new_k = new_k
    case.new_v = new_v
    return case


def config2_decode() -> DecodeCase:
    gen = _gen(seed_for(2))
    lens = uniform_int(512, 4096, 64, gen).tolist()
    return make_decode(lens, 32, 8, 128, 16, torch.bfloat16, seed_for(2) + 100, sink="none",
                       window_left=-1, sm_scale=1.0 / math.sqrt(128), name="config2")


def config3_long(layer: int) -> DecodeCase:
    """Layer 0 (even): window_left 127; layer 1 (odd): no window.  Both layers
    share lengths and block tables; each has its own q, pool values and sink."""
    gen = _gen(seed_for(3))
    lens = uniform_int(32768, 131072, 8, gen).tolist()
    return make_decode(lens, 64, 8, 64, 16, torch.bfloat16, seed_for(3) + 100 + layer,
                       sink="randn", window_left=127 if layer % 2 == 0 else -1,
                       sm_scale=1.0 / 8.0, name=f"config3-layer{layer}")


def config3_lengths() -> List[int]:
    return uniform_int(32768, 131072, 8, _gen(seed_for(3))).tolist()


def config4_prefill(num_qo_heads: int = 32, num_kv_heads: int = 8,
                    head_dim: int = 128) -> VarlenCase:
    """B16 varlen prefill: q ~ U[1, 2048], prefix ~ U[0, 8192] (the lengths do
    not depend on the head shape; head_dim 256 with 16 query heads is the
    same work as 128 with 32)."""
    gen = _gen(seed_for(4))
    ql = uniform_int(1, 2048, 16, gen).tolist()
    pl = uniform_int(0, 8192, 16, gen).tolist()
    return make_varlen(ql, pl, num_qo_heads, num_kv_heads, head_dim, 16, torch.bfloat16,
                       seed_for(4) + 100, sink="randn", window_left=-1,
                       sm_scale=1.0 / math.sqrt(head_dim), name="config4")


@dataclass
class MixedCase:
    """One continuous-batching step: write all new K/V, then decode, then prefill."""
    name: str
    key: torch.Tensor             # [T, Hkv, D] new keys (decode tokens first)
    value: torch.Tensor
    slot_mapping: torch.Tensor    # int64 [T]
    k_cache: torch.Tensor         # pool before the write (new slots hold stale data)
    v_cache: torch.Tensor
    decode: DecodeCase            # attends over cache length + 1
    prefill: VarlenCase
    positions: Optional[torch.Tensor] = None  # int64 [T]: position of each new token

    @property
    def num_new_tokens(self):
        return self.key.shape[0]


def make_mixed(dec_lens, chunk_q: int, chunk_prefix: int, n_chunks: int, num_qo_heads: int,
               num_kv_heads: int, head_dim: int, block_size: int, dtype, seed: int,
               name: str = "mixed") -> MixedCase:
    """dec_lens: cached lengths of the decode sequences (each appends 1 token);
    n_chunks prefill requests of chunk_q new tokens over chunk_prefix cached."""
    gen = _gen(seed)
    dec_lens = [int(x) for x in dec_lens]
    B = len(dec_lens)
    dec_pages = [pages_for(L + 1, block_size) for L in dec_lens]
    kv_pre = chunk_prefix + chunk_q
    pre_pages = [pages_for(kv_pre, block_size)] * n_chunks
    pool = build_pool([dec_pages, pre_pages], block_size, num_kv_heads, head_dim, dtype,
                      gen, spare=64)
    dec_bt, pre_bt = pool.block_tables
    # slots of the new tokens: position L_b of decode sequence b, then
    # positions chunk_prefix .. kv_pre-1 of each prefill request
    slots, positions = [], []
    for b, L in enumerate(dec_lens):
        slots.append(int(dec_bt[b, L // block_size]) * block_size + L % block_size)
        positions.append(L)
    for r in range(n_chunks):
        for p in range(chunk_prefix, kv_pre):
            slots.append(int(pre_bt[r, p // block_size]) * block_size + p % block_size)
            positions.append(p)
    T = len(slots)
    key = randn((T, num_kv_heads, head_dim), dtype, gen)
    value = randn((T, num_kv_heads, head_dim), dtype, gen)
    scale = 1.0 / math.sqrt(head_dim)
    q_dec = randn((B, num_qo_heads, head_dim), dtype, gen)
    q_pre = randn((n_chunks * chunk_q, num_qo_heads, head_dim), dtype, gen)
    dec = DecodeCase(name + "-decode", q_dec, pool.k_cache, pool.v_cache, dec_bt,
                     torch.tensor([L + 1 for L in dec_lens], dtype=torch.int32), None, -1,
                     scale)
    ql = torch.full((n_chunks,), chunk_q, dtype=torch.int32)
    kvl = torch.full((n_chunks,), kv_pre, dtype=torch.int32)
    pre = VarlenCase(name + "-prefill", q_pre, pool.k_cache, pool.v_cache, pre_bt,
                     cumsum0(ql), cumsum0(kvl), None, -1, scale, True)
    return MixedCase(name, key, value, torch.tensor(slots, dtype=torch.int64),
                     pool.k_cache, pool.v_cache, dec, pre,
                     torch.tensor(positions, dtype=torch.int64))


def config5_mixed() -> MixedCase:
    gen = _gen(seed_for(5))
    dec_lens = log_uniform_int(128, 16384, 256, gen).tolist()
    return make_mixed(dec_lens, 2048, 4096, 4, 32, 8, 128, 16, torch.bfloat16,
                      seed_for(5) + 100, name="config5")


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bits (the oracle's bf16 input form)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def to_oracle(t: torch.Tensor):
    """numpy array the oracle accepts: float32 as is, bf16 as raw bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)
