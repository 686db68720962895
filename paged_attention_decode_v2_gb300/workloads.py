"""Seeded synthetic decode batches shaped like the workloads on the pages.

This module only draws random inputs (queries, paged key/value pools, block
tables, sequence lengths).  It holds none of the attention arithmetic, so the
CUDA path and the float64 oracle can both consume what it produces without
sharing any computation.

Each workload is described by a :class:`Workload`; :func:`make` draws one.
Shapes follow the decode setting on the pages: 24 query heads over 4 KV heads
with head_dim 256 and 16-token blocks (commit 4eb83a7e "qwen3_6_scripts",
paragraphs "Prefill (flash_attn_func)" and "Hardware testing confirmed"), up
to ~100K-token contexts split into 512- or 1024-token partitions (commit
1a4e1005 "paged_attn.py", "PARTITION_SIZE 512->1024").
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    partition_sizes: tuple
    seed: int
    seq_lens: Callable[[torch.Generator], torch.Tensor]
    pool_blocks: Optional[int] = None     # None: ceil(1.1 * blocks the batch needs)
    key_outlier_frac: float = 0.0         # fraction of tokens whose K rows are scaled
    key_outlier_scale: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads


def _fixed(n: int, length: int):
    return lambda g: torch.full((n,), length, dtype=torch.int32)


def _mixed_uniform(n: int, hi: int, forced=(1, 8192, 8193)):
    def f(g):
        lens = torch.randint(1, hi + 1, (n,), generator=g, dtype=torch.int64)
        for i, v in enumerate(forced):
            lens[i] = v
        return lens.to(torch.int32)
    return f


def _lognormal(n: int, median: float, sigma: float, lo: int, hi: int):
    def f(g):
        z = torch.randn((n,), generator=g, dtype=torch.float64)
        lens = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
        return lens.to(torch.int32)
    return f


# The five decode batches, in order (tiny fp32 first: the one the oracle runs
# in milliseconds).
WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", torch.float32, 1, 2, 1, 64, 16, (32,), 1001, _fixed(1, 100), pool_blocks=64),
    "gqa_8k": Workload(
        "gqa_8k", torch.bfloat16, 1, 24, 4, 256, 16, (512,), 1002, _fixed(1, 8192),
        pool_blocks=600),
    "long_100k": Workload(
        "long_100k", torch.bfloat16, 1, 24, 4, 256, 16, (512, 1024), 1003, _fixed(1, 100000),
        key_outlier_frac=0.001, key_outlier_scale=30.0),
    "mixed_32": Workload(
        "mixed_32", torch.bfloat16, 32, 24, 4, 256, 16, (512,), 1004, _mixed_uniform(32, 32768)),
    "serving_256": Workload(
        "serving_256", torch.bfloat16, 256, 32, 8, 128, 32, (512,), 1005,
        _lognormal(256, 2048.0, 1.2, 16, 131072)),
}


def scaled(w: Workload, *, name=None, num_seqs=None, seq_len=None, max_len=None,
           partition_sizes=None, pool_blocks=None, dtype=None) -> Workload:
    """A smaller copy of ``w`` with the same head shapes (for oracle-speed tests)."""
    lens = w.seq_lens
    if seq_len is not None:
        lens = _fixed(num_seqs or w.num_seqs, seq_len)
    elif max_len is not None:
        n = num_seqs or w.num_seqs
        lens = lambda g, n=n, hi=max_len: torch.randint(1, hi + 1, (n,), generator=g,
                                                        dtype=torch.int64).to(torch.int32)
    return dataclasses.replace(
        w, name=name or (w.name + "_scaled"), num_seqs=num_seqs or w.num_seqs, seq_lens=lens,
        partition_sizes=partition_sizes or w.partition_sizes, pool_blocks=pool_blocks,
        dtype=dtype or w.dtype)


@dataclasses.dataclass
class Batch:
    """One decode step's inputs.  All tensors live on one device."""
    workload: Workload
    q: torch.Tensor              # [B, Hq, D]
    k_cache: torch.Tensor        # [NB, Hkv, BS, D]
    v_cache: torch.Tensor        # [NB, Hkv, BS, D]
    block_tables: torch.Tensor   # int32 [B, MB]
    seq_lens: torch.Tensor       # int32 [B]
    max_seq_len: int

    @property
    def scale(self) -> float:
        return self.workload.scale

    def kv_bytes(self) -> int:
        """Key+value bytes the batch's tokens occupy (each read once per step)."""
        w = self.workload
        per_tok = 2 * w.num_kv_heads * w.head_dim * self.k_cache.element_size()
        return int(self.seq_lens.to(torch.int64).sum().item()) * per_tok

    def q_bytes(self) -> int:
        return self.q.numel() * self.q.element_size()

    def to(self, device) -> "Batch":
        return dataclasses.replace(
            self, q=self.q.to(device), k_cache=self.k_cache.to(device),
            v_cache=self.v_cache.to(device), block_tables=self.block_tables.to(device),
            seq_lens=self.seq_lens.to(device))


def make(w: Workload, device="cpu", *, seed: Optional[int] = None, poison: bool = False,
         table_pad: int = 0) -> Batch:
    """Draw one batch of ``w``.

    ``poison=True`` writes NaN into every pool block no sequence owns, into the
    slots past each sequence's last token, and -1 into block-table entries past
    each sequence's last block, so a kernel that reads anything outside the
    batch's tokens produces NaN.  ``table_pad`` adds that many extra (-1 or
    unused-block) columns to the block table.
    """
    seed = w.seed if seed is None else seed
    g_cpu = torch.Generator().manual_seed(seed)
    lens = w.seq_lens(g_cpu).to(torch.int32)
    B, BS = w.num_seqs, w.block_size
    blocks_needed = [(int(L) + BS - 1) // BS for L in lens.tolist()]
    total = sum(blocks_needed)
    nb = w.pool_blocks if w.pool_blocks is not None else max(1, math.ceil(1.1 * total))
    if nb < total:
        raise ValueError(f"{w.name}: pool of {nb} blocks < {total} needed")
    max_len = int(lens.max().item()) if B else 0
    mb = max(1, (max_len + BS - 1) // BS) + table_pad
    perm = torch.randperm(nb, generator=g_cpu).to(torch.int32)
    table = torch.full((B, mb), -1 if poison else 0, dtype=torch.int32)
    used = torch.zeros(nb, dtype=torch.bool)
    pos = 0
    for b, n in enumerate(blocks_needed):
        table[b, :n] = perm[pos:pos + n]
        used[perm[pos:pos + n].long()] = True
        if not poison and n < mb:
            # unused tail entries point at valid blocks that are not this sequence's
            table[b, n:] = perm[(pos + n) % nb]
        pos += n

    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed + 7)
    shape = (nb, w.num_kv_heads, BS, w.head_dim)
    k = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    q = torch.randn((B, w.num_heads, w.head_dim), generator=g, device=dev, dtype=torch.float32)
    if w.key_outlier_frac > 0 and B:
        # scale the K rows (all KV heads) of a seeded sample of token positions
        n_out = max(1, int(round(w.key_outlier_frac * max_len)))
        for b in range(B):
            L = int(lens[b])
            pos_t = torch.randperm(L, generator=g_cpu)[:min(n_out, L)]
            blk = table[b, (pos_t // BS).long()].long().to(dev)
            off = (pos_t % BS).long().to(dev)
            k[blk, :, off, :] *= w.key_outlier_scale
    k = k.to(w.dtype)
    v = v.to(w.dtype)
    q = q.to(w.dtype)
    if poison:
        nan = torch.tensor(float("nan"), dtype=w.dtype, device=dev)
        unused = (~used).nonzero().flatten().to(dev)
        k[unused] = nan
        v[unused] = nan
        for b, n in enumerate(blocks_needed):
            L = int(lens[b])
            if n and L % BS:
                last = int(table[b, n - 1])
                k[last, :, L % BS:, :] = nan
                v[last, :, L % BS:, :] = nan
    return Batch(w, q, k, v, table.to(dev), lens.to(dev), max_len)


# ---------------------------------------------------------------------------
# Paged prefix prefill: a chunk of new tokens per sequence after a cached
# context (commit 1a4e1005 "paged_attn.py", opening paragraph; commit
# 4eb83a7e "qwen3_6_scripts", paragraph "Complete rewrite of
# qwen3_6_scripts/paged_attn.py", item 1).  Chunks of up to 8192 tokens
# follow the serving configuration on the same page (max-num-batched-tokens
# 8192 -> 16384 / 32768).
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    dtype: torch.dtype
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    seed: int
    ctx_lens: Callable[[torch.Generator], torch.Tensor]   # cached tokens per sequence
    new_lens: Callable[[torch.Generator], torch.Tensor]   # chunk tokens per sequence

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


@dataclasses.dataclass
class PrefillBatch:
    """One prefill step's inputs.  All tensors live on one device."""
    workload: PrefillWorkload
    q: torch.Tensor              # [T, Hq, D]
    k: torch.Tensor              # [T, Hkv, D]  the chunk's keys
    v: torch.Tensor              # [T, Hkv, D]  the chunk's values
    k_cache: torch.Tensor        # [NB, Hkv, BS, D]  the cached context
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # int32 [B, MB]
    query_start: torch.Tensor    # int32 [B + 1]
    ctx_lens: torch.Tensor       # int32 [B]
    max_query_len: int
    max_ctx_len: int

    @property
    def scale(self) -> float:
        return self.workload.scale

    def to(self, device) -> "PrefillBatch":
        return dataclasses.replace(
            self, q=self.q.to(device), k=self.k.to(device), v=self.v.to(device),
            k_cache=self.k_cache.to(device), v_cache=self.v_cache.to(device),
            block_tables=self.block_tables.to(device), query_start=self.query_start.to(device),
            ctx_lens=self.ctx_lens.to(device))


def _lens(values):
    vals = tuple(int(x) for x in values)
    return lambda g: torch.tensor(vals, dtype=torch.int32)


PREFILL_WORKLOADS = {
    # one 8192-token chunk after 24576 cached tokens, the decode shapes' heads
    "prefill_32k": PrefillWorkload(
        "prefill_32k", torch.bfloat16, 1, 24, 4, 256, 16, 2001, _lens([24576]), _lens([8192])),
    # a mixed batch: four chunks of different sizes over different contexts
    "prefill_mixed": PrefillWorkload(
        "prefill_mixed", torch.bfloat16, 4, 24, 4, 256, 16, 2002,
        _lens([0, 5000, 12000, 30000]), _lens([2048, 1000, 3000, 500])),
}


def prefill_problem(dtype=torch.bfloat16, ctx=(100,), new=(37,), Hq=6, Hkv=2, D=128, BS=16,
                    seed=0) -> PrefillWorkload:
    """A small prefill workload with the given per-sequence lengths."""
    return PrefillWorkload("prefill_pin", dtype, len(ctx), Hq, Hkv, D, BS, seed, _lens(ctx),
                           _lens(new))


def make_prefill(w: PrefillWorkload, device="cpu", *, poison: bool = False) -> PrefillBatch:
    """Draw one prefill batch of ``w``.

    The cache holds each sequence's context in blocks taken from a seeded
    permutation of the pool; the chunk's q, k and v are separate tensors.
    ``poison=True`` writes NaN into every pool block no context owns and into
    the slots past each context's last token, and -1 into block-table entries
    past the last context block.
    """
    g_cpu = torch.Generator().manual_seed(w.seed)
    ctx = w.ctx_lens(g_cpu).to(torch.int32)
    new = w.new_lens(g_cpu).to(torch.int32)
    B, BS = w.num_seqs, w.block_size
    blocks_needed = [(int(c) + BS - 1) // BS for c in ctx.tolist()]
    total = sum(blocks_needed)
    nb = max(1, math.ceil(1.1 * total))
    mb = max(1, max(blocks_needed) if B else 1)
    perm = torch.randperm(nb, generator=g_cpu).to(torch.int32)
    table = torch.full((B, mb), -1 if poison else 0, dtype=torch.int32)
    used = torch.zeros(nb, dtype=torch.bool)
    pos = 0
    for b, n in enumerate(blocks_needed):
        table[b, :n] = perm[pos:pos + n]
        used[perm[pos:pos + n].long()] = True
        pos += n
    qs = torch.zeros(B + 1, dtype=torch.int32)
    qs[1:] = torch.cumsum(new, 0).to(torch.int32)
    T = int(qs[-1])

    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(w.seed + 7)
    shape = (nb, w.num_kv_heads, BS, w.head_dim)
    k_cache = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(w.dtype)
    v_cache = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(w.dtype)
    q = torch.randn((T, w.num_heads, w.head_dim), generator=g, device=dev,
                    dtype=torch.float32).to(w.dtype)
    k = torch.randn((T, w.num_kv_heads, w.head_dim), generator=g, device=dev,
                    dtype=torch.float32).to(w.dtype)
    v = torch.randn((T, w.num_kv_heads, w.head_dim), generator=g, device=dev,
                    dtype=torch.float32).to(w.dtype)
    if poison:
        nan = torch.tensor(float("nan"), dtype=w.dtype, device=dev)
        unused = (~used).nonzero().flatten().to(dev)
        k_cache[unused] = nan
        v_cache[unused] = nan
        for b, n in enumerate(blocks_needed):
            C = int(ctx[b])
            if n and C % BS:
                last = int(table[b, n - 1])
                k_cache[last, :, C % BS:, :] = nan
                v_cache[last, :, C % BS:, :] = nan
    return PrefillBatch(w, q, k, v, k_cache, v_cache, table.to(dev), qs.to(dev), ctx.to(dev),
                        int(new.max()) if B else 0, int(ctx.max()) if B else 0)
