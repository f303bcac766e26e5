"""Seeded synthetic inputs for paged decode attention.

This module is the only code that the CUDA path and the CPU oracle share, and
it holds none of the method's arithmetic: it draws random numbers, lays them
out as block pools, block tables and context lengths, and nothing else.

Recipe (the same for every configuration):
* ``numpy.random.default_rng([seed, stream])``, seed = 1000 + configuration
  index, one sub-stream each for q, K, V, block placement, context lengths and
  outliers;
* q, K, V drawn as float32 N(0, 1) and cast to fp16 (round to nearest even);
* every physical block that some sequence uses is filled in all 16 slots;
  slots past the context end in a sequence's last block ("padding slots") are
  overwritten with NaN when ``nan_padding`` is set, and blocks that no
  sequence uses are NaN, so that a wrong gather or a missing mask shows up as a
  NaN in the output;
* each sequence takes consecutive entries of ``rng.permutation(num_blocks)``
  as its physical blocks (non-contiguous placement); unused table entries are
  -1;
* softmax scale 1/sqrt(head_dim).

Configurations (sizes of the workloads this library is measured on):
  c1_tiny           2 seqs, ctx [37, 16], 8 q / 2 kv heads, d 64, 16 blocks
  c2_8x512          8 x 512, 8 / 8 heads, d 128, 4096 blocks
  c3_32x1024_heavy  32 x 1024, 8 / 8, d 128, 16384 blocks, K heavy-tailed:
                    exactly round(0.001 * numel) K elements x10 before the
                    fp16 cast, V N(0, 1)
  c4_qwen2_b{1,4,8} 14 q / 2 kv heads, d 64, ctx 512, the first 16 blocks of
                    every table are the same physical blocks (shared prefix,
                    refcount = batch), 1024 blocks
  c5a_64x2048       64 x 2048, 32 q / 8 kv heads, d 128, 65536 blocks
  c5b_256_ragged    256 seqs, ctx ~ uniform integers [1, 4096], same heads and
                    pool

``append_tokens`` draws the new K/V rows of an append step (N(0, 1) fp16);
``eviction_state`` draws reference counts and last-use ticks of a block pool
for eviction scoring.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BLOCK_SIZE = 16


@dataclasses.dataclass
class DecodeWorkload:
    name: str
    query: np.ndarray          # [N][Hq][d] fp16
    k_pool: np.ndarray         # [NB][Hkv][B][d] fp16
    v_pool: np.ndarray         # [NB][Hkv][B][d] fp16
    block_tables: np.ndarray   # [N][MB] int32, -1 where unused
    context_lens: np.ndarray   # [N] int32
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    softmax_scale: float
    used_block_ids: np.ndarray  # distinct physical blocks some table uses

    @property
    def num_seqs(self) -> int:
        return int(self.query.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    def tail_block_ids(self) -> np.ndarray:
        """Physical block holding each sequence's newest token (ctx > 0 only)."""
        ids = []
        for s, c in enumerate(self.context_lens.tolist()):
            if c > 0:
                ids.append(int(self.block_tables[s, (c - 1) // self.block_size]))
        return np.asarray(ids, dtype=np.int32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def _normal_f16(rng, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16)


def build(name: str, *, num_heads: int, num_kv_heads: int, head_dim: int,
          num_blocks: int, context_lens, seed: int,
          shared_prefix_blocks: int = 0, heavy_tail: bool = False,
          nan_padding: bool = True, block_size: int = BLOCK_SIZE,
          max_blocks_per_seq: Optional[int] = None, q_std: float = 1.0,
          k_mult: float = 1.0, v_mult: float = 1.0,
          v_hot_mult: float = 1.0) -> DecodeWorkload:
    """Lay out one synthetic decode batch.  See the module docstring.

    Magnitude options (all applied to the float32 draws before the fp16
    cast; the defaults leave the draws unchanged): q ~ N(0, q_std^2); every K
    value times ``k_mult``; every V value times ``v_mult``; and, when
    ``v_hot_mult`` != 1, the V values of one seeded block of each sequence
    (its own sub-stream) times ``v_hot_mult`` as well, so that the blocks of
    one sequence hold V of very different magnitudes.
    """
    ctx = np.asarray(context_lens, dtype=np.int32)
    n = int(ctx.size)
    nblk = [(int(c) + block_size - 1) // block_size for c in ctx]
    mb = max_blocks_per_seq if max_blocks_per_seq is not None else max(nblk + [1])
    perm = _rng(seed, 3).permutation(num_blocks).astype(np.int32)
    tables = np.full((n, mb), -1, dtype=np.int32)
    shared = perm[:shared_prefix_blocks]
    off = shared_prefix_blocks
    for s in range(n):
        k = nblk[s]
        ps = min(shared_prefix_blocks, k)
        tables[s, :ps] = shared[:ps]
        own = k - ps
        if off + own > num_blocks:
            raise ValueError("pool too small for the requested contexts")
        tables[s, ps:k] = perm[off:off + own]
        off += own
    used = np.unique(tables[tables >= 0]).astype(np.int32)

    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_pool = np.full(shape, np.nan, dtype=np.float16)
    v_pool = np.full(shape, np.nan, dtype=np.float16)
    used_shape = (used.size, num_kv_heads, block_size, head_dim)
    k_used = _rng(seed, 1).standard_normal(used_shape, dtype=np.float32)
    if heavy_tail and k_used.size:
        n_out = int(round(0.001 * k_used.size))
        pos = _rng(seed, 5).choice(k_used.size, size=n_out, replace=False)
        k_used.reshape(-1)[pos] *= 10.0
    if k_mult != 1.0:
        k_used *= np.float32(k_mult)
    k_pool[used] = k_used.astype(np.float16)
    del k_used
    v_used = _rng(seed, 2).standard_normal(used_shape, dtype=np.float32)
    if v_mult != 1.0:
        v_used *= np.float32(v_mult)
    if v_hot_mult != 1.0:
        rng_hot = _rng(seed, 9)
        hot = set()
        for s in range(n):
            if nblk[s] > 0:
                hot.add(int(tables[s, int(rng_hot.integers(0, nblk[s]))]))
        rows = np.searchsorted(used, np.asarray(sorted(hot), dtype=np.int32))
        v_used[rows] *= np.float32(v_hot_mult)
    v_pool[used] = v_used.astype(np.float16)
    del v_used

    if nan_padding:
        for s in range(n):
            c = int(ctx[s])
            if c > 0 and c % block_size:
                last = tables[s, (c - 1) // block_size]
                k_pool[last, :, c % block_size:, :] = np.nan
                v_pool[last, :, c % block_size:, :] = np.nan

    q32 = _rng(seed, 0).standard_normal((n, num_heads, head_dim), dtype=np.float32)
    if q_std != 1.0:
        q32 *= np.float32(q_std)
    query = q32.astype(np.float16)
    return DecodeWorkload(
        name=name, query=query, k_pool=k_pool, v_pool=v_pool,
        block_tables=tables, context_lens=ctx, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size,
        softmax_scale=1.0 / math.sqrt(head_dim), used_block_ids=used)


CONFIG_NAMES = ("c1_tiny", "c2_8x512", "c3_32x1024_heavy", "c4_qwen2_b1",
                "c4_qwen2_b4", "c4_qwen2_b8", "c5a_64x2048", "c5b_256_ragged")


def make(name: str, nan_padding: bool = True) -> DecodeWorkload:
    """One of the named configurations (module docstring)."""
    if name == "c1_tiny":
        return build(name, num_heads=8, num_kv_heads=2, head_dim=64, num_blocks=16,
                     context_lens=[37, 16], seed=1001, nan_padding=nan_padding)
    if name == "c2_8x512":
        return build(name, num_heads=8, num_kv_heads=8, head_dim=128, num_blocks=4096,
                     context_lens=[512] * 8, seed=1002, nan_padding=nan_padding)
    if name == "c3_32x1024_heavy":
        return build(name, num_heads=8, num_kv_heads=8, head_dim=128, num_blocks=16384,
                     context_lens=[1024] * 32, seed=1003, heavy_tail=True,
                     nan_padding=nan_padding)
    if name.startswith("c4_qwen2_b"):
        b = int(name[len("c4_qwen2_b"):])
        return build(name, num_heads=14, num_kv_heads=2, head_dim=64, num_blocks=1024,
                     context_lens=[512] * b, seed=1004, shared_prefix_blocks=16,
                     nan_padding=nan_padding)
    if name == "c5a_64x2048":
        return build(name, num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=65536,
                     context_lens=[2048] * 64, seed=1005, nan_padding=nan_padding)
    if name == "c5b_256_ragged":
        lens = _rng(1006, 4).integers(1, 4096, size=256, endpoint=True)
        return build(name, num_heads=32, num_kv_heads=8, head_dim=128, num_blocks=65536,
                     context_lens=lens, seed=1006, max_blocks_per_seq=256,
                     nan_padding=nan_padding)
    raise KeyError(name)


def random_case(seed: int, *, num_seqs: int, num_heads: int, num_kv_heads: int,
                head_dim: int, context_lens=None, max_ctx: int = 100,
                extra_blocks: int = 3, nan_padding: bool = True,
                block_size: int = BLOCK_SIZE, **magnitudes) -> DecodeWorkload:
    """A small seeded case for parity and edge-case tests (``magnitudes``:
    the q_std / k_mult / v_mult / v_hot_mult options of ``build``)."""
    if context_lens is None:
        context_lens = _rng(seed, 4).integers(0, max_ctx, size=num_seqs, endpoint=True)
    ctx = np.asarray(context_lens, dtype=np.int32)
    need = sum((int(c) + block_size - 1) // block_size for c in ctx)
    return build(f"random_{seed}", num_heads=num_heads, num_kv_heads=num_kv_heads,
                 head_dim=head_dim, num_blocks=max(need + extra_blocks, 1),
                 context_lens=ctx, seed=seed, nan_padding=nan_padding,
                 block_size=block_size, **magnitudes)


def append_tokens(w: DecodeWorkload, seed: int):
    """New-token inputs for an append into ``w``'s pools.

    Each sequence with context length c > 0 appends its token at position
    c - 1 (so the table already holds the block, and a decode over c tokens
    reads it); c == 0 gives position -1 (no token).  Returns (k_new, v_new
    [N][Hkv][d] fp16 drawn N(0, 1), positions [N] int32).
    """
    n, hkv, d = w.num_seqs, w.num_kv_heads, w.head_dim
    k_new = _normal_f16(_rng(seed, 6), (n, hkv, d))
    v_new = _normal_f16(_rng(seed, 7), (n, hkv, d))
    positions = (w.context_lens.astype(np.int64) - 1).astype(np.int32)
    return k_new, v_new, positions


@dataclasses.dataclass
class EvictionState:
    refcnt: np.ndarray      # [NB] int32; 0 = free block
    last_used: np.ndarray   # [NB] int64 tick of the last decode step that read it
    current_tick: int


def eviction_state(num_blocks: int, seed: int, *, free_fraction: float = 0.1,
                   current_tick: int = 100_000, max_age: int = 4096) -> EvictionState:
    """Seeded block-manager state to score for eviction.

    refcnt: 0 (free) with probability ``free_fraction``, else 1 + a
    geometric(0.6) count capped at 16 (most blocks owned by one sequence, a
    few shared prefixes); last_used: current_tick minus a uniform integer age
    in [0, max_age].  Both are small integers, so equal scores are common.
    """
    rng = _rng(seed, 8)
    ref = np.minimum(rng.geometric(0.6, size=num_blocks), 16).astype(np.int32)
    ref[rng.random(num_blocks) < free_fraction] = 0
    age = rng.integers(0, max_age, size=num_blocks, endpoint=True)
    last = (current_tick - age).astype(np.int64)
    return EvictionState(refcnt=ref, last_used=last, current_tick=int(current_tick))


def shard_sequences(num_seqs: int, rank: int, world_size: int) -> range:
    """Contiguous sequence range of one rank when a batch is split across GPUs.

    Decode attention of different sequences is independent, so a multi-GPU
    batch is split by sequence with no exchange between ranks.
    """
    if world_size <= 0 or not 0 <= rank < world_size:
        raise ValueError("bad rank/world size")
    lo = (num_seqs * rank) // world_size
    hi = (num_seqs * (rank + 1)) // world_size
    return range(lo, hi)
