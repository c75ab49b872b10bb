"""Seeded synthetic inputs for paged KV decode attention.

This module is the one piece shared by the oracle tests, the GPU tests and
the benchmark.  It only draws random numbers and lays out inputs the way a
caller of the library would (block pool, block tables, context lengths, slot
mapping of the new tokens); it holds none of the attention arithmetic.

Workload shapes follow the design conditions of the web textbook page
"Chapter 8: Inference Optimization" (clxhxhhr.top/posts/4341):
  - chapter opening, design-condition table: short chats of 2048 input
    tokens, long requests of 8192 input tokens whose first 6144 tokens are a
    common prefix, 256 output tokens each;
  - §8.1.2: Qwen3-8B attention shapes (36 layers, 8 KV heads x 128 dims,
    BF16), 16-token blocks, a 12 GiB KV pool, 37 short requests fit in it;
  - §8.3.1/§8.3.2: blocks scattered through a pool via a block table; a
    common prefix stored once and referenced by every sharer;
  - §8.2.3: chunks of c new tokens after h cached tokens.
Values are N(0, 1) drawn with NumPy's PCG64 in float32 and rounded to BF16
(round to nearest even).  Generated-so-far counts are U{0..255} inclusive, so
the longest contexts are 2048 + 255 = 2303 and 8192 + 255 = 8447 tokens.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BLOCK_SIZE = 16
HEAD_DIM = 128
NUM_KV_HEADS = 8
NUM_Q_HEADS = 32
NUM_LAYERS = 36
SCALE = float(np.float32(1.0 / math.sqrt(HEAD_DIM)))
# 12 GiB pool spread over 36 layers, K and V of one 16-token block per layer:
# 2 * 8 * 16 * 128 * 2 B = 64 KiB per block per layer.
POOL_BLOCKS_12GIB = (12 * 1024**3) // (NUM_LAYERS * 2 * NUM_KV_HEADS * BLOCK_SIZE * HEAD_DIM * 2)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) BF16 bit patterns of the given shape."""
    return bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclasses.dataclass
class Workload:
    """One layer-call worth of inputs, all as host NumPy arrays.

    k_cache/v_cache: uint16 [num_blocks][Hkv][16][D] (None when the caller
    fills the pool itself, e.g. on the device for very large pools).
    q: uint16 [B][q_len][Hq][D].  block_tables: int32 [B][max_blocks].
    context_lens: int32 [B] (includes the q_len new tokens).
    k_new/v_new: uint16 [T][Hkv][D] with slot_mapping int64 [T]: the K/V of
    the tokens this step stores before attending (T = B*q_len, padding rows
    get slot -1).
    """

    name: str
    num_blocks: int
    block_tables: np.ndarray
    context_lens: np.ndarray
    q_len: int
    q: Optional[np.ndarray]
    k_cache: Optional[np.ndarray]
    v_cache: Optional[np.ndarray]
    k_new: Optional[np.ndarray]
    v_new: Optional[np.ndarray]
    slot_mapping: np.ndarray
    num_kv_heads: int = NUM_KV_HEADS
    num_q_heads: int = NUM_Q_HEADS
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    scale: float = SCALE
    shared_prefix_blocks: int = 0
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def unique_blocks(self) -> int:
        """Distinct physical blocks referenced by the valid part of the tables."""
        seen = set()
        for r in range(self.num_seqs):
            n = -(-int(self.context_lens[r]) // self.block_size)
            seen.update(int(b) for b in self.block_tables[r, :n])
        return len(seen)

    def unique_tokens(self) -> int:
        """Distinct physical token slots read by attention (shared prefix once)."""
        # a physical block may be read to different depths by different rows;
        # count each block at its deepest use
        deepest = {}
        for r in range(self.num_seqs):
            ctx = int(self.context_lens[r])
            for j in range(-(-ctx // self.block_size)):
                blk = int(self.block_tables[r, j])
                used = min(self.block_size, ctx - j * self.block_size)
                deepest[blk] = max(deepest.get(blk, 0), used)
        return int(sum(deepest.values()))


def _layout(
    rng: np.random.Generator,
    ctx: np.ndarray,
    num_blocks: int,
    shared_prefix_blocks: int = 0,
    sharers: Optional[np.ndarray] = None,
    max_blocks: Optional[int] = None,
):
    """Scatter every request's blocks through a pool by a seeded permutation.

    Requests flagged in `sharers` map logical blocks 0..shared_prefix_blocks-1
    to one common set of physical blocks.  Unused table entries are filled
    with block ids that are valid but unrelated, so reading past the context
    would be noticed as a wrong result, never as a fault.
    """
    b = ctx.shape[0]
    need = [-(-int(c) // BLOCK_SIZE) for c in ctx]
    if max_blocks is None:
        max_blocks = max(max(need), 1)
    perm = rng.permutation(num_blocks).astype(np.int32)
    cursor = 0
    shared = perm[cursor:cursor + shared_prefix_blocks]
    cursor += shared_prefix_blocks
    tables = np.zeros((b, max_blocks), dtype=np.int32)
    for r in range(b):
        n = need[r]
        start = 0
        if sharers is not None and sharers[r] and shared_prefix_blocks:
            assert n >= shared_prefix_blocks
            tables[r, :shared_prefix_blocks] = shared
            start = shared_prefix_blocks
        priv = n - start
        if cursor + priv > num_blocks:
            raise ValueError(f"pool of {num_blocks} blocks too small")
        tables[r, start:n] = perm[cursor:cursor + priv]
        cursor += priv
        if n < max_blocks:
            tables[r, n:] = rng.integers(0, num_blocks, size=max_blocks - n, dtype=np.int32)
    return tables, cursor


def _new_token_slots(tables: np.ndarray, ctx: np.ndarray, q_len: int) -> np.ndarray:
    """Slots of the q_len tokens each request stores this step (positions
    ctx-q_len .. ctx-1), as a caller's allocator would hand them out."""
    b = ctx.shape[0]
    slots = np.full((b, q_len), -1, dtype=np.int64)
    for r in range(b):
        for i in range(q_len):
            pos = int(ctx[r]) - q_len + i
            if pos >= 0:
                slots[r, i] = int(tables[r, pos // BLOCK_SIZE]) * BLOCK_SIZE + pos % BLOCK_SIZE
    return slots.reshape(-1)


def build(
    name: str,
    ctx,
    num_blocks: int,
    q_len: int = 1,
    seed: int = 0,
    shared_prefix_blocks: int = 0,
    sharers=None,
    fill_cache: bool = True,
    num_kv_heads: int = NUM_KV_HEADS,
    max_blocks: Optional[int] = None,
    rng: Optional[np.random.Generator] = None,
) -> Workload:
    """Lay out a batch with the given context lengths and draw its values."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(ctx, dtype=np.int32)
    sh = None if sharers is None else np.asarray(sharers, dtype=bool)
    tables, _ = _layout(rng, ctx, num_blocks, shared_prefix_blocks, sh, max_blocks)
    b = ctx.shape[0]
    hq = 4 * num_kv_heads
    q = randn_bf16(rng, (b, q_len, hq, HEAD_DIM))
    t = b * q_len
    k_new = randn_bf16(rng, (t, num_kv_heads, HEAD_DIM))
    v_new = randn_bf16(rng, (t, num_kv_heads, HEAD_DIM))
    slots = _new_token_slots(tables, ctx, q_len)
    kc = vc = None
    if fill_cache:
        shape = (num_blocks, num_kv_heads, BLOCK_SIZE, HEAD_DIM)
        kc = randn_bf16(rng, shape)
        vc = randn_bf16(rng, shape)
    return Workload(
        name=name, num_blocks=num_blocks, block_tables=tables, context_lens=ctx,
        q_len=q_len, q=q, k_cache=kc, v_cache=vc, k_new=k_new, v_new=v_new,
        slot_mapping=slots, num_kv_heads=num_kv_heads, num_q_heads=hq,
        shared_prefix_blocks=shared_prefix_blocks, seed=seed,
    )


def prefix_groups(w: Workload, max_members: int = 16):
    """Cascade description of a workload's shared prefix, as the caller that
    built the block tables would state it: requests whose tables start with
    the same `shared_prefix_blocks` physical blocks, in groups of at most
    `max_members`.  Returns (group_seqs int32 [G][16] with -1 padding,
    group_blocks int32 [G], seq_prefix_blocks int32 [B])."""
    p = w.shared_prefix_blocks
    seq_pre = np.zeros(w.num_seqs, np.int32)
    if p == 0:
        return np.zeros((0, 16), np.int32), np.zeros(0, np.int32), seq_pre
    head = w.block_tables[:, :p]
    sharers = [r for r in range(w.num_seqs) if -(-int(w.context_lens[r]) // BLOCK_SIZE) >= p]
    # requests share the prefix when their first p table entries are identical
    by_prefix = {}
    for r in sharers:
        by_prefix.setdefault(head[r].tobytes(), []).append(r)
    groups = []
    for members in by_prefix.values():
        if len(members) < 2:
            continue
        for i in range(0, len(members), max_members):
            groups.append(members[i:i + max_members])
    gs = np.full((len(groups), 16), -1, np.int32)
    for gi, members in enumerate(groups):
        gs[gi, :len(members)] = members
        seq_pre[members] = p
    return gs, np.full(len(groups), p, np.int32), seq_pre


def max_suffix_blocks(w: Workload, seq_prefix_blocks: np.ndarray) -> int:
    """Longest run of blocks any request has after its shared prefix."""
    need = np.array([-(-int(c) // BLOCK_SIZE) for c in w.context_lens])
    return int(max(1, (need - seq_prefix_blocks).max()))


# ---------------------------------------------------------------------------
# The five workloads.  Each returns one layer's inputs; multi-layer runs draw
# one Workload per layer (or fill per-layer pools on the device) with the same
# block tables.
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, fill_cache: bool = True) -> Workload:
    """4 requests, contexts {17, 64, 100, 256}, 128-block pool, q_len 1."""
    return build("tiny", [17, 64, 100, 256], 128, seed=seed, fill_cache=fill_cache)


def short_chat_ctx(rng: np.random.Generator, num_seqs: int = 37) -> np.ndarray:
    return 2048 + rng.integers(0, 256, size=num_seqs)


def short_chat(seed: int = 0, fill_cache: bool = True, num_seqs: int = 37,
               num_blocks: int = POOL_BLOCKS_12GIB) -> Workload:
    """37 requests of 2048 + U{0..255} tokens in a ~12 GiB (36-layer) pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = short_chat_ctx(rng, num_seqs)
    return build("short", ctx, num_blocks, seed=seed, fill_cache=fill_cache, rng=rng)


def long_shared(seed: int = 0, fill_cache: bool = True, num_seqs: int = 16,
                num_blocks: int = POOL_BLOCKS_12GIB) -> Workload:
    """16 requests of 8192 + U{0..255} tokens sharing a 6144-token prefix."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = 8192 + rng.integers(0, 256, size=num_seqs)
    return build("long_shared", ctx, num_blocks, seed=seed, shared_prefix_blocks=6144 // BLOCK_SIZE,
                 sharers=np.ones(num_seqs, bool), fill_cache=fill_cache, rng=rng)


def mixed(seed: int = 0, fill_cache: bool = True, num_blocks: Optional[int] = None) -> Workload:
    """48 short + 16 long (shared 6144-token prefix) in shuffled order, then
    8 requests of 1..15 tokens (a partial first block)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    is_long = np.array([False] * 48 + [True] * 16)
    rng.shuffle(is_long)
    ctx_main = np.where(is_long, 8192, 2048) + rng.integers(0, 256, size=64)
    ctx = np.concatenate([ctx_main, rng.integers(1, 16, size=8)])
    sharers = np.concatenate([is_long, np.zeros(8, bool)])
    if num_blocks is None:
        need = 384 + sum(-(-int(c) // BLOCK_SIZE) - (384 if s else 0) for c, s in zip(ctx, sharers))
        num_blocks = int(need * 5 // 4)
    return build("mixed", ctx, num_blocks, seed=seed, shared_prefix_blocks=384, sharers=sharers,
                 fill_cache=fill_cache, rng=rng)


def chunk_history(rng: np.random.Generator, num_seqs: int, lo: int = 1024, hi: int = 32768,
                  aligned: bool = True) -> np.ndarray:
    """Cached history h ~ log-uniform [lo, hi], optionally a multiple of 16."""
    h = np.exp(rng.uniform(math.log(lo), math.log(hi), size=num_seqs)).astype(np.int64)
    if aligned:
        h = (h // BLOCK_SIZE) * BLOCK_SIZE
    return h


def chunk(seed: int = 0, fill_cache: bool = True, num_seqs: int = 128, q_len: int = 16,
          lo: int = 1024, hi: int = 32768, aligned: bool = True,
          num_blocks: Optional[int] = None) -> Workload:
    """q_len-token causal chunks after h ~ logU[lo, hi] cached tokens."""
    rng = np.random.Generator(np.random.PCG64(seed))
    h = chunk_history(rng, num_seqs, lo, hi, aligned)
    ctx = h + q_len
    if num_blocks is None:
        num_blocks = int(sum(-(-int(c) // BLOCK_SIZE) for c in ctx)) + 8
    return build("chunk", ctx, num_blocks, q_len=q_len, seed=seed, fill_cache=fill_cache, rng=rng)


def sweep_point(num_seqs: int, ctx: int, seed: int = 0, fill_cache: bool = True) -> Workload:
    """q_len 1, every request at the same context length."""
    nb = num_seqs * (-(-ctx // BLOCK_SIZE)) + 8
    return build(f"sweep_b{num_seqs}_c{ctx}", [ctx] * num_seqs, nb, seed=seed, fill_cache=fill_cache)


SWEEP_BATCHES = [1 << i for i in range(10)]           # 1 .. 512
SWEEP_CONTEXTS = [128 << i for i in range(10)]        # 128 .. 65536


def fill_pool_device(cache, seed: int, chunk_blocks: int = 8192) -> None:
    """Fill a device pool tensor [num_blocks][Hkv][16][D] (BF16) with seeded
    N(0,1) values drawn by torch's device generator, chunk by chunk (for pools
    too large to draw on the host).  Same recipe as randn_bf16: float32 draws
    rounded to BF16 (torch's conversion rounds to nearest even)."""
    import torch

    gen = torch.Generator(device=cache.device)
    gen.manual_seed(int(seed))
    flat = cache.view(cache.shape[0], -1)
    tmp = None
    for b0 in range(0, cache.shape[0], chunk_blocks):
        b1 = min(cache.shape[0], b0 + chunk_blocks)
        if tmp is None or tmp.shape[0] != b1 - b0:
            tmp = torch.empty((b1 - b0, flat.shape[1]), dtype=torch.float32, device=cache.device)
        tmp.normal_(generator=gen)
        flat[b0:b1].copy_(tmp.to(torch.bfloat16).view(flat.dtype))
