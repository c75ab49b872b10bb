"""Sizing arithmetic of paged KV storage -- TEST INFRASTRUCTURE.

Plain statements of the sizing rules on the web textbook page "Chapter 8:
Inference Optimization" (clxhxhhr.top/posts/4341); the tests pin each one to
the values the page prints.
"""
from __future__ import annotations

MIB = 1 << 20


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """§8.1.2: K and V, in every layer, for every KV head and dimension."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def tokens_stored(prompt: int, outputs: int) -> int:
    """§8.1.2 note: the prompt plus every output token but the last is fed
    back (and stored); the last output token is never written."""
    return prompt + outputs - 1


def blocks_needed(length: int, p: int) -> int:
    """§8.3.1: a sequence of L tokens in blocks of p tokens needs ceil(L/p) blocks."""
    return -(-length // p)


def slots_allocated(length: int, p: int) -> int:
    return p * blocks_needed(length, p)


def tail_waste(length: int, p: int) -> int:
    """§8.3.1: only the last block has unused slots: p*ceil(L/p) - L <= p - 1."""
    return slots_allocated(length, p) - length


def kv_mib(slots: int, bytes_per_token: int) -> float:
    return slots * bytes_per_token / MIB


def max_requests(pool_mib: float, per_request_mib: float) -> int:
    """§8.1.2 capacity table: floor(pool / per-request allocation)."""
    return int(pool_mib // per_request_mib)


def shared_batch_mib(prefix_tokens: int, private_tokens: int, b: int, p: int, bytes_per_token: int) -> float:
    """§8.3.2: one copy of the common prefix plus each request's private blocks."""
    return kv_mib(slots_allocated(prefix_tokens, p) + b * slots_allocated(private_tokens, p), bytes_per_token)


def shared_capacity(pool_mib: float, prefix_tokens: int, private_tokens: int, p: int, bytes_per_token: int) -> int:
    """Largest b with shared_batch_mib(b) <= pool."""
    b = 0
    while shared_batch_mib(prefix_tokens, private_tokens, b + 1, p, bytes_per_token) <= pool_mib:
        b += 1
    return b


def paged_slots(lengths, p: int, shared_full_blocks: int = 0, sharers: int = 0) -> int:
    """§8.3.1 worked example: slots allocated when each sequence gets whole
    blocks, and `sharers` sequences reference `shared_full_blocks` common
    full blocks stored once."""
    total = sum(slots_allocated(n, p) for n in lengths)
    if sharers > 1:
        total -= (sharers - 1) * shared_full_blocks * p
    return total


def branch_blocks(prefix_blocks: int, private_blocks: int, branches: int):
    """§8.3.2: (physical blocks stored, block-table references)."""
    return prefix_blocks + branches * private_blocks, branches * (prefix_blocks + private_blocks)


def step_read_bytes(weight_bytes: int, b: int, context: int, bytes_per_token: int) -> int:
    """§8.2.1: bytes read by one decode step: shared weights once plus every
    request's KV, D_w + b * L * k."""
    return weight_bytes + b * context * bytes_per_token


def kv_dominance_batch(weight_bytes: int, context: int, bytes_per_token: int) -> int:
    """§8.2.1: smallest b whose KV reads reach the shared weight reads, ceil(D_w / (L k))."""
    return -(-weight_bytes // (context * bytes_per_token))


def group_bytes(values: int, code_bits: int, scale_bytes: int = 2) -> float:
    """§8.4.2, Fig. 8-23: a group of `values` numbers stores its codes at
    `code_bits` each plus one scale of `scale_bytes`."""
    return values * code_bits / 8 + scale_bytes


def quantized_mib(bf16_mib: float, code_bits: int, group: int = 32) -> float:
    """§8.4.2: the same values regrouped -- BF16 spends 2*group bytes per
    group, the quantized format group_bytes(group, code_bits)."""
    return bf16_mib * group_bytes(group, code_bits) / (2 * group)


def bits_per_value(code_bits: int, group: int = 32, scale_bytes: int = 2) -> float:
    """§8.4.2: average storage per value, the scale included."""
    return group_bytes(group, code_bits, scale_bytes) * 8 / group


def saved_time_s(delta_bytes: float, bandwidth_bytes_per_s: float, convert_s: float) -> float:
    """§8.4.2: net time saved by reading fewer bytes, dT = dD / beta - T_c."""
    return delta_bytes / bandwidth_bytes_per_s - convert_s
