"""Dense brute force for tiny inputs -- TEST INFRASTRUCTURE.

An independent restatement of the same definition for cross-checking the C
oracle: it rebuilds each request's logical K/V sequence token by token from
the block table (web textbook page "Chapter 8: Inference Optimization",
§8.3.1, Fig. 8-10: logical block j of a request lives in the physical block
its table names), then evaluates causal softmax attention with NumPy/SciPy on
the dense arrays.  Pure-Python loops: only for B <= a few, ctx <= a few
hundred.
"""
from __future__ import annotations

import numpy as np
from scipy.special import softmax


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gather_dense(cache: np.ndarray, table_row: np.ndarray, ctx: int) -> np.ndarray:
    """[Hkv][ctx][D] float64: token t of the request from block table_row[t // p], offset t % p."""
    nb, hkv, p, d = cache.shape
    dense = np.zeros((hkv, ctx, d), dtype=np.float64)
    for t in range(ctx):
        dense[:, t, :] = bf16_to_f64(cache[int(table_row[t // p]), :, t % p, :])
    return dense


def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """q [q_len][Hq][D], k/v [Hkv][ctx][D] float64; query i sees keys 0..ctx-q_len+i."""
    q_len, hq, d = q.shape
    hkv, ctx, _ = k.shape
    group = hq // hkv
    out = np.zeros((q_len, hq, d), dtype=np.float64)
    for i in range(q_len):
        last = ctx - q_len + i  # inclusive
        if last < 0:
            continue
        for h in range(hq):
            kk = k[h // group, : last + 1]
            vv = v[h // group, : last + 1]
            w = softmax(scale * (kk @ q[i, h]))
            out[i, h] = w @ vv
    return out


def paged_attention(q_bits, k_cache, v_cache, block_tables, context_lens, q_len, scale):
    b = q_bits.shape[0]
    out = np.zeros(q_bits.shape, dtype=np.float64)
    for r in range(b):
        ctx = int(context_lens[r])
        if ctx == 0:
            continue
        k = gather_dense(k_cache, block_tables[r], ctx)
        v = gather_dense(v_cache, block_tables[r], ctx)
        out[r] = dense_attention(bf16_to_f64(q_bits[r]), k, v, scale)
    return out
