"""Pins of the FP64 oracle's attention and append to things other than itself:
an independent dense restatement (NumPy/SciPy), PyTorch's own
scaled_dot_product_attention in float64, closed forms, and the invariances
that paging and prefix sharing must leave intact (web textbook page
"Chapter 8: Inference Optimization", §8.3.1 Fig. 8-10, §8.3.2 Fig. 8-13,
§8.2.3 Fig. 8-8/8-9)."""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
import workloads as W
from oracle import brute

NAN_BF16 = np.uint16(0x7FC0)


def _small(seed, ctx, q_len=1, num_blocks=None, kv_heads=2):
    nb = num_blocks or sum(-(-c // 16) for c in ctx) + 5
    return W.build("t", ctx, nb, q_len=q_len, seed=seed, num_kv_heads=kv_heads)


@pytest.mark.parametrize("q_len", [1, 3, 16])
@pytest.mark.parametrize("seed", [0, 1])
def test_oracle_matches_dense_brute_force(seed, q_len):
    w = _small(seed, [q_len, 17, 40 + q_len], q_len=q_len)
    got, lse = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                      q_len, w.scale, with_lse=True)
    ref = brute.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, q_len, w.scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # lse of the last request, first head, last query: all keys visible
    r, h = 2, 0
    k = brute.gather_dense(w.k_cache, w.block_tables[r], int(w.context_lens[r]))
    s = w.scale * (k[h // 4] @ brute.bf16_to_f64(w.q[r, q_len - 1, h]))
    assert abs(lse[r, q_len - 1, h] - logsumexp(s)) < 1e-12


def test_oracle_matches_torch_sdpa_float64():
    # dense causal GQA attention is a library routine: torch's SDPA in float64
    q_len = 5
    w = _small(3, [33, 64, 21], q_len=q_len)
    got = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, q_len, w.scale)
    for r, ctx in enumerate(w.context_lens):
        ctx = int(ctx)
        k = torch.from_numpy(brute.gather_dense(w.k_cache, w.block_tables[r], ctx))
        v = torch.from_numpy(brute.gather_dense(w.v_cache, w.block_tables[r], ctx))
        q = torch.from_numpy(brute.bf16_to_f64(w.q[r])).permute(1, 0, 2)  # [Hq][q_len][D]
        k = k.repeat_interleave(4, dim=0)
        v = v.repeat_interleave(4, dim=0)
        i = torch.arange(q_len)[:, None]
        t = torch.arange(ctx)[None, :]
        mask = t <= (ctx - q_len + i)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=w.scale)
        np.testing.assert_allclose(got[r], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_context_one_returns_v0():
    w = _small(4, [1, 1], kv_heads=2)
    out = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    for r in range(2):
        blk = w.block_tables[r, 0]
        for h in range(8):
            np.testing.assert_array_equal(out[r, 0, h], brute.bf16_to_f64(w.v_cache[blk, h // 4, 0]))


def test_identical_v_rows_give_that_row():
    w = _small(5, [50, 97])
    row = W.randn_bf16(np.random.default_rng(9), (w.num_kv_heads, 128))
    w.v_cache[:] = row[None, :, None, :]
    out = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    for h in range(w.num_q_heads):
        np.testing.assert_allclose(out[:, 0, h], np.broadcast_to(brute.bf16_to_f64(row[h // 4]), (2, 128)),
                                   rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    q_len = 4
    w = _small(6, [30, 45], q_len=q_len)
    w.q[:] = 0
    out = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, q_len, w.scale)
    for r in range(2):
        ctx = int(w.context_lens[r])
        v = brute.gather_dense(w.v_cache, w.block_tables[r], ctx)
        for i in range(q_len):
            last = ctx - q_len + i
            for h in range(w.num_q_heads):
                np.testing.assert_allclose(out[r, i, h], v[h // 4, :last + 1].mean(axis=0), rtol=0, atol=1e-13)


def test_chunk_row_equals_decode_at_shorter_context():
    # §8.2.3: new token i of a chunk sees exactly what a one-token decode at
    # context ctx - q_len + 1 + i would see
    q_len = 6
    w = _small(7, [70, 23], q_len=q_len)
    full = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, q_len, w.scale)
    for i in range(q_len):
        ctx_i = w.context_lens - q_len + 1 + i
        one = oracle.paged_attention(np.ascontiguousarray(w.q[:, i:i + 1]), w.k_cache, w.v_cache,
                                     w.block_tables, ctx_i, 1, w.scale)
        np.testing.assert_array_equal(full[:, i], one[:, 0])


def test_physical_placement_does_not_matter():
    # Fig. 8-10: only the table decides which physical block holds a logical
    # block; relabelling the pool (and the tables with it) changes nothing
    w = _small(8, [37, 80, 16, 5])
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    inv = np.argsort(perm)
    kc = w.k_cache[perm]            # new block j holds old block perm[j]
    vc = w.v_cache[perm]
    tables = inv[w.block_tables].astype(np.int32)
    a = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    b = oracle.paged_attention(w.q, kc, vc, tables, w.context_lens, 1, w.scale)
    np.testing.assert_array_equal(a, b)


def test_fig_8_10_hand_built_table_and_free_block_is_never_read():
    # logical blocks 0,1,2 -> physical 2,0,3; physical block 1 free and
    # holding NaN patterns, which must not reach the result
    rng = np.random.default_rng(2)
    kc = W.randn_bf16(rng, (4, 1, 16, 128))
    vc = W.randn_bf16(rng, (4, 1, 16, 128))
    kc[1] = NAN_BF16
    vc[1] = NAN_BF16
    q = W.randn_bf16(rng, (1, 1, 4, 128))
    table = np.array([[2, 0, 3]], np.int32)
    ctx = np.array([40], np.int32)
    out = oracle.paged_attention(q, kc, vc, table, ctx, 1, W.SCALE)
    assert np.isfinite(out).all()
    # dense identity: the logical sequence laid out contiguously
    kd = np.concatenate([kc[2, 0], kc[0, 0], kc[3, 0]])[:40]
    vd = np.concatenate([vc[2, 0], vc[0, 0], vc[3, 0]])[:40]
    ref = brute.dense_attention(brute.bf16_to_f64(q[0]), brute.bf16_to_f64(kd)[None],
                                brute.bf16_to_f64(vd)[None], W.SCALE)
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)


def test_shared_prefix_equals_duplicated_prefix():
    # Fig. 8-13: sharers of a stored-once prefix see the same result as if
    # each had its own copy
    ctx = [70, 90, 65]
    w = W.build("s", ctx, 40, seed=11, shared_prefix_blocks=4, sharers=[True, True, True], num_kv_heads=2)
    assert (w.block_tables[:, :4] == w.block_tables[0, :4]).all()
    shared = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    # give requests 1 and 2 private copies of the prefix blocks
    kc = np.concatenate([w.k_cache, w.k_cache[w.block_tables[0, :4]], w.k_cache[w.block_tables[0, :4]]])
    vc = np.concatenate([w.v_cache, w.v_cache[w.block_tables[0, :4]], w.v_cache[w.block_tables[0, :4]]])
    tables = w.block_tables.copy()
    tables[1, :4] = np.arange(40, 44)
    tables[2, :4] = np.arange(44, 48)
    dup = oracle.paged_attention(w.q, kc, vc, tables, w.context_lens, 1, w.scale)
    np.testing.assert_array_equal(shared, dup)


def test_padding_row_is_zero_and_lse_neg_inf():
    w = _small(12, [0, 20])
    out, lse = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1,
                                      w.scale, with_lse=True)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(out[1]).all()


def test_peaky_logits_match_brute_force():
    w = _small(13, [120, 33])
    qf = brute.bf16_to_f64(w.q) * 8.0
    w.q = W.bf16_bits(qf.astype(np.float32))
    got = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    ref = brute.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    w = _small(14, [20, 50, 33, 70])
    full = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    part = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale,
                                  seq_ids=[3, 1])
    np.testing.assert_array_equal(part, full[[3, 1]])


def test_table_entry_outside_pool_is_rejected():
    w = _small(15, [20])
    w.block_tables[0, 1] = w.num_blocks
    with pytest.raises(ValueError):
        oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)


# ----------------------------------------------------------------------------
# kv_append
# ----------------------------------------------------------------------------

def test_kv_append_round_trip_and_untouched_slots():
    w = W.tiny(seed=3)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    written = set()
    for t, slot in enumerate(w.slot_mapping):
        blk, off = divmod(int(slot), 16)
        np.testing.assert_array_equal(kc[blk, :, off], w.k_new[t])
        np.testing.assert_array_equal(vc[blk, :, off], w.v_new[t])
        written.add((blk, off))
    mask = np.ones((w.num_blocks, 16), bool)
    for blk, off in written:
        mask[blk, off] = False
    np.testing.assert_array_equal(kc.transpose(0, 2, 1, 3)[mask], w.k_cache.transpose(0, 2, 1, 3)[mask])
    np.testing.assert_array_equal(vc.transpose(0, 2, 1, 3)[mask], w.v_cache.transpose(0, 2, 1, 3)[mask])


def test_kv_append_skips_negative_and_out_of_pool_slots():
    w = W.tiny(seed=4)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    slots = w.slot_mapping.copy()
    slots[0] = -1
    slots[1] = w.num_blocks * 16
    oracle.kv_append(kc, vc, slots, w.k_new, w.v_new)
    changed = np.argwhere((kc != w.k_cache).any(axis=(1, 3)))
    got = {(int(b) * 16 + int(o)) for b, o in changed}
    assert got <= {int(s) for s in slots[2:]}
    assert int(w.slot_mapping[0]) not in got


def test_appended_token_is_the_last_visible_key():
    # the new token's slot is found through the table at position ctx - 1
    # (§8.1.1: append, then attend); its K/V are what attention reads there
    w = W.tiny(seed=5)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    for r, ctx in enumerate(w.context_lens):
        k = brute.gather_dense(kc, w.block_tables[r], int(ctx))
        np.testing.assert_array_equal(k[:, -1], brute.bf16_to_f64(w.k_new[r]))


def test_workload_shapes():
    w = W.short_chat(seed=0, fill_cache=False)
    assert w.num_seqs == 37 and w.context_lens.min() >= 2048 and w.context_lens.max() <= 2303
    assert w.max_blocks_per_seq <= 144 and w.num_blocks == W.POOL_BLOCKS_12GIB == 5461
    lw = W.long_shared(seed=0, fill_cache=False)
    assert (lw.block_tables[:, :384] == lw.block_tables[0, :384]).all()
    assert lw.max_blocks_per_seq <= 528
    m = W.mixed(seed=0, fill_cache=False)
    assert m.num_seqs == 72 and (m.context_lens[64:] < 16).all()
    c = W.chunk(seed=0, fill_cache=False, num_seqs=8)
    assert ((c.context_lens - 16) % 16 == 0).all() and c.q_len == 16


def test_combine_of_range_results_equals_whole_context():
    # attention over [0, ctx) equals the lse-weighted merge of attention over
    # block-aligned key ranges, each evaluated by the oracle as its own request
    w = _small(16, [150, 77, 16])
    full, full_lse = oracle.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1,
                                            w.scale, with_lse=True)
    hq, d = w.num_q_heads, 128
    cuts = [0, 32, 48, 112, 1000]  # token boundaries (multiples of 16); last range may be empty
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sub_ctx = np.clip(np.minimum(w.context_lens, b) - a, 0, None).astype(np.int32)
        sub_tables = np.zeros_like(w.block_tables)
        nb = w.block_tables.shape[1] - a // 16
        sub_tables[:, :max(nb, 0)] = w.block_tables[:, a // 16:]
        o, l = oracle.paged_attention(w.q, w.k_cache, w.v_cache, sub_tables, sub_ctx, 1, w.scale, with_lse=True)
        parts_o.append(o.reshape(-1, d))
        parts_l.append(l.reshape(-1))
    po = np.stack(parts_o, axis=1)
    pl = np.stack(parts_l, axis=1)
    out, lse = oracle.attn_combine(po, pl)
    np.testing.assert_allclose(out, full.reshape(-1, d), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, full_lse.reshape(-1), rtol=0, atol=1e-12)
    assert hq == 8
    # a row whose ranges are all empty merges to zeros
    z, zl = oracle.attn_combine(np.ones((1, 3, 4)), np.full((1, 3), -np.inf))
    assert (z == 0).all() and np.isneginf(zl).all()
