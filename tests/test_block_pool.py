"""The host block pool (reference counts, copy-on-write reservation) against
the worked examples of the web textbook page "Chapter 8: Inference
Optimization" (§8.3.1 paging example, §8.3.2 branch sharing, Fig. 8-14 and
Fig. 8-15), from tests/golden/ch8_printed_values.json.  Host code only."""
import json
import os

import pytest

import paged_kv_decode_attention_gb300 as pkv

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ch8_printed_values.json")))


def _used_blocks(pool, total):
    return total - pool.num_free


def test_paging_example_allocates_52_slots_and_44_with_sharing():
    g = GOLD["paging_example"]
    p = g["p"]
    pool = pkv.BlockPool(64, p)
    rows = []
    for n in g["lengths"]:
        row = []
        assert pool.reserve(row, 0, n, 16) == []
        rows.append(row)
    assert _used_blocks(pool, 64) * p == g["paged"]
    assert _used_blocks(pool, 64) * p - sum(g["lengths"]) == g["unused_paged"]
    # A and B share their first two full blocks (8 tokens): B references A's
    pool2 = pkv.BlockPool(64, p)
    a = []
    pool2.reserve(a, 0, g["lengths"][0], 16)
    b = a[:g["shared_full_blocks"]]
    pool2.share(b)
    pool2.reserve(b, g["shared_full_blocks"] * p, g["lengths"][1] - g["shared_full_blocks"] * p, 16)
    for n in g["lengths"][2:]:
        pool2.reserve([], 0, n, 16)
    assert _used_blocks(pool2, 64) * p == g["paged_shared"]
    assert pool2.refcount(a[0]) == 2 and b[:2] == a[:2]


def test_four_branches_store_131_blocks_for_416_references():
    g = GOLD["branches"]
    total = 1000
    pool = pkv.BlockPool(total, 16)
    prefix = pool.alloc(g["prefix_blocks"])
    rows = []
    for _ in range(g["branches"]):
        row = list(prefix)
        pool.share(prefix)
        pool.reserve(row, g["prefix_blocks"] * 16, g["private_blocks"] * 16, 200)
        rows.append(row)
    pool.release(prefix)  # the allocation's own reference; the branches hold theirs
    assert _used_blocks(pool, total) == g["physical"]
    refs = sum(pool.refcount(b) for b in set(x for r in rows for x in r))
    assert refs == g["references"]


def test_shared_partial_tail_is_copied_before_writing_fig_8_15():
    # blocks of 4 tokens; the common tail block already holds a, b, c
    pool = pkv.BlockPool(16, 4)
    base = []
    pool.reserve(base, 0, 7, 8)                  # one full block + a tail holding 3 tokens
    x, y = list(base), list(base)
    pool.share(base)                             # second branch references both blocks
    copies_x = pool.reserve(x, 7, 1, 8)          # branch x appends: its tail is shared -> copy
    assert copies_x == [(base[1], x[1])] and x[1] != base[1] and x[0] == base[0]
    copies_y = pool.reserve(y, 7, 1, 8)          # y now holds the only reference: write in place
    assert copies_y == [] and y[1] == base[1]
    assert x[1] != y[1]                          # different physical tail blocks
    assert pool.refcount(base[0]) == 2           # the full block stays shared
    assert pool.refcount(x[1]) == 1 and pool.refcount(y[1]) == 1


def test_release_frees_only_the_last_reference_fig_8_14():
    pool = pkv.BlockPool(8, 16)
    a = pool.alloc(2)
    pool.share(a)            # B references A's blocks
    pool.release(a)          # A finishes
    assert pool.num_free == 6 and pool.refcount(a[0]) == 1
    pool.release(a)          # B finishes
    assert pool.num_free == 8 and pool.refcount(a[0]) == 0


def test_long_requests_sharing_a_prefix_fit_the_6048_mib_layout():
    g = GOLD["shared_prefix"]
    kib = GOLD["kv_bytes_per_token"]["value"]
    pool = pkv.BlockPool(5461, 16)
    prefix = []
    pool.reserve(prefix, 0, g["prefix_tokens"], 528)
    for _ in range(g["batch"]):
        row = list(prefix)
        pool.share(prefix)
        pool.reserve(row, g["prefix_tokens"], g["private_tokens"], 528)
    used = 5461 - pool.num_free
    assert used * 16 * kib / 2**20 == g["total_mib"]


def test_errors_leave_the_pool_unchanged():
    pool = pkv.BlockPool(4, 16)
    with pytest.raises(pkv.PkvError) as e:
        pool.alloc(5)
    assert e.value.status == 6 and pool.num_free == 4
    a = pool.alloc(1)
    with pytest.raises(pkv.PkvError):
        pool.release(a + a)  # two references dropped, one held
    assert pool.refcount(a[0]) == 1
    row = []
    with pytest.raises(pkv.PkvError):
        pool.reserve(row, 0, 16 * 4, 8)   # 4 blocks needed, 3 free
    assert pool.num_free == 3 and row == []
