"""Pins of the oracle's sizing and pair-count arithmetic to values printed on
the web textbook page "Chapter 8: Inference Optimization" (fixtures in
tests/golden/ch8_printed_values.json, each with its section)."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import sizes

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ch8_printed_values.json")))


def test_kv_bytes_per_token():
    g = GOLD["kv_bytes_per_token"]
    assert sizes.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], g["elem_bytes"]) == g["value"]
    assert g["value"] == 144 * 1024


def test_prefill_kv_mib():
    g = GOLD["prefill_kv_mib"]
    k = GOLD["kv_bytes_per_token"]["value"]
    assert sizes.kv_mib(g["short_prompt"], k) == g["short"]
    assert sizes.kv_mib(g["long_prompt"], k) == g["long"]


def test_tokens_and_slots():
    g = GOLD["tokens_stored"]
    assert sizes.tokens_stored(2048, g["outputs"]) == g["short"]
    assert sizes.tokens_stored(8192, g["outputs"]) == g["long"]
    assert sizes.slots_allocated(g["short"], g["block_size"]) == g["short_slots"]
    assert sizes.slots_allocated(g["long"], g["block_size"]) == g["long_slots"]
    assert sizes.blocks_needed(g["short"], 16) == 144
    assert sizes.blocks_needed(g["long"], 16) == 528


def test_capacity_table():
    g = GOLD["capacity_table"]
    k = GOLD["kv_bytes_per_token"]["value"]
    short_mib = sizes.kv_mib(sizes.slots_allocated(2303, 16), k)
    long_mib = sizes.kv_mib(sizes.slots_allocated(8447, 16), k)
    assert short_mib == g["short_mib"] and long_mib == g["long_mib"]
    assert sizes.max_requests(g["pool_mib"], short_mib) == g["short_requests"]
    assert sizes.max_requests(g["pool_mib"], long_mib) == g["long_requests"]
    n = GOLD["no_output_reservation"]
    assert sizes.max_requests(g["pool_mib"], sizes.kv_mib(2048, k)) == n["requests"]
    assert n["requests"] * short_mib == n["mib_after_outputs"]


def test_shared_prefix_capacity():
    g = GOLD["shared_prefix"]
    k = GOLD["kv_bytes_per_token"]["value"]
    assert sizes.kv_mib(g["prefix_tokens"], k) == g["prefix_mib"]
    assert sizes.tokens_stored(8192 - 6144, 256) == g["private_tokens"]
    assert sizes.kv_mib(sizes.slots_allocated(g["private_tokens"], 16), k) == g["private_mib"]
    assert sizes.shared_batch_mib(g["prefix_tokens"], g["private_tokens"], g["batch"], 16, k) == g["total_mib"]
    assert g["batch"] * GOLD["capacity_table"]["long_mib"] == g["unshared_total_mib"]
    assert sizes.shared_capacity(12288, g["prefix_tokens"], g["private_tokens"], 16, k) == g["capacity"]


def test_paging_example():
    g = GOLD["paging_example"]
    lengths, p = g["lengths"], g["p"]
    assert len(lengths) * g["max_len"] == g["reserved"]
    assert sizes.paged_slots(lengths, p) == g["paged"]
    assert sum(lengths) == g["used"]
    assert g["reserved"] - g["used"] == g["unused_reserved"]
    assert sum(sizes.tail_waste(n, p) for n in lengths) == g["unused_paged"]
    assert sizes.paged_slots(lengths, p, g["shared_full_blocks"], sharers=2) == g["paged_shared"]
    # waste never reaches a whole block
    for n in range(1, 200):
        for pp in (1, 2, 4, 8, 16):
            assert 0 <= sizes.tail_waste(n, pp) <= pp - 1


def test_block_size_exercise_derived():
    # Exercise 8-3 asks for p = 2, 4, 8; the page prints p = 4 (above).  The
    # p = 2 and p = 8 values are worked by hand: table entries = sum ceil(L/p),
    # unused slots = sum tail waste.
    lengths = [9, 13, 5, 15]
    for p, entries, unused in ((2, 23, 4), (4, 13, 10), (8, 7, 14)):
        assert sum(sizes.blocks_needed(n, p) for n in lengths) == entries
        assert sum(sizes.tail_waste(n, p) for n in lengths) == unused


def test_branch_sharing():
    g = GOLD["branches"]
    phys, refs = sizes.branch_blocks(g["prefix_blocks"], g["private_blocks"], g["branches"])
    assert (phys, refs) == (g["physical"], g["references"])
    assert round(1 - phys / refs, 2) == 0.69


def test_read_bytes_table():
    g = GOLD["read_bytes"]
    k = g["kib_per_token"] * 1024
    for b, gb in zip(g["batches"], g["gb"]):
        assert round(sizes.step_read_bytes(g["weight_bytes"], b, g["context"], k) / 1e9, 2) == gb
    for ctx, b in g["kv_dominance_batch"].items():
        assert sizes.kv_dominance_batch(g["weight_bytes"], int(ctx), k) == b


@pytest.mark.parametrize("case", GOLD["chunk_pairs"], ids=lambda c: f"c{c['c']}_h{c['h']}")
def test_chunk_pair_count_from_oracle_mask(case):
    # The oracle's causal rule, counted over a chunk of c new tokens after h
    # cached ones, must admit exactly the printed number of (query, key) pairs.
    c, h = case["c"], case["h"]
    assert oracle.visible_pairs([h + c], c) == case["pairs"]


def test_pair_count_closed_form_sweep():
    # the count equals c*h + c(c+1)/2 for any chunk, and c*h... summed over a batch
    rng = np.random.default_rng(0)
    for _ in range(20):
        c = int(rng.integers(1, 40))
        h = int(rng.integers(0, 300))
        assert oracle.visible_pairs([h + c], c) == c * h + c * (c + 1) // 2
    assert oracle.visible_pairs([0, 5], 1) == 5
