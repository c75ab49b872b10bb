"""Cascade decode (shared prefixes contracted once per group on tensor
cores) through the C ABI against the FP64 oracle: the result must equal
plain attention over each request's whole context (web textbook page
"Chapter 8: Inference Optimization", §8.3.1 Fig. 8-13, §8.3.2)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, dev, to_device

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_decode_attention_gb300 as pkv
else:
    pkv = None

NAN_BF16 = np.uint16(0x7FC0)


def run_cascade(w, gs, gb, sp, pbps=0, sbps=0, append=True, d=None):
    if d is None:
        d = to_device(w)
    if append:
        pkv.kv_append(d["k_cache"], d["v_cache"], d["slot_mapping"], d["k_new"], d["v_new"])
    maxp = int(gb.max()) if gb.size else 0
    maxs = W.max_suffix_blocks(w, sp)
    p0, s0 = pkv.cascade_plan(w.num_seqs, w.num_kv_heads, gs.shape[0], maxp, maxs)
    pbps, sbps = pbps or p0, sbps or s0
    ws = torch.empty(max(1, pkv.cascade_workspace_size(w.num_seqs, w.num_q_heads, maxp, maxs, pbps, sbps)),
                     dtype=torch.uint8, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    gs_d = dev(gs) if gs.size else torch.zeros((0, 16), dtype=torch.int32, device="cuda")
    gb_d = dev(gb) if gb.size else torch.zeros(0, dtype=torch.int32, device="cuda")
    pkv.paged_attention_cascade(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                w.scale, gs_d, gb_d, dev(sp), maxp, maxs, ws, pbps, sbps)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == 0
    return out


def _shared(ctx, prefix_blocks, sharers, num_blocks, seed):
    return W.build("casc", ctx, num_blocks, seed=seed, shared_prefix_blocks=prefix_blocks, sharers=sharers)


@pytest.mark.parametrize("pbps,sbps", [(0, 0), (4, 3), (16, 1000), (100, 5)])
def test_cascade_small_groups(pbps, sbps):
    # 5 sharers of an 8-block prefix, 3 requests outside the group
    ctx = [130, 200, 129, 140, 300, 50, 77, 16]
    sharers = [True, True, True, True, True, False, False, False]
    w = _shared(ctx, 8, sharers, 120, seed=50)
    gs, gb, sp = W.prefix_groups(w)
    assert gs.shape[0] == 1 and (sp[:5] == 8).all() and (sp[5:] == 0).all()
    out = run_cascade(w, gs, gb, sp, pbps, sbps)
    assert_close(bf16_to_f64(out), oracle.run_workload(w), what=f"cascade pbps={pbps} sbps={sbps}")


def test_cascade_more_than_16_sharers_and_nan_slots():
    # 21 sharers -> two groups; NaN in every slot no context covers
    ctx = [100 + 7 * i for i in range(21)] + [33]
    sharers = [True] * 21 + [False]
    w = _shared(ctx, 4, sharers, 200, seed=51)
    gs, gb, sp = W.prefix_groups(w)
    assert gs.shape[0] == 2 and (gs[1, 5:] == -1).all()
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    used = np.zeros((w.num_blocks, 16), bool)
    for r, c in enumerate(ctx):
        for t in range(c):
            used[w.block_tables[r, t // 16], t % 16] = True
    kc.transpose(0, 2, 1, 3)[~used] = NAN_BF16
    vc.transpose(0, 2, 1, 3)[~used] = NAN_BF16
    w2 = W.Workload(**{**w.__dict__, "k_cache": kc, "v_cache": vc})
    out = run_cascade(w2, gs, gb, sp, append=False)
    assert_close(bf16_to_f64(out), oracle.run_workload(w2, append=False), what="cascade 21 sharers")


def test_cascade_member_shorter_than_prefix_and_no_groups():
    # a group member whose context ends inside the declared prefix still gets
    # the exact result; a call with no groups is plain decode
    ctx = [160, 150, 170]
    w = _shared(ctx, 10, [True, True, True], 60, seed=52)
    gs, gb, sp = W.prefix_groups(w)
    w.context_lens[1] = 70  # now ends inside the 10-block prefix
    out = run_cascade(w, gs, gb, sp, append=False)
    assert_close(bf16_to_f64(out), oracle.run_workload(w, append=False), what="short member")
    out = run_cascade(w, np.zeros((0, 16), np.int32), np.zeros(0, np.int32), np.zeros(3, np.int32), append=False)
    assert_close(bf16_to_f64(out), oracle.run_workload(w, append=False), what="no groups")


@pytest.mark.parametrize("name", ["long_shared", "mixed"])
def test_cascade_full_size_workloads(name):
    w = {"long_shared": W.long_shared, "mixed": W.mixed}[name](seed=0)
    gs, gb, sp = W.prefix_groups(w)
    out = run_cascade(w, gs, gb, sp)
    assert_close(bf16_to_f64(out), oracle.run_workload(w), what=f"cascade {name}")


def large_cascade_batch(seed, prefix_blocks=12):
    """A batch of 24+ requests: 21 sharers of a prefix (two groups), the rest
    outside every group, one padding row (context 0) and one member whose
    context ends inside the prefix."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = max(24, -(-sms // 16) + 6)
    rng = np.random.default_rng(seed)
    ctx = rng.integers(prefix_blocks * 16 + 1, prefix_blocks * 16 + 600, size=n)
    ctx[n - 1] = 0
    ctx[n - 2] = 37
    sharers = [i < 21 for i in range(n)]
    need = prefix_blocks + int(sum(-(-int(c) // 16) for c in ctx))
    w = _shared(ctx, prefix_blocks, sharers, need + 32, seed=seed)
    gs, gb, sp = W.prefix_groups(w)
    assert gs.shape[0] == 2
    w.context_lens[3] = prefix_blocks * 16 - 40  # a member ending inside its prefix
    return w, gs, gb, sp


def nan_unused(w):
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    used = np.zeros((w.num_blocks, 16), bool)
    for r, c in enumerate(w.context_lens):
        for t in range(int(c)):
            used[w.block_tables[r, t // 16], t % 16] = True
    kc.transpose(0, 2, 1, 3)[~used] = NAN_BF16
    vc.transpose(0, 2, 1, 3)[~used] = NAN_BF16
    return W.Workload(**{**w.__dict__, "k_cache": kc, "v_cache": vc})


@pytest.mark.parametrize("pbps,sbps", [(0, 0), (4, 0), (0, 8), (8, 16), (12, 1000), (4, 3)])
def test_cascade_large_batch_with_nan_in_unused_slots(pbps, sbps):
    # suffix splits merged in a cluster (prefix folded in), or more than 8
    # splits through workspace slots and the combine pass
    w, gs, gb, sp = large_cascade_batch(seed=53)
    w2 = nan_unused(w)
    out = bf16_to_f64(run_cascade(w2, gs, gb, sp, pbps, sbps, append=False))
    assert not out[w.context_lens == 0].any()
    assert_close(out, oracle.run_workload(w2, append=False), what=f"large cascade pbps={pbps} sbps={sbps}")


def test_cascade_large_batch_append_and_placement_invariance():
    w, gs, gb, sp = large_cascade_batch(seed=54, prefix_blocks=20)
    a = run_cascade(w, gs, gb, sp)
    assert_close(bf16_to_f64(a), oracle.run_workload(w), what="large cascade append+attention")
    perm = np.random.default_rng(8).permutation(w.num_blocks)
    inv = np.argsort(perm)
    w2 = W.Workload(**{**w.__dict__, "k_cache": np.ascontiguousarray(w.k_cache[perm]),
                       "v_cache": np.ascontiguousarray(w.v_cache[perm]),
                       "block_tables": inv[w.block_tables].astype(np.int32),
                       "slot_mapping": np.where(w.slot_mapping >= 0,
                                                inv[w.slot_mapping // 16] * 16 + w.slot_mapping % 16, -1)})
    assert torch.equal(a, run_cascade(w2, gs, gb, sp))


def test_cascade_peaky_logits():
    w, gs, gb, sp = large_cascade_batch(seed=55)
    w.q = W.bf16_bits((w.q.astype(np.uint32) << 16).view(np.float32) * 8.0)
    for pbps, sbps in ((0, 0), (8, 16)):
        assert_close(bf16_to_f64(run_cascade(w, gs, gb, sp, pbps, sbps)), oracle.run_workload(w),
                     what=f"cascade peaky pbps={pbps} sbps={sbps}")
