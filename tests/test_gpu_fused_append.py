"""pkv_paged_attention_append: the append and the attention of a decode step
in one call.  Where it fuses them into one kernel (q_len 1 on the CTA-per-row
decode kernel) and where it issues the two launches, its output and the pools
it leaves must equal pkv_kv_append followed by pkv_paged_attention bit for
bit; the result must also match the FP64 oracle; and a slot that is not the
one the block table gives the new token's position sets the device error
word."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, to_device

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_decode_attention_gb300 as pkv
else:  # collected on CPU-only machines, every test skipped
    pkv = None


@pytest.fixture(autouse=True)
def _clear_device_error():
    if pkv is not None:
        pkv.get_device_error(reset=True)
    yield
    if pkv is not None:
        assert pkv.get_device_error(reset=True) == 0


def _both(w, bps=0, d=None):
    """(fused call, separate calls) on copies of the same device state: outputs and pools."""
    if d is None:
        d = to_device(w)
    maxb = w.max_blocks_per_seq
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split(w.num_seqs, w.num_kv_heads, w.q_len, maxb)
    ws = torch.empty(max(pkv.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    res = []
    for fused in (True, False):
        kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
        out = torch.full_like(d["q"], float("nan"))
        if fused:
            pkv.paged_attention_append(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.q_len, w.scale,
                                       d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=bps,
                                       workspace=ws)
        else:
            pkv.kv_append(kc, vc, d["slot_mapping"], d["k_new"], d["v_new"])
            pkv.paged_attention(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.q_len, w.scale,
                                kv_blocks_per_split=bps, workspace=ws)
        torch.cuda.synchronize()
        res.append((out, kc, vc))
    return res


def _assert_same(res, what):
    (of, kf, vf), (os_, ks, vs) = res
    assert torch.equal(of.view(torch.int16), os_.view(torch.int16)), f"{what}: outputs differ"
    assert torch.equal(kf.view(torch.int16), ks.view(torch.int16)), f"{what}: K pools differ"
    assert torch.equal(vf.view(torch.int16), vs.view(torch.int16)), f"{what}: V pools differ"


# contexts that put the new token at a block's first slot (17, 2049), last slot (16, 32) or
# alone (1), and a padding row (0, slot -1)
RAGGED = [17, 300, 1, 16, 700, 0, 32, 2049, 129, 55]


@pytest.mark.parametrize("bps", [0, 1000, 5, 24])
def test_fused_decode_equals_append_then_attention(bps):
    """One kernel on the CTA-per-row decode: no split (1000), cluster-merged
    splits (0, 24) and workspace splits merged by the combine kernel (5)."""
    ctx = np.asarray(RAGGED)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("fused", ctx, need + 30, seed=61)
    res = _both(w, bps)
    _assert_same(res, f"fused bps={bps}")
    assert not res[0][0][ctx == 0].float().abs().sum()
    assert_close(bf16_to_f64(res[0][0]), oracle.run_workload(w), what=f"fused vs oracle bps={bps}")


@pytest.mark.parametrize("num_seqs,q_len", [(24, 1), (6, 4), (5, 16)])
def test_shapes_that_issue_two_launches(num_seqs, q_len):
    """Tensor-core decode (24 requests of ~2K tokens), a 4-position query and
    a 16-position chunk: the append, then the attention; same results."""
    rng = np.random.default_rng(num_seqs + q_len)
    ctx = rng.integers(1900 if q_len == 1 else q_len, 2300, size=num_seqs)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("two-launch", ctx, need + 30, q_len=q_len, seed=62)
    res = _both(w)
    _assert_same(res, f"two launches {num_seqs}x{q_len}")
    assert_close(bf16_to_f64(res[0][0]), oracle.run_workload(w), what=f"two launches {num_seqs}x{q_len}")


def test_unstored_token_reads_the_pool_as_it_is():
    """A request whose new token is not stored (slot -1) attends over the pool
    as it stands, as the separate calls do."""
    ctx = np.asarray(RAGGED)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("unstored", ctx, need + 30, seed=63)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[[1, 7]] = -1
    _assert_same(_both(w), "unstored token")


def test_slot_other_than_the_tables_sets_the_error_word():
    ctx = np.asarray([100, 200, 300])
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("bad-slot", ctx, need + 30, seed=64)
    used = set()
    for r, c in enumerate(ctx):
        used.update(int(b) for b in w.block_tables[r, :-(-int(c) // 16)])
    spare = next(b for b in range(w.num_blocks) if b not in used)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[1] = spare * 16 + 3  # stored there, but not at request 1's position
    d = to_device(w)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_attention_append(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], 1,
                               w.scale, d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=1000,
                               workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    # the token is stored where the slot says, as the append would
    kc = d["k_cache"].view(torch.int16).cpu().numpy()
    assert np.array_equal(kc[spare, :, 3, :], w.k_new.view(np.int16)[1])


def _cascade_both(w, pbps, sbps):
    gs, gb, sp = W.prefix_groups(w)
    maxp, maxs = int(gb.max()), W.max_suffix_blocks(w, sp)
    b, hq = w.num_seqs, w.num_q_heads
    pb, sb = pkv.cascade_plan(b, w.num_kv_heads, gs.shape[0], maxp, maxs)
    pb, sb = pbps or pb, sbps or sb
    ws = torch.empty(max(256, pkv.cascade_workspace_size(b, hq, maxp, maxs, pb, sb)), dtype=torch.uint8,
                     device="cuda")
    d = to_device(w)
    gs_d, gb_d, sp_d = (torch.from_numpy(x).cuda() for x in (gs, gb, sp))
    res = []
    for fused in (True, False):
        kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
        out = torch.full_like(d["q"], float("nan"))
        if fused:
            pkv.paged_attention_cascade_append(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                               gs_d, gb_d, sp_d, maxp, maxs, ws, d["slot_mapping"], d["k_new"],
                                               d["v_new"], pb, sb)
        else:
            pkv.kv_append(kc, vc, d["slot_mapping"], d["k_new"], d["v_new"])
            pkv.paged_attention_cascade(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale, gs_d,
                                        gb_d, sp_d, maxp, maxs, ws, pb, sb)
        torch.cuda.synchronize()
        res.append((out, kc, vc))
    return res


@pytest.mark.parametrize("pbps,sbps", [(0, 0), (4, 3), (16, 2)])
def test_fused_cascade_equals_append_then_cascade(pbps, sbps):
    """Five sharers of an 8-block prefix and three requests outside it; suffix
    splits merged in a cluster (0, 3) or through the workspace (2)."""
    ctx = [130, 200, 129, 140, 300, 50, 77, 16]
    w = W.build("casc-fused", ctx, 120, seed=65, shared_prefix_blocks=8, sharers=[True] * 5 + [False] * 3)
    res = _cascade_both(w, pbps, sbps)
    _assert_same(res, f"fused cascade pbps={pbps} sbps={sbps}")
    assert_close(bf16_to_f64(res[0][0]), oracle.run_workload(w), what=f"fused cascade pbps={pbps} sbps={sbps}")


def test_fused_cascade_token_inside_the_shared_prefix_sets_the_error_word():
    ctx = [130, 200, 129, 140, 300, 50]
    w = W.build("casc-inside", ctx, 120, seed=66, shared_prefix_blocks=8, sharers=[True] * 5 + [False])
    gs, gb, sp = W.prefix_groups(w)
    # request 0 now ends inside the 8-block prefix: its new token (position 99) would go to a shared block
    w.context_lens = w.context_lens.copy()
    w.context_lens[0] = 100
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[0] = int(w.block_tables[0, 99 // 16]) * 16 + 99 % 16
    maxp, maxs = int(gb.max()), W.max_suffix_blocks(w, sp)
    ws = torch.empty(max(256, pkv.cascade_workspace_size(w.num_seqs, w.num_q_heads, maxp, maxs,
                                                         *pkv.cascade_plan(w.num_seqs, w.num_kv_heads, gs.shape[0],
                                                                           maxp, maxs))), dtype=torch.uint8,
                     device="cuda")
    d = to_device(w)
    out = torch.empty_like(d["q"])
    pkv.paged_attention_cascade_append(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                       d["context_lens"], w.scale, *(torch.from_numpy(x).cuda() for x in (gs, gb, sp)),
                                       maxp, maxs, ws, d["slot_mapping"], d["k_new"], d["v_new"])
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT


@pytest.mark.parametrize("seed", range(12))
def test_fused_random_shapes(seed):
    """Seeded random batches (1-60 requests, 0-3000 tokens, some tokens not
    stored, any split): every dispatch path, bit-equal to the separate calls."""
    rng = np.random.default_rng(1000 + seed)
    b = int(rng.integers(1, 61))
    ctx = rng.integers(0, 3001, size=b)
    ctx[rng.random(b) < 0.1] = 0
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("fused-rand", ctx, need + 16, seed=2000 + seed)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[rng.random(b) < 0.1] = -1
    bps = int(rng.choice([0, 0, 3, 16, 40, 1000]))
    _assert_same(_both(w, bps), f"random seed={seed} b={b} bps={bps}")


def _tokens_of_pool(pool: np.ndarray) -> np.ndarray:
    nb, hkv, bs, d = pool.shape
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))


def _fp8_host_pools(k_pool: np.ndarray, v_pool: np.ndarray):
    """E4M3 pools holding BF16 host pools, stored by the oracle's append."""
    nb, hkv = k_pool.shape[:2]
    kq = np.zeros((nb, hkv, 16, 128), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_fp8(kq, vq, np.arange(nb * 16, dtype=np.int64), _tokens_of_pool(k_pool),
                         _tokens_of_pool(v_pool))
    return kq, vq


def _fp8_pools(d, w):
    """Device E4M3 pools holding the workload's BF16 cache (the oracle's rounding)."""
    kq, vq = _fp8_host_pools(w.k_cache, w.v_cache)
    return torch.from_numpy(kq).cuda(), torch.from_numpy(vq).cuda()


def _fp8_oracle(w, kq: np.ndarray, vq: np.ndarray, q=None, tables=None, ctx=None, slots=None, k_new=None,
                v_new=None):
    """The step with the oracle on copies of host E4M3 pools: the rounding
    append of the new tokens, then FP64 attention over the stored values."""
    kq, vq = kq.copy(), vq.copy()
    oracle.kv_append_fp8(kq, vq, w.slot_mapping if slots is None else slots, w.k_new if k_new is None else k_new,
                         w.v_new if v_new is None else v_new)
    out = oracle.paged_attention_f64(w.q if q is None else q, oracle.dequantize_fp8(kq), oracle.dequantize_fp8(vq),
                                     w.block_tables if tables is None else tables,
                                     w.context_lens if ctx is None else ctx, 1, w.scale)
    return out, kq, vq


def _assert_fp8_oracle(res, w, what):
    """The fused call's output and pools against the oracle's step."""
    out, kf, vf = res[0]
    ref, kq, vq = _fp8_oracle(w, *_fp8_host_pools(w.k_cache, w.v_cache))
    assert np.array_equal(kf.cpu().numpy(), kq) and np.array_equal(vf.cpu().numpy(), vq), \
        f"{what}: E4M3 pools differ from the oracle's append"
    assert_close(bf16_to_f64(out), ref, what=f"{what} vs oracle")


def _fp8_both(w, bps=0):
    d = to_device(w)
    kq, vq = _fp8_pools(d, w)
    maxb = w.max_blocks_per_seq
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split_fp8_e4m3(w.num_seqs, w.num_kv_heads, maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(w.num_seqs, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    res = []
    for fused in (True, False):
        kc, vc = kq.clone(), vq.clone()
        out = torch.full_like(d["q"], float("nan"))
        if fused:
            pkv.paged_attention_fp8_e4m3_append(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                                d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=bps,
                                                workspace=ws)
        else:
            pkv.kv_append_fp8_e4m3(kc, vc, d["slot_mapping"], d["k_new"], d["v_new"])
            pkv.paged_attention_fp8_e4m3(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                         kv_blocks_per_split=bps, workspace=ws)
        torch.cuda.synchronize()
        res.append((out, kc, vc))
    return res


def _assert_same_fp8(res, what):
    (of, kf, vf), (os_, ks, vs) = res
    assert torch.equal(of.view(torch.int16), os_.view(torch.int16)), f"{what}: outputs differ"
    assert torch.equal(kf, ks) and torch.equal(vf, vs), f"{what}: E4M3 pools differ"


# new tokens in the first and second 128-row half of a 256-token tile, at a block's first and last
# slot, alone, and a padding row
RAGGED_FP8 = [17, 300, 1, 16, 700, 0, 32, 2049, 129, 200, 4000]


@pytest.mark.parametrize("bps", [0, 8, 24, 5, 1000])
def test_fused_fp8_equals_append_then_attention(bps):
    ctx = np.asarray(RAGGED_FP8)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("fused-fp8", ctx, need + 30, seed=71)
    res = _fp8_both(w, bps)
    _assert_same_fp8(res, f"fused fp8 bps={bps}")
    assert not res[0][0][ctx == 0].float().abs().sum()
    _assert_fp8_oracle(res, w, f"fused fp8 bps={bps}")


@pytest.mark.parametrize("seed", range(6))
def test_fused_fp8_random_shapes(seed):
    rng = np.random.default_rng(3000 + seed)
    b = int(rng.integers(1, 61))
    ctx = rng.integers(0, 3001, size=b)
    ctx[rng.random(b) < 0.1] = 0
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("fused-fp8-rand", ctx, need + 16, seed=4000 + seed)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[rng.random(b) < 0.1] = -1
    bps = int(rng.choice([0, 0, 5, 16, 40, 1000]))
    res = _fp8_both(w, bps)
    _assert_same_fp8(res, f"fp8 random seed={seed} b={b} bps={bps}")
    _assert_fp8_oracle(res, w, f"fp8 random seed={seed} b={b} bps={bps}")


def test_fused_fp8_wrong_slot_sets_the_error_word():
    ctx = np.asarray([100, 200, 300])
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("bad-slot-fp8", ctx, need + 30, seed=72)
    used = set()
    for r, c in enumerate(ctx):
        used.update(int(b) for b in w.block_tables[r, :-(-int(c) // 16)])
    spare = next(b for b in range(w.num_blocks) if b not in used)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[2] = spare * 16 + 5
    d = to_device(w)
    kq, vq = _fp8_pools(d, w)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_attention_fp8_e4m3_append(out, d["q"], kq, vq, d["block_tables"], d["context_lens"], w.scale,
                                        d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=1000,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    ref_k, ref_v = kq.clone(), vq.clone()
    pkv.kv_append_fp8_e4m3(ref_k, ref_v, d["slot_mapping"], d["k_new"], d["v_new"])
    torch.cuda.synchronize()
    assert torch.equal(kq[spare], ref_k[spare]) and torch.equal(vq[spare], ref_v[spare])  # stored as the append would


def test_fused_fp8_short_chat_full_size():
    """The 2K-context batch at full size (37 requests, 5461-block pools filled
    on the device) in the launch configuration of the benchmark's step (the
    library's split choice): the fused call equals the E4M3 append followed by
    the attention, outputs and pools bit for bit."""
    w = W.short_chat(seed=21, fill_cache=False)
    nb, hkv = w.num_blocks, w.num_kv_heads
    kb = torch.empty((nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    vb = torch.empty_like(kb)
    W.fill_pool_device(kb, seed=21)
    W.fill_pool_device(vb, seed=22)
    tok = lambda p: p.permute(0, 2, 1, 3).contiguous().view(nb * 16, hkv, 128)
    kq = torch.empty((nb, hkv, 16, 128), dtype=torch.uint8, device="cuda")
    vq = torch.empty_like(kq)
    pkv.kv_append_fp8_e4m3(kq, vq, torch.arange(nb * 16, dtype=torch.int64, device="cuda"), tok(kb), tok(vb))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, kn, vn = (dev(x).view(torch.bfloat16) for x in (w.q, w.k_new, w.v_new))
    tables, ctx, slots = dev(w.block_tables), dev(w.context_lens), dev(w.slot_mapping)
    maxb = w.max_blocks_per_seq
    bps = pkv.choose_kv_blocks_per_split_fp8_e4m3(w.num_seqs, hkv, maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(w.num_seqs, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    kf, vf = kq.clone(), vq.clone()
    out_s, out_f = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
    pkv.kv_append_fp8_e4m3(kq, vq, slots, kn, vn)
    pkv.paged_attention_fp8_e4m3(out_s, q, kq, vq, tables, ctx, w.scale, kv_blocks_per_split=bps, workspace=ws)
    pkv.paged_attention_fp8_e4m3_append(out_f, q, kf, vf, tables, ctx, w.scale, slots, kn, vn,
                                        kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16)), "full-size fp8: outputs differ"
    assert torch.equal(kf, kq) and torch.equal(vf, vq), "full-size fp8: pools differ"
    assert torch.isfinite(out_f.float()).all()
    _sampled_oracle_check(w, kb, vb, out_f, kf, vf, fp8=True)


def _sampled_oracle_check(w, kb, vb, out, kpool, vpool, fp8):
    """Requests 0, 17 and 36 of a full-size batch against the oracle: their
    blocks of the device-filled BF16 pools (E4M3-rounded by the oracle for
    fp8) plus the new token appended by the oracle, compared with the blocks
    the fused call left (bit for bit) and with its output."""
    got = bf16_to_f64(out)
    for r in [0, 17, 36]:
        n = -(-int(w.context_lens[r]) // 16)
        idx = torch.from_numpy(w.block_tables[r, :n].astype(np.int64)).cuda()
        sub = lambda p: p.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)
        kh, vh = sub(kb), sub(vb)
        slot = int(w.slot_mapping[r])
        assert slot // 16 == int(w.block_tables[r, n - 1])
        sub_slot = np.array([(n - 1) * 16 + slot % 16], np.int64)
        table = np.arange(n, dtype=np.int32)[None, :]
        if fp8:
            ref, kq_ref, vq_ref = _fp8_oracle(w, *_fp8_host_pools(kh, vh), q=w.q[r:r + 1], tables=table,
                                              ctx=w.context_lens[r:r + 1], slots=sub_slot,
                                              k_new=w.k_new[r:r + 1], v_new=w.v_new[r:r + 1])
            k_got, v_got = kpool.index_select(0, idx).cpu().numpy(), vpool.index_select(0, idx).cpu().numpy()
        else:
            kq_ref, vq_ref = kh.copy(), vh.copy()
            oracle.kv_append(kq_ref, vq_ref, sub_slot, w.k_new[r:r + 1], w.v_new[r:r + 1])
            ref = oracle.paged_attention(w.q[r:r + 1], kq_ref, vq_ref, table, w.context_lens[r:r + 1], 1, w.scale)
            k_got, v_got = sub(kpool), sub(vpool)
        assert np.array_equal(k_got, kq_ref) and np.array_equal(v_got, vq_ref), f"request {r}: pool bytes"
        assert_close(got[r:r + 1], ref, what=f"full-size fused request {r} vs oracle")


def test_fused_bf16_short_chat_full_size():
    """The benchmark's default step at full size (37 requests, 5461-block BF16
    pools filled on the device, the library's split choice): the fused call
    equals the append followed by the attention, outputs and pools bit for
    bit."""
    w = W.short_chat(seed=23, fill_cache=False)
    nb, hkv = w.num_blocks, w.num_kv_heads
    kc = torch.empty((nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    W.fill_pool_device(kc, seed=23)
    W.fill_pool_device(vc, seed=24)
    kb0, vb0 = kc.clone(), vc.clone()  # the pools before the step, for the oracle
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, kn, vn = (dev(x).view(torch.bfloat16) for x in (w.q, w.k_new, w.v_new))
    tables, ctx, slots = dev(w.block_tables), dev(w.context_lens), dev(w.slot_mapping)
    maxb = w.max_blocks_per_seq
    bps = pkv.choose_kv_blocks_per_split(w.num_seqs, hkv, 1, maxb)
    ws = torch.empty(max(pkv.workspace_size(w.num_seqs, 1, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    kf, vf = kc.clone(), vc.clone()
    out_s, out_f = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
    pkv.kv_append(kc, vc, slots, kn, vn)
    pkv.paged_attention(out_s, q, kc, vc, tables, ctx, 1, w.scale, kv_blocks_per_split=bps, workspace=ws)
    pkv.paged_attention_append(out_f, q, kf, vf, tables, ctx, 1, w.scale, slots, kn, vn, kv_blocks_per_split=bps,
                               workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16)), "full-size bf16: outputs differ"
    assert torch.equal(kf.view(torch.int16), kc.view(torch.int16)) and \
        torch.equal(vf.view(torch.int16), vc.view(torch.int16)), "full-size bf16: pools differ"
    assert torch.isfinite(out_f.float()).all()
    _sampled_oracle_check(w, kb0, vb0, out_f, kf, vf, fp8=False)


def _empty_row_with_slot(fp8):
    """Request 1 has context 0 but a slot >= 0 (a spare block of the pool):
    the fused call stores nothing there and reports PKV_DEVERR_SLOT; the other
    rows are unaffected."""
    ctx = np.asarray([100, 0, 300])
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("empty-row-slot", ctx, need + 30, seed=67)
    used = set()
    for r, c in enumerate(ctx):
        used.update(int(b) for b in w.block_tables[r, :-(-int(c) // 16)])
    spare = next(b for b in range(w.num_blocks) if b not in used)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[1] = spare * 16 + 7
    d = to_device(w)
    out = torch.full_like(d["q"], float("nan"))
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    if fp8:
        kc, vc = _fp8_pools(d, w)
        k0, v0 = kc.clone(), vc.clone()
        pkv.paged_attention_fp8_e4m3_append(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                            d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=1000,
                                            workspace=ws)
    else:
        kc, vc = d["k_cache"], d["v_cache"]
        k0, v0 = kc.clone(), vc.clone()
        pkv.paged_attention_append(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], 1, w.scale,
                                   d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=1000,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    assert torch.equal(kc[spare], k0[spare]) and torch.equal(vc[spare], v0[spare]), "token stored for an empty row"
    assert not out[1].float().abs().sum(), "empty row must output zeros"
    w.slot_mapping[1] = -1  # what the other rows must see: the step without request 1's token
    if fp8:
        ref = _fp8_oracle(w, *_fp8_host_pools(w.k_cache, w.v_cache))[0]
    else:
        ref = oracle.run_workload(w)
    assert_close(bf16_to_f64(out), ref, what="rows beside an empty row with a slot")


def test_fused_empty_row_with_a_slot_stores_nothing_and_sets_the_error_word():
    _empty_row_with_slot(fp8=False)


def test_fused_fp8_empty_row_with_a_slot_stores_nothing_and_sets_the_error_word():
    _empty_row_with_slot(fp8=True)


# ---------------------------------------------------------------------------
# q8_0: the append fused into the q8_0 decode kernel (pkv_paged_attention_q8_0_append)
# ---------------------------------------------------------------------------

def _q8_host_pools(k_pool: np.ndarray, v_pool: np.ndarray):
    """q8_0 pools holding BF16 host pools, stored by the oracle's quantising append."""
    nb, hkv = k_pool.shape[:2]
    kq = np.zeros((nb, hkv, oracle.Q8_TILE_BYTES), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_q8_0(kq, vq, np.arange(nb * 16, dtype=np.int64), _tokens_of_pool(k_pool),
                          _tokens_of_pool(v_pool))
    return kq, vq


def _q8_oracle(w, kq: np.ndarray, vq: np.ndarray):
    """The step with the oracle on copies of host q8_0 pools: the quantising
    append of the new tokens, then FP64 attention over the stored values."""
    kq, vq = kq.copy(), vq.copy()
    oracle.kv_append_q8_0(kq, vq, w.slot_mapping, w.k_new, w.v_new)
    out = oracle.paged_attention_f64(w.q, oracle.dequantize_q8_0(kq), oracle.dequantize_q8_0(vq), w.block_tables,
                                     w.context_lens, 1, w.scale)
    return out, kq, vq


def _q8_both(w, bps=0):
    d = to_device(w)
    kh, vh = _q8_host_pools(w.k_cache, w.v_cache)
    kq, vq = torch.from_numpy(kh).cuda(), torch.from_numpy(vh).cuda()
    maxb = w.max_blocks_per_seq
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split_q8_0(w.num_seqs, w.num_kv_heads, maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(w.num_seqs, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    res = []
    for fused in (True, False):
        kc, vc = kq.clone(), vq.clone()
        out = torch.full_like(d["q"], float("nan"))
        if fused:
            pkv.paged_attention_q8_0_append(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                            d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=bps,
                                            workspace=ws)
        else:
            pkv.kv_append_q8_0(kc, vc, d["slot_mapping"], d["k_new"], d["v_new"])
            pkv.paged_attention_q8_0(out, d["q"], kc, vc, d["block_tables"], d["context_lens"], w.scale,
                                     kv_blocks_per_split=bps, workspace=ws)
        torch.cuda.synchronize()
        res.append((out, kc, vc))
    return res, (kh, vh)


def _assert_q8(res, host, w, what):
    (of, kf, vf), (os_, ks, vs) = res
    assert torch.equal(of.view(torch.int16), os_.view(torch.int16)), f"{what}: outputs differ"
    assert torch.equal(kf, ks) and torch.equal(vf, vs), f"{what}: q8_0 pools differ"
    ref, kq, vq = _q8_oracle(w, *host)
    assert np.array_equal(kf.cpu().numpy(), kq) and np.array_equal(vf.cpu().numpy(), vq), \
        f"{what}: q8_0 pools differ from the oracle's append"
    assert_close(bf16_to_f64(of), ref, what=f"{what} vs oracle")


# new tokens at every row of a 128-token tile modulo 8 and in each of its four
# 32-row quarters (the dequantisation warp and the attention warp that take
# the row), at a block's first and last slot, alone, and a padding row
RAGGED_Q8 = [17, 300, 1, 16, 700, 0, 32, 2049, 129, 200, 4000, 46, 87, 110, 128, 77, 94, 123, 42]


@pytest.mark.parametrize("bps", [0, 8, 24, 5, 1000])
def test_fused_q8_equals_append_then_attention_and_oracle(bps):
    ctx = np.asarray(RAGGED_Q8)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("fused-q8", ctx, need + 30, seed=73)
    res, host = _q8_both(w, bps)
    _assert_q8(res, host, w, f"fused q8_0 bps={bps}")
    assert not res[0][0][ctx == 0].float().abs().sum()


@pytest.mark.parametrize("seed", range(6))
def test_fused_q8_random_shapes(seed):
    rng = np.random.default_rng(7000 + seed)
    b = int(rng.integers(1, 61))
    ctx = rng.integers(0, 3001, size=b)
    ctx[rng.random(b) < 0.1] = 0
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("fused-q8-rand", ctx, need + 16, seed=8000 + seed)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[rng.random(b) < 0.1] = -1
    bps = int(rng.choice([0, 0, 8, 16, 40, 1000]))
    res, host = _q8_both(w, bps)
    _assert_q8(res, host, w, f"q8_0 random seed={seed} b={b} bps={bps}")


def test_fused_q8_wrong_slot_sets_the_error_word():
    ctx = np.asarray([100, 200, 300])
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("bad-slot-q8", ctx, need + 30, seed=74)
    used = set()
    for r, c in enumerate(ctx):
        used.update(int(b) for b in w.block_tables[r, :-(-int(c) // 16)])
    spare = next(b for b in range(w.num_blocks) if b not in used)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[2] = spare * 16 + 5
    d = to_device(w)
    kh, vh = _q8_host_pools(w.k_cache, w.v_cache)
    kq, vq = torch.from_numpy(kh).cuda(), torch.from_numpy(vh).cuda()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_attention_q8_0_append(out, d["q"], kq, vq, d["block_tables"], d["context_lens"], w.scale,
                                    d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=1000, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    # stored where the slot says, as the append would
    ref_k, ref_v = kh.copy(), vh.copy()
    oracle.kv_append_q8_0(ref_k, ref_v, w.slot_mapping, w.k_new, w.v_new)
    assert np.array_equal(kq.cpu().numpy()[spare], ref_k[spare]) and np.array_equal(vq.cpu().numpy()[spare],
                                                                                     ref_v[spare])


def test_fused_q8_empty_row_with_a_slot_stores_nothing_and_sets_the_error_word():
    ctx = np.asarray([100, 0, 300])
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("empty-row-q8", ctx, need + 30, seed=75)
    used = set()
    for r, c in enumerate(ctx):
        used.update(int(b) for b in w.block_tables[r, :-(-int(c) // 16)])
    spare = next(b for b in range(w.num_blocks) if b not in used)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[1] = spare * 16 + 7
    d = to_device(w)
    kh, vh = _q8_host_pools(w.k_cache, w.v_cache)
    kq, vq = torch.from_numpy(kh).cuda(), torch.from_numpy(vh).cuda()
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    pkv.paged_attention_q8_0_append(out, d["q"], kq, vq, d["block_tables"], d["context_lens"], w.scale,
                                    d["slot_mapping"], d["k_new"], d["v_new"], kv_blocks_per_split=1000, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    assert np.array_equal(kq.cpu().numpy()[spare], kh[spare]) and np.array_equal(vq.cpu().numpy()[spare], vh[spare])
    assert not out[1].float().abs().sum()
    w.slot_mapping[1] = -1
    assert_close(bf16_to_f64(out), _q8_oracle(w, kh, vh)[0], what="rows beside an empty q8_0 row with a slot")


def test_fused_q8_short_chat_full_size():
    """The 2K-context batch at full size (37 requests, 5461-block pools filled
    on the device and quantised by the append) in the benchmark's launch
    configuration: the fused call equals the append followed by the attention,
    outputs and pools bit for bit, and sampled requests match the oracle."""
    w = W.short_chat(seed=25, fill_cache=False)
    nb, hkv = w.num_blocks, w.num_kv_heads
    kb = torch.empty((nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    vb = torch.empty_like(kb)
    W.fill_pool_device(kb, seed=25)
    W.fill_pool_device(vb, seed=26)
    tok = lambda p: p.permute(0, 2, 1, 3).contiguous().view(nb * 16, hkv, 128)
    kq = torch.empty((nb, hkv, pkv.Q8_TILE_BYTES), dtype=torch.uint8, device="cuda")
    vq = torch.empty_like(kq)
    pkv.kv_append_q8_0(kq, vq, torch.arange(nb * 16, dtype=torch.int64, device="cuda"), tok(kb), tok(vb))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, kn, vn = (dev(x).view(torch.bfloat16) for x in (w.q, w.k_new, w.v_new))
    tables, ctx, slots = dev(w.block_tables), dev(w.context_lens), dev(w.slot_mapping)
    maxb = w.max_blocks_per_seq
    bps = pkv.choose_kv_blocks_per_split_q8_0(w.num_seqs, hkv, maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(w.num_seqs, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    kf, vf = kq.clone(), vq.clone()
    out_s, out_f = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
    pkv.kv_append_q8_0(kq, vq, slots, kn, vn)
    pkv.paged_attention_q8_0(out_s, q, kq, vq, tables, ctx, w.scale, kv_blocks_per_split=bps, workspace=ws)
    pkv.paged_attention_q8_0_append(out_f, q, kf, vf, tables, ctx, w.scale, slots, kn, vn, kv_blocks_per_split=bps,
                                    workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16)), "full-size q8_0: outputs differ"
    assert torch.equal(kf, kq) and torch.equal(vf, vq), "full-size q8_0: pools differ"
    got = bf16_to_f64(out_f)
    for r in [0, 17, 36]:
        n = -(-int(w.context_lens[r]) // 16)
        idx = torch.from_numpy(w.block_tables[r, :n].astype(np.int64)).cuda()
        sub = lambda p: p.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)
        kq_ref, vq_ref = _q8_host_pools(sub(kb), sub(vb))
        slot = int(w.slot_mapping[r])
        sub_slot = np.array([(n - 1) * 16 + slot % 16], np.int64)
        oracle.kv_append_q8_0(kq_ref, vq_ref, sub_slot, w.k_new[r:r + 1], w.v_new[r:r + 1])
        assert np.array_equal(kf.index_select(0, idx).cpu().numpy(), kq_ref) and \
            np.array_equal(vf.index_select(0, idx).cpu().numpy(), vq_ref), f"request {r}: q8_0 pool bytes"
        ref = oracle.paged_attention_f64(w.q[r:r + 1], oracle.dequantize_q8_0(kq_ref), oracle.dequantize_q8_0(vq_ref),
                                         np.arange(n, dtype=np.int32)[None, :], w.context_lens[r:r + 1], 1, w.scale)
        assert_close(got[r:r + 1], ref, what=f"full-size fused q8_0 request {r} vs oracle")


# contexts that fill the whole block table (the new token in its last slot) or
# stop one token short of it or one past a block, beside a short row and a
# padding row; 41 blocks per table leave a ragged last tile in every format
FULL_TABLE_BLOCKS = 41
FULL_TABLE_CTX = [41 * 16, 41 * 16, 41 * 16 - 1, 40 * 16 + 1, 17, 0]


@pytest.mark.parametrize("fmt", ["bf16", "q8_0", "fp8_e4m3"])
@pytest.mark.parametrize("bps", [0, 8, 1000])
def test_contexts_that_fill_the_block_table(fmt, bps):
    ctx = np.asarray(FULL_TABLE_CTX)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("full-table", ctx, need + 12, seed=91, max_blocks=FULL_TABLE_BLOCKS)
    assert w.max_blocks_per_seq == FULL_TABLE_BLOCKS
    what = f"full table {fmt} bps={bps}"
    if fmt == "bf16":
        res = _both(w, bps)
        _assert_same(res, what)
        out, kf, vf = res[0]
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
        assert np.array_equal(kf.cpu().view(torch.int16).numpy().view(np.uint16), kc), f"{what}: K pool"
        assert np.array_equal(vf.cpu().view(torch.int16).numpy().view(np.uint16), vc), f"{what}: V pool"
        assert_close(bf16_to_f64(out), oracle.run_workload(w), what=f"{what} vs oracle")
    elif fmt == "q8_0":
        res, host = _q8_both(w, bps)
        _assert_q8(res, host, w, what)
    else:
        res = _fp8_both(w, bps)
        _assert_same_fp8(res, what)
        _assert_fp8_oracle(res, w, what)
    assert not res[0][0][ctx == 0].float().abs().sum()


@pytest.mark.parametrize("fmt", ["q8_0", "fp8_e4m3"])
def test_fused_quantised_many_units_per_cta(fmt):
    """130 requests x 8 KV heads = 1040 units with a new token over at most
    152 persistent CTAs: every CTA handles 6 or more, so the q8_0 append
    warp's 4-slot ready ring wraps and the E4M3 kernel's per-unit (parity)
    buffers are reused many times."""
    rng = np.random.default_rng(95)
    ctx = rng.integers(1, 300, size=130)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("many-units-" + fmt, ctx, need + 16, seed=96)
    if fmt == "q8_0":
        res, host = _q8_both(w, 1000)
        _assert_q8(res, host, w, "q8_0 many units per CTA")
    else:
        res = _fp8_both(w, 1000)
        _assert_same_fp8(res, "E4M3 many units per CTA")
        _assert_fp8_oracle(res, w, "E4M3 many units per CTA")
