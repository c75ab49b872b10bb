"""Decode batches of at least two (request, KV head) rows per SM run on the
persistent tensor-core decode kernel.  Same bar as the other parity tests:
bit-exact indexing (placement invariance), attention within max-abs 1e-2 and
relative L2 5e-3 of the FP64 oracle, device errors reported, nothing read
from unused slots."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, dev, to_device

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_decode_attention_gb300 as pkv
else:  # collected on CPU-only machines, every test skipped
    pkv = None

NAN_BF16 = np.uint16(0x7FC0)


@pytest.fixture(autouse=True)
def _clear_device_error():
    if pkv is not None:
        pkv.get_device_error(reset=True)
    yield
    if pkv is not None:
        assert pkv.get_device_error(reset=True) == 0


def big_batch_rows() -> int:
    """Requests needed for the tensor-core decode (8 KV heads, 2 rows per SM)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return -(-2 * sms // 8)


def run(w, bps=0, append=True, d=None):
    if d is None:
        d = to_device(w)
    if append:
        pkv.kv_append(d["k_cache"], d["v_cache"], d["slot_mapping"], d["k_new"], d["v_new"])
    maxb = w.max_blocks_per_seq
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split(w.num_seqs, w.num_kv_heads, 1, maxb)
    ws = torch.empty(max(pkv.workspace_size(w.num_seqs, 1, w.num_q_heads, maxb, bps), 1), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_attention(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], 1, w.scale,
                        kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    return out


def ragged_contexts(n, seed):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, 700, size=n)
    ctx[:12] = [0, 1, 2, 15, 16, 17, 127, 128, 129, 255, 256, 0]
    return ctx


@pytest.mark.parametrize("num_seqs,lo,hi", [(24, 2048, 2304), (16, 3000, 4200), (34, 1900, 2100)])
def test_mid_batch_that_would_underfill_the_row_kernel(num_seqs, lo, hi):
    """Batches of 3/4 to 2 rows per SM whose CTA-per-row plan leaves more than a
    tenth of its slots empty also run on the persistent tensor-core kernel
    (split by its makespan model): same bar against the oracle."""
    rng = np.random.default_rng(num_seqs)
    ctx = rng.integers(lo, hi, size=num_seqs)
    ctx[0] = hi  # the longest request sets the block count the dispatch reads
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("tc-mid", ctx, need + 40, seed=num_seqs)
    bps = pkv.choose_kv_blocks_per_split(w.num_seqs, w.num_kv_heads, 1, w.max_blocks_per_seq)
    assert bps % 8 == 0 or bps == w.max_blocks_per_seq  # the persistent kernel's split, in whole tiles
    assert_close(bf16_to_f64(run(w)), oracle.run_workload(w), what=f"tc mid batch {num_seqs}")


@pytest.mark.parametrize("bps", [0, 8, 24, 5, 1000])
def test_big_batch_ragged_with_nan_in_unused_slots(bps):
    ctx = ragged_contexts(big_batch_rows() + 9, seed=21)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("tc-ragged", ctx, need + 40, seed=21)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    used = np.zeros((w.num_blocks, 16), bool)
    for r, c in enumerate(ctx):
        for t in range(int(c)):
            used[w.block_tables[r, t // 16], t % 16] = True
    kc.transpose(0, 2, 1, 3)[~used] = NAN_BF16
    vc.transpose(0, 2, 1, 3)[~used] = NAN_BF16
    w2 = W.Workload(**{**w.__dict__, "k_cache": kc, "v_cache": vc})
    got = bf16_to_f64(run(w2, bps=bps, append=False))
    assert not got[ctx == 0].any()
    assert_close(got, oracle.run_workload(w2, append=False), what=f"tc ragged bps={bps}")


def test_big_batch_append_then_attention_and_placement_invariance():
    n = big_batch_rows() + 2
    rng = np.random.default_rng(22)
    ctx = rng.integers(200, 1500, size=n)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("tc-perm", ctx, need + 16, seed=22)
    a = run(w, bps=24)
    assert_close(bf16_to_f64(a), oracle.run_workload(w), what="tc append+attention")
    perm = np.random.default_rng(7).permutation(w.num_blocks)
    inv = np.argsort(perm)
    w2 = W.Workload(**{**w.__dict__, "k_cache": np.ascontiguousarray(w.k_cache[perm]),
                       "v_cache": np.ascontiguousarray(w.v_cache[perm]),
                       "block_tables": inv[w.block_tables].astype(np.int32),
                       "slot_mapping": np.where(w.slot_mapping >= 0,
                                                inv[w.slot_mapping // 16] * 16 + w.slot_mapping % 16, -1)})
    b = run(w2, bps=24)
    assert torch.equal(a, b)


def test_big_batch_peaky_logits():
    n = big_batch_rows() + 1
    rng = np.random.default_rng(23)
    ctx = rng.integers(30, 1200, size=n)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("tc-peaky", ctx, need + 8, seed=23)
    w.q = W.bf16_bits((w.q.astype(np.uint32) << 16).view(np.float32) * 8.0)
    for bps in (16, 1000):
        assert_close(bf16_to_f64(run(w, bps=bps)), oracle.run_workload(w), what=f"tc peaky bps={bps}")


def test_big_batch_special_cases():
    n = big_batch_rows()
    # ctx = 1 everywhere: the output is v0 exactly
    w = W.build("tc-one", [1] * n, n + 4, seed=24)
    out = run(w)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    for r in range(n):
        blk = w.block_tables[r, 0]
        assert np.array_equal(got[r, 0], np.repeat(vc[blk, :, 0], 4, axis=0))
    # identical V rows: that row, to BF16 rounding
    rng = np.random.default_rng(25)
    ctx = rng.integers(20, 400, size=n)
    need = int(sum(-(-int(c) // 16) for c in ctx))
    w = W.build("tc-same", ctx, need + 4, seed=25)
    row = W.randn_bf16(np.random.default_rng(3), (8, 128))
    w.v_cache[:] = row[None, :, None, :]
    w.v_new[:] = row[None]
    ref = np.broadcast_to(np.repeat((row.astype(np.uint32) << 16).view(np.float32), 4, axis=0), (n, 1, 32, 128))
    assert_close(bf16_to_f64(run(w, bps=8)), ref.astype(np.float64), max_abs=8e-3, what="tc same-V")


def test_big_batch_bad_block_id_sets_error():
    n = big_batch_rows()
    w = W.build("tc-bad", [100] * n, 7 * n + 4, seed=26)
    d = to_device(w)
    tables = w.block_tables.copy()
    tables[5, 3] = w.num_blocks + 11
    d["block_tables"] = dev(tables)
    run(w, d=d)
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_BLOCK_ID


def test_big_batch_full_size_sampled():
    """64 requests x 4096 tokens (a sweep point) at full size, pools filled
    on the device; sampled requests checked against the oracle."""
    b, ctxlen = 64, 4096
    w = W.build("tc-full", [ctxlen] * b, b * ctxlen // 16 + 64, seed=27, fill_cache=False)
    nb = w.num_blocks
    kd = torch.empty((nb, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    W.fill_pool_device(kd, 27)
    W.fill_pool_device(vd, 28)
    d = {"q": dev(w.q), "k_cache": kd, "v_cache": vd, "block_tables": dev(w.block_tables),
         "context_lens": dev(w.context_lens)}
    got = bf16_to_f64(run(w, append=False, d=d))
    for r in (0, 31, 63):
        n = ctxlen // 16
        idx = torch.from_numpy(w.block_tables[r, :n].astype(np.int64)).cuda()
        sub = W.Workload(**{**w.__dict__, "num_blocks": n,
                            "k_cache": kd.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16),
                            "v_cache": vd.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16),
                            "q": w.q[r:r + 1], "block_tables": np.arange(n, dtype=np.int32)[None, :],
                            "context_lens": w.context_lens[r:r + 1], "slot_mapping": w.slot_mapping[:0],
                            "k_new": w.k_new[:0], "v_new": w.v_new[:0]})
        assert_close(got[r:r + 1], oracle.run_workload(sub, append=False), what=f"tc full-size request {r}")
