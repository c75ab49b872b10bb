"""FP8 (E4M3) KV path (through the C ABI) against the FP64 oracle on the same
seeded inputs: the rounding append must be bit-exact; attention over the E4M3
pools must be within max-abs 1e-2 and relative L2 5e-3 of the oracle's
attention over the stored values (query in BF16)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, dev

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


def tokens_of_pool(pool: np.ndarray) -> np.ndarray:
    nb, hkv, bs, d = pool.shape
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))


def fp8_pools_oracle(k_pool: np.ndarray, v_pool: np.ndarray):
    nb, hkv = k_pool.shape[:2]
    kq = np.zeros((nb, hkv, 16, 128), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_fp8(kq, vq, np.arange(nb * 16, dtype=np.int64), tokens_of_pool(k_pool), tokens_of_pool(v_pool))
    return kq, vq


def run_fp8(q, kq, vq, tables, ctx, scale, bps=0):
    b = ctx.shape[0]
    maxb = tables.shape[1]
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split_fp8_e4m3(b, kq.shape[1], maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(b, q.shape[2], maxb, bps), 1), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    pkv.paged_attention_fp8_e4m3(out, q, kq, vq, tables, ctx, scale, kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    return out


def oracle_fp8(q, kq, vq, tables, ctx, scale):
    return oracle.paged_attention_f64(q, oracle.dequantize_fp8(kq), oracle.dequantize_fp8(vq), tables, ctx, 1, scale)


def wide_range(rng, rows: np.ndarray) -> np.ndarray:
    """BF16 rows scaled by per-value powers of two from 2^-14 to 2^10: subnormal
    E4M3 results, saturation beyond 448, signed zeros."""
    x = (rows.astype(np.uint32) << 16).view(np.float32)
    x = x * np.float32(2.0) ** rng.integers(-14, 11, size=x.shape).astype(np.float32)
    x[rng.random(x.shape) < 0.01] = -0.0
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("seed", [1, 2])
def test_fp8_append_bit_exact(seed):
    rng = np.random.default_rng(seed)
    w = W.tiny(seed=seed)
    k_new, v_new = wide_range(rng, w.k_new), wide_range(rng, w.v_new)
    slots = w.slot_mapping.copy()
    slots[1] = -1
    kq, vq = fp8_pools_oracle(w.k_cache, w.v_cache)
    kd, vd = dev(kq), dev(vq)
    pkv.kv_append_fp8_e4m3(kd, vd, dev(slots), dev(k_new), dev(v_new))
    oracle.kv_append_fp8(kq, vq, slots, k_new, v_new)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq)


def test_fp8_append_every_bf16_value():
    """All finite BF16 patterns through the GPU append equal the oracle's codes."""
    bits = np.arange(65536, dtype=np.uint32)
    finite = np.isfinite((bits << 16).view(np.float32))
    vals = bits[finite].astype(np.uint16)
    n = -(-vals.size // 1024) * 1024
    vals = np.concatenate([vals, np.zeros(n - vals.size, np.uint16)])
    rows = vals.reshape(-1, 8, 128)  # tokens x 8 heads x 128
    t = rows.shape[0]
    nb = -(-t // 16)
    kq = np.zeros((nb, 8, 16, 128), np.uint8)
    vq = np.zeros_like(kq)
    slots = np.arange(t, dtype=np.int64)
    kd, vd = dev(kq), dev(vq)
    pkv.kv_append_fp8_e4m3(kd, vd, dev(slots), dev(rows), dev(rows[::-1].copy()))
    oracle.kv_append_fp8(kq, vq, slots, rows, rows[::-1].copy())
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq)


def test_fp8_append_slot_outside_pool_sets_error():
    w = W.tiny(seed=3)
    kq, vq = fp8_pools_oracle(w.k_cache, w.v_cache)
    kd, vd = dev(kq), dev(vq)
    slots = np.full(w.slot_mapping.shape, -1, np.int64)
    slots[0] = w.num_blocks * 16 + 5
    pkv.kv_append_fp8_e4m3(kd, vd, dev(slots), dev(w.k_new), dev(w.v_new))
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    assert np.array_equal(kd.cpu().numpy(), kq)


def test_fp8_tiny_append_then_attention():
    w = W.tiny(seed=4)
    kq, vq = fp8_pools_oracle(w.k_cache, w.v_cache)
    kd, vd = dev(kq), dev(vq)
    pkv.kv_append_fp8_e4m3(kd, vd, dev(w.slot_mapping), dev(w.k_new), dev(w.v_new))
    oracle.kv_append_fp8(kq, vq, w.slot_mapping, w.k_new, w.v_new)
    out = run_fp8(dev(w.q), kd, vd, dev(w.block_tables), dev(w.context_lens), w.scale)
    assert_close(bf16_to_f64(out), oracle_fp8(w.q, kq, vq, w.block_tables, w.context_lens, w.scale), what="fp8 tiny")


def _ragged(seed, ctx, hkv=8):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    need = sum(-(-int(c) // 16) for c in ctx)
    nb = need + 7
    maxb = max(1, max(-(-int(c) // 16) for c in ctx))
    perm = rng.permutation(nb)
    tables = np.zeros((len(ctx), maxb), np.int32)
    k = 0
    for r, c in enumerate(ctx):
        n = -(-int(c) // 16)
        tables[r, :n] = perm[k:k + n]
        tables[r, n:] = rng.integers(0, nb, size=maxb - n)
        k += n
    kq, vq = fp8_pools_oracle(W.randn_bf16(rng, (nb, hkv, 16, 128)), W.randn_bf16(rng, (nb, hkv, 16, 128)))
    q = W.randn_bf16(rng, (len(ctx), 1, 4 * hkv, 128))
    return q, kq, vq, tables, ctx


@pytest.mark.parametrize("bps", [0, 8, 24, 5])
def test_fp8_ragged_contexts_and_splits(bps):
    q, kq, vq, tables, ctx = _ragged(5, [1, 17, 128, 129, 300, 640, 1000, 2055])
    scale = 128 ** -0.5
    out = run_fp8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale, bps=bps)
    assert_close(bf16_to_f64(out), oracle_fp8(q, kq, vq, tables, ctx, scale), what=f"fp8 ragged bps={bps}")


def unused_slots(tables, ctx, nb):
    """(block, offset) pairs no context covers."""
    used = np.zeros((nb, 16), bool)
    for r, c in enumerate(ctx):
        for t in range(int(c)):
            used[tables[r, t // 16], t % 16] = True
    return np.argwhere(~used)


@pytest.mark.parametrize("bps", [0, 5])
def test_fp8_nan_patterns_in_unused_slots(bps):
    """Slots past every context hold E4M3 NaN codes (0x7F, 0xFF): a zero
    weight times NaN is NaN, so those keys must not enter P.V at all."""
    q, kq, vq, tables, ctx = _ragged(12, [1, 17, 129, 250, 333])
    kq, vq = kq.copy(), vq.copy()
    for n, (blk, off) in enumerate(unused_slots(tables, ctx, kq.shape[0])):
        kq[blk, :, off] = 0x7F if n % 2 else 0xFF
        vq[blk, :, off] = 0xFF if n % 2 else 0x7F
    scale = 128 ** -0.5
    out = run_fp8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale, bps=bps)
    assert_close(bf16_to_f64(out), oracle_fp8(q, kq, vq, tables, ctx, scale), what=f"fp8 NaN slots bps={bps}")


def test_fp8_empty_context_and_many_units():
    rng = np.random.default_rng(7)
    ctx = rng.integers(0, 400, size=48)
    ctx[[3, 20]] = 0
    q, kq, vq, tables, ctx = _ragged(7, ctx)
    scale = 128 ** -0.5
    got = bf16_to_f64(run_fp8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale))
    assert not got[3].any() and not got[20].any()
    assert_close(got, oracle_fp8(q, kq, vq, tables, ctx, scale), what="fp8 many units")


def test_fp8_large_queries():
    q, kq, vq, tables, ctx = _ragged(8, [90, 333], hkv=2)
    big = (((q.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 20)).view(np.uint32) >> 16)
    big = big.astype(np.uint16)
    scale = 128 ** -0.5 * 2.0 ** -20
    out = run_fp8(dev(big), dev(kq), dev(vq), dev(tables), dev(ctx), scale)
    assert_close(bf16_to_f64(out), oracle_fp8(big, kq, vq, tables, ctx, scale), what="fp8 large q")


def test_fp8_query_heads_of_mixed_magnitude():
    """The tensor cores take each query head as two E4M3 parts under its own
    power-of-two scale: heads 2^-12 and 2^10 times the usual size (below
    E4M3's normal range and beyond its largest value), an all-zero head
    (uniform weights: the mean of the V rows) and an 8x sharper head (peaked
    weights that move the running maximum often) must all match the oracle."""
    q, kq, vq, tables, ctx = _ragged(10, [700, 1, 129, 2000, 37], hkv=2)
    x = (q.astype(np.uint32) << 16).view(np.float32).copy()
    factors = np.array([2.0 ** -12, 2.0 ** 10, 0.0, 8.0, 1.0, 2.0 ** -3, 3.0, 0.5], np.float32)
    x *= factors[None, None, :, None]
    qm = (x.view(np.uint32) >> 16).astype(np.uint16)
    scale = 128 ** -0.5
    for bps in (0, 24):
        out = run_fp8(dev(qm), dev(kq), dev(vq), dev(tables), dev(ctx), scale, bps=bps)
        assert_close(bf16_to_f64(out), oracle_fp8(qm, kq, vq, tables, ctx, scale), what=f"fp8 mixed heads bps={bps}")


def test_fp8_bad_block_id_sets_error():
    q, kq, vq, tables, ctx = _ragged(9, [50, 70], hkv=2)
    tables = tables.copy()
    tables[1, 2] = kq.shape[0] + 10
    run_fp8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), 128 ** -0.5)
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_BLOCK_ID


def test_fp8_copy_blocks_bit_copy():
    rng = np.random.default_rng(10)
    kq = rng.integers(0, 256, size=(12, 8, 16, 128), dtype=np.uint8)
    vq = rng.integers(0, 256, size=(12, 8, 16, 128), dtype=np.uint8)
    kd, vd = dev(kq), dev(vq)
    src, dst = np.array([1, 4, 7], np.int32), np.array([9, 0, 11], np.int32)
    pkv.copy_blocks_fp8_e4m3(kd, vd, dev(src), dev(dst))
    kq[dst], vq[dst] = kq[src], vq[src]
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq)


def test_fp8_short_chat_full_size_sampled():
    """The 2K-context batch at full size (37 requests, 5461-block pool), pools
    filled on the device and rounded by the GPU append; sampled requests
    checked against the oracle (bytes and attention)."""
    w = W.short_chat(seed=13, fill_cache=False)
    nb, hkv = w.num_blocks, w.num_kv_heads
    kb = torch.empty((nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    vb = torch.empty_like(kb)
    W.fill_pool_device(kb, seed=13)
    W.fill_pool_device(vb, seed=14)
    kd = torch.empty((nb, hkv, 16, 128), dtype=torch.uint8, device="cuda")
    vd = torch.empty_like(kd)
    tok = lambda p: p.permute(0, 2, 1, 3).contiguous().view(nb * 16, hkv, 128)
    pkv.kv_append_fp8_e4m3(kd, vd, torch.arange(nb * 16, dtype=torch.int64, device="cuda"), tok(kb), tok(vb))
    got = bf16_to_f64(run_fp8(dev(w.q), kd, vd, dev(w.block_tables), dev(w.context_lens), w.scale))
    for r in [0, 17, 36]:
        n = -(-int(w.context_lens[r]) // 16)
        idx = torch.from_numpy(w.block_tables[r, :n].astype(np.int64)).cuda()
        kq_ref, vq_ref = fp8_pools_oracle(kb.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16),
                                          vb.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16))
        kq_sub, vq_sub = kd.index_select(0, idx).cpu().numpy(), vd.index_select(0, idx).cpu().numpy()
        assert np.array_equal(kq_sub, kq_ref) and np.array_equal(vq_sub, vq_ref), f"request {r}: fp8 bytes"
        table = np.arange(n, dtype=np.int32)[None, :]
        ref = oracle_fp8(w.q[r:r + 1], kq_sub, vq_sub, table, w.context_lens[r:r + 1], w.scale)
        assert_close(got[r:r + 1], ref, what=f"fp8 short request {r}")
