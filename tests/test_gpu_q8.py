"""q8_0 KV path (through the C ABI) against the FP64 oracle on the same seeded
inputs: the quantising append must be bit-exact; attention over the q8_0
pools must be within max-abs 1e-2 and relative L2 5e-3 of the oracle's
attention over the dequantised values."""
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

TILE = oracle.Q8_TILE_BYTES


@pytest.fixture(autouse=True)
def _clear_device_error():
    if pkv is not None:
        pkv.get_device_error(reset=True)
    yield
    if pkv is not None:
        assert pkv.get_device_error(reset=True) == 0


def tokens_of_pool(pool: np.ndarray) -> np.ndarray:
    """BF16 pool [nb][Hkv][16][128] -> token-major rows [nb*16][Hkv][128] (slot order)."""
    nb, hkv, bs, d = pool.shape
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))


def q8_pools_oracle(k_pool: np.ndarray, v_pool: np.ndarray):
    """Quantise whole BF16 pools with the oracle."""
    nb, hkv = k_pool.shape[:2]
    kq = np.zeros((nb, hkv, TILE), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_q8_0(kq, vq, np.arange(nb * 16, dtype=np.int64), tokens_of_pool(k_pool), tokens_of_pool(v_pool))
    return kq, vq


def run_q8(q, kq, vq, tables, ctx, scale, bps=0):
    b = ctx.shape[0]
    maxb = tables.shape[1]
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split_q8_0(b, kq.shape[1], maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(b, q.shape[2], maxb, bps), 1), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    pkv.paged_attention_q8_0(out, q, kq, vq, tables, ctx, scale, kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    return out


def oracle_q8(q, kq, vq, tables, ctx, scale):
    return oracle.paged_attention_f64(q, oracle.dequantize_q8_0(kq), oracle.dequantize_q8_0(vq), tables, ctx, 1,
                                      scale)


def spread_magnitudes(rng, rows: np.ndarray) -> np.ndarray:
    """Scale each 32-value group of BF16 rows by its own power of two (exact)
    and zero a few groups, so scales span a wide range."""
    x = (rows.astype(np.uint32) << 16).view(np.float32).reshape(*rows.shape[:-1], 4, 32)
    e = rng.integers(-6, 7, size=x.shape[:-1] + (1,)).astype(np.float32)
    x = x * np.float32(2.0) ** e
    x[rng.random(x.shape[:-1]) < 0.05] = 0.0
    return (x.reshape(rows.shape).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [1, 2])
def test_q8_append_bit_exact(seed):
    rng = np.random.default_rng(seed)
    w = W.tiny(seed=seed)
    k_new, v_new = spread_magnitudes(rng, w.k_new), spread_magnitudes(rng, w.v_new)
    slots = w.slot_mapping.copy()
    slots[1] = -1  # padding row: skipped
    kq, vq = q8_pools_oracle(w.k_cache, w.v_cache)
    kd, vd = dev(kq), dev(vq)
    pkv.kv_append_q8_0(kd, vd, dev(slots), dev(k_new), dev(v_new))
    oracle.kv_append_q8_0(kq, vq, slots, k_new, v_new)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq)


def test_q8_append_whole_pool_bit_exact():
    """Every slot of a pool quantised on the GPU equals the oracle's bytes."""
    rng = np.random.default_rng(9)
    nb, hkv = 96, 8
    k_pool = spread_magnitudes(rng, W.randn_bf16(rng, (nb, hkv, 16, 128)))
    v_pool = spread_magnitudes(rng, W.randn_bf16(rng, (nb, hkv, 16, 128)))
    kq, vq = q8_pools_oracle(k_pool, v_pool)
    kd = torch.zeros((nb, hkv, TILE), dtype=torch.uint8, device="cuda")
    vd = torch.zeros_like(kd)
    pkv.kv_append_q8_0(kd, vd, dev(np.arange(nb * 16, dtype=np.int64)), dev(tokens_of_pool(k_pool)),
                       dev(tokens_of_pool(v_pool)))
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq)


def test_q8_append_slot_outside_pool_sets_error():
    w = W.tiny(seed=3)
    kq, vq = q8_pools_oracle(w.k_cache, w.v_cache)
    kd, vd = dev(kq), dev(vq)
    slots = np.full(w.slot_mapping.shape, -1, np.int64)
    slots[0] = w.num_blocks * 16 + 5
    pkv.kv_append_q8_0(kd, vd, dev(slots), dev(w.k_new), dev(w.v_new))
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_SLOT
    assert np.array_equal(kd.cpu().numpy(), kq)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def test_q8_tiny_append_then_attention():
    """The small workload: 4 requests {17, 64, 100, 256}, append of this step's token, then attention."""
    w = W.tiny(seed=4)
    kq, vq = q8_pools_oracle(w.k_cache, w.v_cache)
    kd, vd = dev(kq), dev(vq)
    pkv.kv_append_q8_0(kd, vd, dev(w.slot_mapping), dev(w.k_new), dev(w.v_new))
    oracle.kv_append_q8_0(kq, vq, w.slot_mapping, w.k_new, w.v_new)
    out = run_q8(dev(w.q), kd, vd, dev(w.block_tables), dev(w.context_lens), w.scale)
    ref = oracle_q8(w.q, kq, vq, w.block_tables, w.context_lens, w.scale)
    assert_close(bf16_to_f64(out), ref, what="q8 tiny")


def _ragged(seed, ctx, num_blocks=None, hkv=8):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    need = sum(-(-int(c) // 16) for c in ctx)
    nb = num_blocks or need + 7
    maxb = max(1, max(-(-int(c) // 16) for c in ctx))
    perm = rng.permutation(nb)
    tables = np.zeros((len(ctx), maxb), np.int32)
    k = 0
    for r, c in enumerate(ctx):
        n = -(-int(c) // 16)
        tables[r, :n] = perm[k:k + n]
        tables[r, n:] = rng.integers(0, nb, size=maxb - n)  # unused entries: arbitrary but inside the pool
        k += n
    k_pool = W.randn_bf16(rng, (nb, hkv, 16, 128))
    v_pool = W.randn_bf16(rng, (nb, hkv, 16, 128))
    q = W.randn_bf16(rng, (len(ctx), 1, 4 * hkv, 128))
    kq, vq = q8_pools_oracle(k_pool, v_pool)
    return q, kq, vq, tables, ctx


@pytest.mark.parametrize("bps", [0, 8, 16, 24, 5])
def test_q8_ragged_contexts_and_splits(bps):
    """Ragged tails, a 1-token request, a full 8-block tile boundary, splits
    that cut tiles (bps 5, 24) and the combine pass."""
    q, kq, vq, tables, ctx = _ragged(5, [1, 17, 128, 129, 300, 640, 1000, 2055])
    scale = 128 ** -0.5
    out = run_q8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale, bps=bps)
    assert_close(bf16_to_f64(out), oracle_q8(q, kq, vq, tables, ctx, scale), what=f"q8 ragged bps={bps}")


def test_q8_empty_context_gives_zeros():
    q, kq, vq, tables, ctx = _ragged(6, [0, 40, 0, 200], hkv=2)
    scale = 128 ** -0.5
    out = run_q8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale, bps=8)
    got = bf16_to_f64(out)
    assert not got[0].any() and not got[2].any()
    assert_close(got, oracle_q8(q, kq, vq, tables, ctx, scale), what="q8 empty rows")


def test_q8_many_units_per_cta():
    """More (request, KV head) units than SMs: every persistent CTA walks
    several units with different lengths."""
    rng = np.random.default_rng(7)
    ctx = rng.integers(1, 400, size=48)
    q, kq, vq, tables, ctx = _ragged(7, ctx)
    scale = 128 ** -0.5
    out = run_q8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale)
    assert_close(bf16_to_f64(out), oracle_q8(q, kq, vq, tables, ctx, scale), what="q8 many units")


def unused_slots(tables, ctx, nb):
    """(block, offset) pairs no context covers: the tails of last blocks and
    blocks no table reaches within its context."""
    used = np.zeros((nb, 16), bool)
    for r, c in enumerate(ctx):
        for t in range(int(c)):
            used[tables[r, t // 16], t % 16] = True
    return np.argwhere(~used)


@pytest.mark.parametrize("bps", [0, 5])
def test_q8_nan_patterns_in_unused_slots(bps):
    """Slots past every context hold NaN scales and extreme codes: they must
    never reach a result (ragged last tiles read them into shared memory)."""
    q, kq, vq, tables, ctx = _ragged(12, [1, 17, 129, 250, 333])
    kq, vq = kq.copy(), vq.copy()
    for blk, off in unused_slots(tables, ctx, kq.shape[0]):
        for pool in (kq, vq):
            pool[blk, :, off * 128:(off + 1) * 128] = 0x7F
            pool[blk, :, 2048 + off * 8:2048 + (off + 1) * 8] = 0xFF  # FP16 NaN scales
    scale = 128 ** -0.5
    out = run_q8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), scale, bps=bps)
    assert_close(bf16_to_f64(out), oracle_q8(q, kq, vq, tables, ctx, scale), what=f"q8 NaN slots bps={bps}")


def test_q8_large_queries_are_rescaled_into_fp16_range():
    """Queries of magnitude ~2^20 (beyond FP16) with the scale shrunk to
    match: the kernel shifts them by a power of two, the result is unchanged."""
    q, kq, vq, tables, ctx = _ragged(8, [90, 333], hkv=2)
    big = ((q.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** 20)).view(np.uint32) >> 16
    big = big.astype(np.uint16)
    scale = 128 ** -0.5 * 2.0 ** -20
    out = run_q8(dev(big), dev(kq), dev(vq), dev(tables), dev(ctx), scale)
    assert_close(bf16_to_f64(out), oracle_q8(big, kq, vq, tables, ctx, scale), what="q8 large q")


def test_q8_bad_block_id_sets_error():
    q, kq, vq, tables, ctx = _ragged(9, [50, 70], hkv=2)
    tables = tables.copy()
    tables[1, 2] = kq.shape[0] + 10
    run_q8(dev(q), dev(kq), dev(vq), dev(tables), dev(ctx), 128 ** -0.5)
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_BLOCK_ID


def test_q8_copy_blocks_bit_copy():
    rng = np.random.default_rng(10)
    kq = rng.integers(0, 256, size=(12, 8, TILE), dtype=np.uint8)
    vq = rng.integers(0, 256, size=(12, 8, TILE), dtype=np.uint8)
    kd, vd = dev(kq), dev(vq)
    src, dst = np.array([1, 4, 7], np.int32), np.array([9, 0, 11], np.int32)
    pkv.copy_blocks_q8_0(kd, vd, dev(src), dev(dst))
    kq[dst], vq[dst] = kq[src], vq[src]
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq)


def test_q8_short_chat_full_size_sampled():
    """The 2K-context batch at full size (37 requests, 2048 + U[0,255] tokens,
    a pool of 5461 blocks): pools filled on the device, quantised by the GPU
    append (its bytes checked against the oracle on the sampled requests'
    blocks), attention checked on sampled requests."""
    w = W.short_chat(seed=11, fill_cache=False)
    nb, hkv = w.num_blocks, w.num_kv_heads
    kb = torch.empty((nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    vb = torch.empty_like(kb)
    W.fill_pool_device(kb, seed=11)
    W.fill_pool_device(vb, seed=12)
    kd = torch.empty((nb, hkv, TILE), dtype=torch.uint8, device="cuda")
    vd = torch.empty_like(kd)
    tok = lambda p: p.permute(0, 2, 1, 3).contiguous().view(nb * 16, hkv, 128)
    pkv.kv_append_q8_0(kd, vd, torch.arange(nb * 16, dtype=torch.int64, device="cuda"), tok(kb), tok(vb))
    q = dev(w.q)
    out = run_q8(q, kd, vd, dev(w.block_tables), dev(w.context_lens), w.scale)
    got = bf16_to_f64(out)
    sample = [0, 13, 36]
    for r in sample:
        n = -(-int(w.context_lens[r]) // 16)
        blocks = w.block_tables[r, :n]
        idx = torch.from_numpy(blocks.astype(np.int64)).cuda()
        k_sub = kb.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)
        v_sub = vb.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)
        kq_ref, vq_ref = q8_pools_oracle(k_sub, v_sub)
        kq_sub, vq_sub = kd.index_select(0, idx).cpu().numpy(), vd.index_select(0, idx).cpu().numpy()
        assert np.array_equal(kq_sub, kq_ref) and np.array_equal(vq_sub, vq_ref), f"request {r}: q8 bytes"
        table = np.arange(n, dtype=np.int32)[None, :]
        ref = oracle_q8(w.q[r:r + 1], kq_sub, vq_sub, table, w.context_lens[r:r + 1], w.scale)
        assert_close(got[r:r + 1], ref, what=f"q8 short request {r}")
