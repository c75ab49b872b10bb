"""Every attention path with KV-head counts other than the 8 of the pages'
workloads (1, 2, 4 and 16 KV heads, each with its GQA group of 4 query
heads), through the C ABI against the FP64 oracle: pool tiles are indexed
(block, KV head), the tensor maps view a pool as blocks x heads x 16 rows,
and the split heuristics count (request, KV head) rows, so a head-count
mistake anywhere shows here ("Chapter 8: Inference Optimization", §8.1.1
GQA decode step; §8.3.1 block tables; §8.3.2 shared prefixes; §8.4.2 /
§8.4.4 quantised KV)."""
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

KV_HEADS = [1, 2, 4, 16]


@pytest.fixture(autouse=True)
def _clear_device_error():
    if pkv is not None:
        pkv.get_device_error(reset=True)
    yield
    if pkv is not None:
        assert pkv.get_device_error(reset=True) == 0


def _blocks(ctx, q_len=1):
    return int(sum(-(-(int(c) + q_len) // 16) for c in ctx))


def _bf16_step(w):
    """kv_append then paged_attention with the library's default split."""
    d = to_device(w)
    pkv.kv_append(d["k_cache"], d["v_cache"], d["slot_mapping"], d["k_new"], d["v_new"])
    maxb = w.max_blocks_per_seq
    bps = pkv.choose_kv_blocks_per_split(w.num_seqs, w.num_kv_heads, w.q_len, maxb)
    ws = torch.empty(max(pkv.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    pkv.paged_attention(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], w.q_len,
                        w.scale, kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("hkv", KV_HEADS)
@pytest.mark.parametrize("shape", ["few_rows", "many_rows", "chunk"])
def test_bf16_paths(hkv, shape):
    """few_rows: the CTA-per-row decode with splits; many_rows: at least 2
    (request, KV head) rows per SM, the persistent tensor-core decode;
    chunk: q_len 16 on the tensor-core chunk kernel."""
    rng = np.random.default_rng(100 + hkv)
    q_len = 1
    if shape == "few_rows":
        ctx = [1, 17, 300, 2049, 700, 0, 128]
    elif shape == "many_rows":
        b = -(-320 // hkv)
        ctx = rng.integers(1, 400, size=b)
    else:
        q_len = 16
        ctx = [16, 40, 333, 1000, 17]
    w = W.build("heads", ctx, _blocks(ctx) + 24, q_len=q_len, seed=200 + hkv, num_kv_heads=hkv)
    assert w.num_kv_heads == hkv and w.num_q_heads == 4 * hkv
    out = _bf16_step(w)
    assert_close(bf16_to_f64(out), oracle.run_workload(w), what=f"{shape} with {hkv} KV heads")


@pytest.mark.parametrize("hkv", KV_HEADS)
def test_cascade(hkv):
    ctx = [130, 200, 129, 140, 300, 50, 77, 16]
    sharers = [True, True, True, True, True, False, False, False]
    w = W.build("heads-casc", ctx, 140, seed=300 + hkv, shared_prefix_blocks=8, sharers=sharers, num_kv_heads=hkv)
    gs, gb, sp = W.prefix_groups(w)
    d = to_device(w)
    pkv.kv_append(d["k_cache"], d["v_cache"], d["slot_mapping"], d["k_new"], d["v_new"])
    maxp = int(gb.max())
    maxs = W.max_suffix_blocks(w, sp)
    pbps, sbps = pkv.cascade_plan(w.num_seqs, w.num_kv_heads, gs.shape[0], maxp, maxs)
    ws = torch.empty(max(1, pkv.cascade_workspace_size(w.num_seqs, w.num_q_heads, maxp, maxs, pbps, sbps)),
                     dtype=torch.uint8, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    pkv.paged_attention_cascade(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                                w.scale, dev(gs), dev(gb), dev(sp), maxp, maxs, ws, pbps, sbps)
    torch.cuda.synchronize()
    assert_close(bf16_to_f64(out), oracle.run_workload(w), what=f"cascade with {hkv} KV heads")


def _tokens_of_pool(pool: np.ndarray) -> np.ndarray:
    nb, h, bs, d = pool.shape
    return np.ascontiguousarray(pool.transpose(0, 2, 1, 3).reshape(nb * bs, h, d))


@pytest.mark.parametrize("hkv", KV_HEADS)
@pytest.mark.parametrize("fmt", ["q8_0", "fp8_e4m3"])
def test_quantised_paths(hkv, fmt):
    """The fused append + decode of each quantised format: pools bit-exact
    against the oracle's append, output within tolerance of FP64 attention
    over the stored values."""
    ctx = np.asarray([17, 300, 1, 700, 0, 2049, 128, 45])
    w = W.build("heads-" + fmt, ctx, _blocks(ctx) + 24, seed=400 + hkv, num_kv_heads=hkv)
    nb = w.k_cache.shape[0]
    q8 = fmt == "q8_0"
    if q8:
        kq = np.zeros((nb, hkv, oracle.Q8_TILE_BYTES), np.uint8)
        append, deq = oracle.kv_append_q8_0, oracle.dequantize_q8_0
    else:
        kq = np.zeros((nb, hkv, 16, 128), np.uint8)
        append, deq = oracle.kv_append_fp8, oracle.dequantize_fp8
    vq = np.zeros_like(kq)
    append(kq, vq, np.arange(nb * 16, dtype=np.int64), _tokens_of_pool(w.k_cache), _tokens_of_pool(w.v_cache))
    d = to_device(w)
    kd, vd = torch.from_numpy(kq).cuda(), torch.from_numpy(vq).cuda()
    maxb = w.max_blocks_per_seq
    choose = pkv.choose_kv_blocks_per_split_q8_0 if q8 else pkv.choose_kv_blocks_per_split_fp8_e4m3
    bps = choose(w.num_seqs, w.num_kv_heads, maxb)
    ws = torch.empty(max(pkv.workspace_size_q8_0(w.num_seqs, w.num_q_heads, maxb, bps), 256), dtype=torch.uint8,
                     device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    call = pkv.paged_attention_q8_0_append if q8 else pkv.paged_attention_fp8_e4m3_append
    call(out, d["q"], kd, vd, d["block_tables"], d["context_lens"], w.scale, d["slot_mapping"], d["k_new"],
         d["v_new"], kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    append(kq, vq, w.slot_mapping, w.k_new, w.v_new)
    assert np.array_equal(kd.cpu().numpy(), kq) and np.array_equal(vd.cpu().numpy(), vq), \
        f"{fmt} with {hkv} KV heads: pools differ from the oracle's append"
    ref = oracle.paged_attention_f64(w.q, deq(kq), deq(vq), w.block_tables, w.context_lens, 1, w.scale)
    assert_close(bf16_to_f64(out), ref, what=f"{fmt} with {hkv} KV heads")
