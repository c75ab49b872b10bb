"""The benchmark workloads at full size, in the launch configuration the
benchmark times (library split heuristic), against the FP64 oracle: every
request where the oracle is quick, sampled requests elsewhere."""
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


def gpu_step(w, d, bps=0):
    pkv.kv_append(d["k_cache"], d["v_cache"], d["slot_mapping"], d["k_new"], d["v_new"])
    maxb = w.max_blocks_per_seq
    if bps == 0:
        bps = pkv.choose_kv_blocks_per_split(w.num_seqs, w.num_kv_heads, w.q_len, maxb)
    ws = torch.empty(max(1, pkv.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, maxb, bps)), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_attention(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], w.q_len,
                        w.scale, kv_blocks_per_split=bps, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error(reset=True) == 0
    return out


def compact_host_pools(w, d_k, d_v, seq_ids):
    """Copy the blocks the sampled requests read (after the step's append,
    which the oracle re-applies) into a small host pool, with remapped tables."""
    need = {}
    for r in seq_ids:
        n = -(-int(w.context_lens[r]) // 16)
        for b in w.block_tables[r, :n]:
            need.setdefault(int(b), len(need))
    ids = torch.tensor(sorted(need, key=need.get), dtype=torch.long, device="cuda")
    kc = d_k.index_select(0, ids).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    vc = d_v.index_select(0, ids).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    remap = np.vectorize(lambda b: need.get(int(b), 0))
    tables = remap(w.block_tables[seq_ids]).astype(np.int32)
    return kc, vc, tables


def check_sampled(w, d_pre_k, d_pre_v, out, seq_ids):
    """d_pre_*: device pools BEFORE the step's append."""
    kc, vc, tables = compact_host_pools(w, d_pre_k, d_pre_v, seq_ids)
    # re-express the new tokens' slots in the compact pool
    need_map = {}
    for r in seq_ids:
        n = -(-int(w.context_lens[r]) // 16)
        for b in w.block_tables[r, :n]:
            need_map.setdefault(int(b), len(need_map))
    sl = w.slot_mapping.reshape(w.num_seqs, w.q_len)[seq_ids].reshape(-1)
    sl = np.array([need_map[int(s) // 16] * 16 + int(s) % 16 if s >= 0 else -1 for s in sl], np.int64)
    kn = w.k_new.reshape(w.num_seqs, w.q_len, w.num_kv_heads, 128)[seq_ids].reshape(-1, w.num_kv_heads, 128)
    vn = w.v_new.reshape(w.num_seqs, w.q_len, w.num_kv_heads, 128)[seq_ids].reshape(-1, w.num_kv_heads, 128)
    oracle.kv_append(kc, vc, sl, kn, vn)
    ref = oracle.paged_attention(w.q[seq_ids], kc, vc, tables, w.context_lens[seq_ids], w.q_len, w.scale)
    assert_close(bf16_to_f64(out[torch.as_tensor(seq_ids, device="cuda")]), ref, what=w.name)


def _device_pools(w, seed):
    shape = (w.num_blocks, w.num_kv_heads, 16, 128)
    k = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    W.fill_pool_device(k, seed * 2 + 1)
    W.fill_pool_device(v, seed * 2 + 2)
    return k, v


@pytest.mark.parametrize("name", ["short", "long_shared", "mixed"])
def test_decode_configs_full_size_all_requests(name):
    maker = {"short": W.short_chat, "long_shared": W.long_shared, "mixed": W.mixed}[name]
    w = maker(seed=0)
    d = to_device(w)
    out = gpu_step(w, d)
    assert_close(bf16_to_f64(out), oracle.run_workload(w), what=name)


def test_chunk_config_full_size_sampled():
    w = W.chunk(seed=0, fill_cache=False)
    d = to_device(w)
    d["k_cache"], d["v_cache"] = _device_pools(w, 0)
    pre_k, pre_v = d["k_cache"].clone(), d["v_cache"].clone()
    out = gpu_step(w, d)
    order = np.argsort(w.context_lens)
    seq_ids = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 7, 64})
    check_sampled(w, pre_k, pre_v, out, seq_ids)
    del pre_k, pre_v


@pytest.mark.parametrize("b,ctx", [(1, 65536), (2, 32768), (512, 128), (64, 2048), (16, 8192), (256, 1024)])
def test_sweep_points(b, ctx):
    w = W.sweep_point(b, ctx, seed=1, fill_cache=False)
    d = to_device(w)
    d["k_cache"], d["v_cache"] = _device_pools(w, 1)
    pre_k, pre_v = d["k_cache"].clone(), d["v_cache"].clone()
    out = gpu_step(w, d)
    if b * ctx <= (1 << 21):
        seq_ids = list(range(b)) if b <= 64 else list(range(0, b, b // 32))
    else:
        seq_ids = [0, b - 1]
    check_sampled(w, pre_k, pre_v, out, seq_ids)
