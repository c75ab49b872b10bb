"""pkv_decode_graph_*: a decode step of several layers (per layer: append the
step's new tokens, then attention) captured as one CUDA graph per buffer set.
The graphs run the very kernels of the direct calls, so after the same
sequence of steps -- buffer set 0, set 1, set 0 again -- their outputs and the
layers' pools must equal the direct calls' bit for bit, for every KV format,
the cascade and a query chunk."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_decode_attention_gb300 as pkv
else:  # collected on CPU-only machines, every test skipped
    pkv = None

LAYERS = 3


@pytest.fixture(autouse=True)
def _clear_device_error():
    if pkv is not None:
        pkv.get_device_error(reset=True)
    yield
    if pkv is not None:
        assert pkv.get_device_error(reset=True) == 0


def _dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a).view(torch.bfloat16).cuda()


def _buffer_set(w, rng, cascade):
    """One step's buffers: per-layer queries and new K/V; slots, tables and lengths shared by the layers."""
    b, ql, hq, hkv, t = w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, w.slot_mapping.size
    st = {
        "q": _dev_bf16(W.randn_bf16(rng, (LAYERS, b, ql, hq, 128))),
        "k_new": _dev_bf16(W.randn_bf16(rng, (LAYERS, t, hkv, 128))),
        "v_new": _dev_bf16(W.randn_bf16(rng, (LAYERS, t, hkv, 128))),
        "slot_mapping": torch.from_numpy(w.slot_mapping).cuda(),
        "block_tables": torch.from_numpy(w.block_tables).cuda(),
        "context_lens": torch.from_numpy(w.context_lens).cuda(),
        "out": torch.full((LAYERS, b, ql, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda"),
    }
    if cascade is not None:
        gs, gb, sp = cascade
        st.update(group_seqs=torch.from_numpy(gs).cuda(), group_blocks=torch.from_numpy(gb).cuda(),
                  seq_prefix_blocks=torch.from_numpy(sp).cuda())
    return st


def _pools(fmt, w, seed):
    """Per-layer K and V pools of the format, every slot holding seeded values."""
    nb, hkv = w.num_blocks, w.num_kv_heads
    if fmt == pkv.KV_BF16:
        k = torch.empty((LAYERS, nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        for l in range(LAYERS):
            W.fill_pool_device(k[l], seed + 2 * l)
            W.fill_pool_device(v[l], seed + 2 * l + 1)
        return k, v
    tile = (pkv.Q8_TILE_BYTES,) if fmt == pkv.KV_Q8_0 else (16, 128)
    k = torch.empty((LAYERS, nb, hkv) + tile, dtype=torch.uint8, device="cuda")
    v = torch.empty_like(k)
    tmp_k = torch.empty((nb, hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    tmp_v = torch.empty_like(tmp_k)
    slots = torch.arange(nb * 16, dtype=torch.int64, device="cuda")
    tok = lambda p: p.permute(0, 2, 1, 3).contiguous().view(nb * 16, hkv, 128)
    append = pkv.kv_append_q8_0 if fmt == pkv.KV_Q8_0 else pkv.kv_append_fp8_e4m3
    for l in range(LAYERS):
        W.fill_pool_device(tmp_k, seed + 2 * l)
        W.fill_pool_device(tmp_v, seed + 2 * l + 1)
        append(k[l], v[l], slots, tok(tmp_k), tok(tmp_v))
    return k, v


def _direct_step(fmt, kp, vp, st, w, bps, ws, cascade):
    """The step through the direct calls, layer by layer."""
    append = {pkv.KV_BF16: pkv.kv_append, pkv.KV_Q8_0: pkv.kv_append_q8_0,
              pkv.KV_FP8_E4M3: pkv.kv_append_fp8_e4m3}[fmt]
    for l in range(LAYERS):
        append(kp[l], vp[l], st["slot_mapping"], st["k_new"][l], st["v_new"][l])
        q, out = st["q"][l], st["out"][l]
        if fmt == pkv.KV_BF16 and cascade is not None:
            pkv.paged_attention_cascade(out, q, kp[l], vp[l], st["block_tables"], st["context_lens"], w.scale,
                                        st["group_seqs"], st["group_blocks"], st["seq_prefix_blocks"],
                                        cascade["max_prefix_blocks"], cascade["max_suffix_blocks"], ws)
        elif fmt == pkv.KV_BF16:
            pkv.paged_attention(out, q, kp[l], vp[l], st["block_tables"], st["context_lens"], w.q_len, w.scale,
                                kv_blocks_per_split=bps, workspace=ws)
        elif fmt == pkv.KV_Q8_0:
            pkv.paged_attention_q8_0(out, q, kp[l], vp[l], st["block_tables"], st["context_lens"], w.scale,
                                     kv_blocks_per_split=bps, workspace=ws)
        else:
            pkv.paged_attention_fp8_e4m3(out, q, kp[l], vp[l], st["block_tables"], st["context_lens"], w.scale,
                                         kv_blocks_per_split=bps, workspace=ws)


CASES = {
    "bf16": dict(fmt=0, ctx=[37, 300, 129, 16, 700, 1, 0, 2049], bps=0),
    "bf16_split_workspace": dict(fmt=0, ctx=[37, 300, 129, 16, 700, 1, 0, 2049], bps=5),
    "bf16_chunk": dict(fmt=0, ctx=[40, 300, 129, 16, 700, 17], bps=0, q_len=16),
    "bf16_q_len_4": dict(fmt=0, ctx=[40, 300, 129, 16, 700, 17], bps=0, q_len=4),
    "cascade": dict(fmt=0, ctx=[130, 200, 129, 140, 300, 50, 77, 16], bps=0, prefix=8,
                    sharers=[True] * 5 + [False] * 3),
    "q8_0": dict(fmt=1, ctx=[37, 300, 129, 16, 700, 1, 0, 2049], bps=0),
    "fp8_e4m3": dict(fmt=2, ctx=[37, 300, 129, 16, 700, 1, 0, 2049], bps=0),
}


@pytest.mark.parametrize("case", list(CASES))
def test_graph_equals_direct_calls_on_both_buffer_sets(case):
    c = CASES[case]
    fmt, ql = c["fmt"], c.get("q_len", 1)
    ctx = np.asarray(c["ctx"]) + (ql if ql > 1 else 0)
    need = int(sum(-(-int(x) // 16) for x in ctx))
    w = W.build(case, ctx, need + 24, q_len=ql, seed=31, fill_cache=False,
                shared_prefix_blocks=c.get("prefix", 0), sharers=c.get("sharers"))
    b, hq, maxb = w.num_seqs, w.num_q_heads, w.max_blocks_per_seq
    casc_arrays = casc = None
    if "prefix" in c:
        casc_arrays = W.prefix_groups(w)
        casc = {"num_groups": int(casc_arrays[0].shape[0]), "max_prefix_blocks": int(casc_arrays[1].max()),
                "max_suffix_blocks": W.max_suffix_blocks(w, casc_arrays[2])}
        pb, sb = pkv.cascade_plan(b, w.num_kv_heads, casc["num_groups"], casc["max_prefix_blocks"],
                                  casc["max_suffix_blocks"])
        ws_bytes = pkv.cascade_workspace_size(b, hq, casc["max_prefix_blocks"], casc["max_suffix_blocks"], pb, sb)
        bps = 0
    elif fmt == pkv.KV_BF16:
        bps = c["bps"] or pkv.choose_kv_blocks_per_split(b, w.num_kv_heads, ql, maxb)
        ws_bytes = pkv.workspace_size(b, ql, hq, maxb, bps)
    else:
        choose = pkv.choose_kv_blocks_per_split_q8_0 if fmt == pkv.KV_Q8_0 else pkv.choose_kv_blocks_per_split_fp8_e4m3
        bps = choose(b, w.num_kv_heads, maxb)
        ws_bytes = pkv.workspace_size_q8_0(b, hq, maxb, bps)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")

    rng = np.random.default_rng(77)
    sets = [_buffer_set(w, rng, casc_arrays) for _ in range(2)]
    kp, vp = _pools(fmt, w, seed=900)
    kp_d, vp_d = kp.clone(), vp.clone()
    desc = pkv.CacheDesc(w.num_blocks, 16, w.num_kv_heads, 128)
    g = pkv.DecodeGraph(list(kp), list(vp), desc, sets, num_seqs=b, q_len=ql, num_q_heads=hq,
                        max_blocks_per_seq=maxb, num_tokens=int(w.slot_mapping.size), scale=w.scale, kv_format=fmt,
                        kv_blocks_per_split=bps, workspace=ws, cascade=casc)
    for s in (0, 1, 0):
        g.launch(s)
    torch.cuda.synchronize()
    g.close()

    sets_d = [dict(st, out=torch.full_like(st["out"], float("nan"))) for st in sets]
    for s in (0, 1, 0):
        _direct_step(fmt, kp_d, vp_d, sets_d[s], w, bps, ws, casc)
    torch.cuda.synchronize()
    for s in (0, 1):
        got, ref = sets[s]["out"].view(torch.int16), sets_d[s]["out"].view(torch.int16)
        assert torch.equal(got, ref), f"{case}: buffer set {s} differs from the direct calls"
        assert torch.isfinite(sets[s]["out"].float()).all()
    assert torch.equal(kp, kp_d) and torch.equal(vp, vp_d), f"{case}: pools differ after the appends"
