"""pkv_decode_graph_*: a decode step of several layers (per layer: append the
step's new tokens, then attention) captured as one CUDA graph per buffer set.
After the same sequence of steps -- buffer set 0, set 1, set 0 again -- the
graphs' outputs and the layers' pools must
  * equal the direct calls' bit for bit (the graphs run the very kernels of
    the direct calls), and
  * match the FP64 oracle replaying the same steps on host copies: pools
    bit-exact (the oracle's append, BF16 / q8_0 / E4M3), every layer's output
    of both buffer sets within the attention tolerance,
for every KV format, the cascade and query chunks."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close

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
    """One step's buffers: per-layer queries and new K/V; slots, tables and lengths shared by the layers.
    Returns (device buffers, host copies of the per-layer values)."""
    b, ql, hq, hkv, t = w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, w.slot_mapping.size
    host = {
        "q": W.randn_bf16(rng, (LAYERS, b, ql, hq, 128)),
        "k_new": W.randn_bf16(rng, (LAYERS, t, hkv, 128)),
        "v_new": W.randn_bf16(rng, (LAYERS, t, hkv, 128)),
    }
    st = {
        "q": _dev_bf16(host["q"]),
        "k_new": _dev_bf16(host["k_new"]),
        "v_new": _dev_bf16(host["v_new"]),
        "slot_mapping": torch.from_numpy(w.slot_mapping).cuda(),
        "block_tables": torch.from_numpy(w.block_tables).cuda(),
        "context_lens": torch.from_numpy(w.context_lens).cuda(),
        "out": torch.full((LAYERS, b, ql, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda"),
    }
    if cascade is not None:
        gs, gb, sp = cascade
        st.update(group_seqs=torch.from_numpy(gs).cuda(), group_blocks=torch.from_numpy(gb).cuda(),
                  seq_prefix_blocks=torch.from_numpy(sp).cuda())
    return st, host


def _host_pools(fmt, w, seed):
    """Per-layer K and V pools of the format, every slot holding seeded N(0,1)
    values; the quantised formats are stored by the oracle's append.  Host
    arrays, uploaded by the caller."""
    nb, hkv = w.num_blocks, w.num_kv_heads
    rng = np.random.default_rng(seed)
    ks, vs = [], []
    for _ in range(LAYERS):
        kb = W.randn_bf16(rng, (nb, hkv, 16, 128))
        vb = W.randn_bf16(rng, (nb, hkv, 16, 128))
        if fmt == pkv.KV_BF16:
            ks.append(kb)
            vs.append(vb)
            continue
        tok = lambda p: np.ascontiguousarray(p.transpose(0, 2, 1, 3).reshape(nb * 16, hkv, 128))
        slots = np.arange(nb * 16, dtype=np.int64)
        if fmt == pkv.KV_Q8_0:
            kq = np.zeros((nb, hkv, oracle.Q8_TILE_BYTES), np.uint8)
            vq = np.zeros_like(kq)
            oracle.kv_append_q8_0(kq, vq, slots, tok(kb), tok(vb))
        else:
            kq = np.zeros((nb, hkv, 16, 128), np.uint8)
            vq = np.zeros_like(kq)
            oracle.kv_append_fp8(kq, vq, slots, tok(kb), tok(vb))
        ks.append(kq)
        vs.append(vq)
    return np.stack(ks), np.stack(vs)


def _upload_pools(fmt, kh, vh):
    if fmt == pkv.KV_BF16:
        return _dev_bf16(kh), _dev_bf16(vh)
    return torch.from_numpy(kh).cuda(), torch.from_numpy(vh).cuda()


def _oracle_step(fmt, kh, vh, host, w):
    """The step on the host with the oracle: per layer the append, then the
    attention (FP64; over the stored values for the quantised formats).
    Updates the host pools in place; returns float64 [LAYERS][B][q_len][Hq][D]."""
    outs = []
    for l in range(LAYERS):
        if fmt == pkv.KV_BF16:
            oracle.kv_append(kh[l], vh[l], w.slot_mapping, host["k_new"][l], host["v_new"][l])
            outs.append(oracle.paged_attention(host["q"][l], kh[l], vh[l], w.block_tables, w.context_lens, w.q_len,
                                               w.scale))
            continue
        if fmt == pkv.KV_Q8_0:
            oracle.kv_append_q8_0(kh[l], vh[l], w.slot_mapping, host["k_new"][l], host["v_new"][l])
            kd, vd = oracle.dequantize_q8_0(kh[l]), oracle.dequantize_q8_0(vh[l])
        else:
            oracle.kv_append_fp8(kh[l], vh[l], w.slot_mapping, host["k_new"][l], host["v_new"][l])
            kd, vd = oracle.dequantize_fp8(kh[l]), oracle.dequantize_fp8(vh[l])
        outs.append(oracle.paged_attention_f64(host["q"][l], kd, vd, w.block_tables, w.context_lens, w.q_len,
                                               w.scale))
    return np.stack(outs)


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
def test_graph_equals_direct_calls_and_oracle_on_both_buffer_sets(case):
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
    sets, hosts = zip(*[_buffer_set(w, rng, casc_arrays) for _ in range(2)])
    sets = list(sets)
    kh, vh = _host_pools(fmt, w, seed=900)
    kp, vp = _upload_pools(fmt, kh, vh)
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

    # the same three steps on the host with the oracle
    expect = {}
    for s in (0, 1, 0):
        expect[s] = _oracle_step(fmt, kh, vh, hosts[s], w)
    for s in (0, 1):
        got = sets[s]["out"].float().cpu().numpy().astype(np.float64)
        for l in range(LAYERS):
            assert_close(got[l], expect[s][l], what=f"{case}: buffer set {s}, layer {l} vs oracle")
    if fmt == pkv.KV_BF16:
        kg, vg = kp.view(torch.int16).cpu().numpy().view(np.uint16), vp.view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        kg, vg = kp.cpu().numpy(), vp.cpu().numpy()
    assert np.array_equal(kg, kh) and np.array_equal(vg, vh), f"{case}: pools differ from the oracle's appends"
