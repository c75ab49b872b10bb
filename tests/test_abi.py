"""The C ABI on the host: the library builds and loads, exports every
function include/pkv.h declares, and rejects bad arguments with the
documented status before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import paged_kv_decode_attention_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(pkv_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert {"pkv_kv_append", "pkv_paged_attention", "pkv_attn_combine", "pkv_workspace_size"} <= set(names)
    lib = ctypes.CDLL(pkv.library_path())
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings():
    lib = pkv.lib()
    for code in range(7):
        assert lib.pkv_status_string(code).startswith(b"PKV_")


def test_workspace_size_and_split_heuristic_are_host_arithmetic():
    lib = pkv.lib()
    # no split -> no workspace
    assert lib.pkv_workspace_size(37, 1, 32, 128, 144, 144) == 0
    # up to 8 splits merge inside a thread-block cluster: no workspace
    assert lib.pkv_workspace_size(37, 1, 32, 128, 144, 48) == 0
    assert lib.pkv_workspace_size(37, 1, 32, 128, 144, 18) == 0
    rows, splits = 37 * 32, 9
    need = lib.pkv_workspace_size(37, 1, 32, 128, 144, 16)
    o_bytes = -(-rows * splits * 128 * 4 // 256) * 256
    l_bytes = -(-rows * splits * 4 // 256) * 256
    assert need == o_bytes + l_bytes
    # a full GPU needs no split; a small batch over a long context does
    assert lib.pkv_choose_kv_blocks_per_split(512, 8, 1, 144, 152) == 144
    bps = lib.pkv_choose_kv_blocks_per_split(4, 8, 1, 528, 152)
    assert 16 <= bps < 528
    assert lib.pkv_choose_kv_blocks_per_split(1, 8, 1, 8, 152) == 8
    # the split never goes below 16 blocks
    assert lib.pkv_choose_kv_blocks_per_split(1, 1, 1, 4096, 152) >= 16
    # 24 requests (192 rows) would fill 192 of the CTA-per-row kernel's 304 slots: the persistent
    # tensor-core kernel takes them, split by its makespan model in 8-block tiles (3 x 48 blocks)
    assert lib.pkv_choose_kv_blocks_per_split(24, 8, 1, 144, 152) == 48
    # 37 requests fill 296 of 304 slots: CTA-per-row, no split; short requests stay there too
    assert lib.pkv_choose_kv_blocks_per_split(37, 8, 1, 144, 152) == 144
    assert lib.pkv_choose_kv_blocks_per_split(24, 8, 1, 64, 152) == 64


def _desc(**kw):
    d = dict(num_blocks=4, block_size=16, num_kv_heads=8, head_dim=128)
    d.update(kw)
    return pkv.CacheDesc(**d)


def test_kv_append_argument_errors():
    lib = pkv.lib()
    one = ctypes.c_void_p(16)
    assert lib.pkv_kv_append(one, one, None, one, one, one, 1, None) == 1                       # NULL desc
    assert lib.pkv_kv_append(one, one, ctypes.byref(_desc(block_size=8)), one, one, one, 1, None) == 3
    assert lib.pkv_kv_append(one, one, ctypes.byref(_desc(head_dim=64)), one, one, one, 1, None) == 3
    assert lib.pkv_kv_append(one, one, ctypes.byref(_desc()), one, one, one, -1, None) == 2
    assert lib.pkv_kv_append(None, one, ctypes.byref(_desc()), one, one, one, 1, None) == 1
    assert lib.pkv_kv_append(one, one, ctypes.byref(_desc()), one, one, one, 0, None) == 0      # nothing to do


def test_paged_attention_argument_errors():
    lib = pkv.lib()
    p = ctypes.c_void_p(256)
    d = ctypes.byref(_desc())
    args = lambda **kw: dict(dict(out=p, q=p, k=p, v=p, desc=d, bt=p, maxb=4, cl=p, b=2, ql=1, hq=32, scale=0.1,
                                  bps=4, ws=None, wsb=0, s=None), **kw)

    def call(**kw):
        a = args(**kw)
        return lib.pkv_paged_attention(a["out"], a["q"], a["k"], a["v"], a["desc"], a["bt"], a["maxb"], a["cl"],
                                       a["b"], a["ql"], a["hq"], a["scale"], a["bps"], a["ws"], a["wsb"], a["s"])

    assert call(desc=None) == 1
    assert call(out=None) == 1
    assert call(ql=0) == 2
    assert call(maxb=0) == 2
    assert call(b=-1) == 2
    assert call(hq=16) == 3                        # not 4 query heads per KV head
    assert call(desc=ctypes.byref(_desc(block_size=32))) == 3
    assert call(scale=float("nan")) == 2
    assert call(q=ctypes.c_void_p(258)) == 3       # misaligned
    assert call(b=0) == 0                          # empty batch: nothing enqueued


def test_attn_combine_argument_errors():
    lib = pkv.lib()
    p = ctypes.c_void_p(256)
    assert lib.pkv_attn_combine(p, None, p, p, 4, 64, 2, None) == 3
    assert lib.pkv_attn_combine(p, None, p, p, 4, 128, 0, None) == 2
    assert lib.pkv_attn_combine(None, None, p, p, 4, 128, 2, None) == 1
    assert lib.pkv_attn_combine(p, None, p, p, 0, 128, 2, None) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.kv_append(x, x, torch.zeros(1, dtype=torch.int64), torch.zeros(1, 8, 128, dtype=torch.bfloat16),
                      torch.zeros(1, 8, 128, dtype=torch.bfloat16))


def test_q8_split_heuristic_and_workspace_are_host_arithmetic():
    lib = pkv.lib()
    # 37 requests x 8 KV heads = 296 units on 152 SMs: two units per CTA, no split
    assert lib.pkv_choose_kv_blocks_per_split_q8_0(37, 8, 144, 152) == 144
    # few long rows: split into whole 8-block tiles, at least 16 blocks each
    bps = lib.pkv_choose_kv_blocks_per_split_q8_0(2, 8, 528, 152)
    assert 16 <= bps < 528 and bps % 8 == 0
    assert lib.pkv_workspace_size_q8_0(37, 32, 144, 144) == 0
    # the E4M3 kernel reads 16-block tiles: splits in whole 16-block tiles, at least 32 blocks each
    assert lib.pkv_choose_kv_blocks_per_split_fp8_e4m3(37, 8, 144, 152) == 144
    bps8 = lib.pkv_choose_kv_blocks_per_split_fp8_e4m3(2, 8, 528, 152)
    assert 32 <= bps8 < 528 and bps8 % 16 == 0
    rows, splits = 2 * 32, -(-528 // bps)
    o_bytes = -(-rows * splits * 128 * 4 // 256) * 256
    l_bytes = -(-rows * splits * 4 // 256) * 256
    assert lib.pkv_workspace_size_q8_0(2, 32, 528, bps) == o_bytes + l_bytes


def test_q8_argument_errors():
    lib = pkv.lib()
    p = ctypes.c_void_p(256)
    d = ctypes.byref(_desc())
    assert lib.pkv_kv_append_q8_0(p, p, None, p, p, p, 1, None) == 1
    assert lib.pkv_kv_append_q8_0(p, p, ctypes.byref(_desc(head_dim=64)), p, p, p, 1, None) == 3
    assert lib.pkv_kv_append_q8_0(p, p, d, p, p, p, -1, None) == 2
    assert lib.pkv_kv_append_q8_0(p, p, d, p, ctypes.c_void_p(264), p, 1, None) == 3  # k_new misaligned
    assert lib.pkv_kv_append_q8_0(p, p, d, p, p, p, 0, None) == 0

    def call(**kw):
        a = dict(out=p, q=p, k=p, v=p, desc=d, bt=p, maxb=64, cl=p, b=2, hq=32, scale=0.1, bps=16, ws=None, wsb=0)
        a.update(kw)
        return lib.pkv_paged_attention_q8_0(a["out"], a["q"], a["k"], a["v"], a["desc"], a["bt"], a["maxb"],
                                            a["cl"], a["b"], a["hq"], a["scale"], a["bps"], a["ws"], a["wsb"], None)

    assert call(desc=None) == 1
    assert call(v=None) == 1
    assert call(hq=8) == 3
    assert call(maxb=0) == 2
    assert call(scale=float("inf")) == 2
    assert call(k=ctypes.c_void_p(260)) == 3
    assert call() == 4                      # 4 splits need a workspace
    assert call(ws=ctypes.c_void_p(256), wsb=16) == 4
    assert call(b=0) == 0
    assert lib.pkv_copy_blocks_q8_0(p, p, ctypes.byref(_desc(block_size=8)), p, p, 1, None) == 3
    assert lib.pkv_copy_blocks_q8_0(p, p, d, p, p, 0, None) == 0


def test_fp8_argument_errors():
    lib = pkv.lib()
    p = ctypes.c_void_p(256)
    d = ctypes.byref(_desc())
    assert lib.pkv_kv_append_fp8_e4m3(p, p, None, p, p, p, 1, None) == 1
    assert lib.pkv_kv_append_fp8_e4m3(p, p, ctypes.byref(_desc(block_size=8)), p, p, p, 1, None) == 3
    assert lib.pkv_kv_append_fp8_e4m3(p, p, d, p, p, p, -2, None) == 2
    assert lib.pkv_kv_append_fp8_e4m3(p, p, d, p, p, p, 0, None) == 0

    def call(**kw):
        a = dict(out=p, q=p, k=p, v=p, desc=d, bt=p, maxb=64, cl=p, b=2, hq=32, scale=0.1, bps=16, ws=None, wsb=0)
        a.update(kw)
        return lib.pkv_paged_attention_fp8_e4m3(a["out"], a["q"], a["k"], a["v"], a["desc"], a["bt"], a["maxb"],
                                                a["cl"], a["b"], a["hq"], a["scale"], a["bps"], a["ws"], a["wsb"],
                                                None)

    assert call(desc=None) == 1
    assert call(hq=16) == 3
    assert call(scale=float("nan")) == 2
    assert call() == 4
    assert call(b=0) == 0
    assert lib.pkv_copy_blocks_fp8_e4m3(p, p, d, p, p, 0, None) == 0


def test_decode_graph_argument_errors():
    """pkv_decode_graph_create checks its description on the host and returns
    before any CUDA call; launch and destroy reject a NULL graph."""
    lib = pkv.lib()
    h = ctypes.c_void_p()
    d = pkv.DecodeGraphDesc()
    assert lib.pkv_decode_graph_create(None, ctypes.byref(h)) == 1
    assert lib.pkv_decode_graph_create(ctypes.byref(d), None) == 1
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 2  # no layers
    d.num_layers, d.q_len, d.num_q_heads, d.num_seqs, d.num_tokens = 2, 1, 32, 4, 4
    d.cache = _desc()
    d.kv_format = 7
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 3
    d.kv_format, d.q_len = pkv.KV_Q8_0, 2  # quantised pools: decode only
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 3
    d.kv_format, d.q_len, d.num_groups = pkv.KV_FP8_E4M3, 1, 1  # no cascade over quantised pools
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 3
    d.kv_format, d.num_groups = pkv.KV_BF16, 0
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 1  # no pool arrays
    fake = (ctypes.c_void_p * 2)(4096, 0)
    d.k_caches = d.v_caches = ctypes.cast(fake, ctypes.POINTER(ctypes.c_void_p))
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 1  # layer 1 has no pool
    fake[1] = 8192
    assert lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)) == 1  # buffer sets unset
    assert not h.value
    assert lib.pkv_decode_graph_launch(None, 0, None) == 1
    lib.pkv_decode_graph_destroy(None)


def test_paged_attention_append_argument_errors():
    """The fused call checks its own arguments on the host before anything
    else (no CUDA call on these paths)."""
    f = pkv.lib().pkv_paged_attention_append
    d = _desc()
    # no cache descriptor; a negative token count; new tokens without their K
    assert f(None, None, None, None, None, None, 1, None, 1, 1, 32, 1.0, 0, None, 0, None, None, None, 0, None) == 1
    assert f(None, None, None, None, ctypes.byref(d), None, 1, None, 1, 1, 32, 1.0, 0, None, 0, None, None, None, -1,
             None) == 2
    assert f(None, None, 4096, 4096, ctypes.byref(d), None, 1, None, 1, 1, 32, 1.0, 0, None, 0, 4096, None, 4096, 1,
             None) == 1
    assert f(None, None, 4096, 4096, ctypes.byref(d), None, 1, None, 1, 1, 32, 1.0, 0, None, 0, 4096, 4100, 4096, 1,
             None) == 3  # k_new not 16-byte aligned


@pytest.mark.parametrize("name", ["pkv_paged_attention_fp8_e4m3_append", "pkv_paged_attention_q8_0_append"])
def test_paged_attention_quantised_append_argument_errors(name):
    """The E4M3 and q8_0 append-and-attention calls check their own arguments
    on the host before anything else (no CUDA call on these paths)."""
    f = getattr(pkv.lib(), name)
    d = _desc()
    # no cache descriptor; a negative token count; new tokens without their K; a misaligned K
    assert f(None, None, None, None, None, None, 1, None, 1, 32, 1.0, 0, None, 0, None, None, None, 0, None) == 1
    assert f(None, None, None, None, ctypes.byref(d), None, 1, None, 1, 32, 1.0, 0, None, 0, None, None, None, -1,
             None) == 2
    assert f(None, None, 4096, 4096, ctypes.byref(d), None, 1, None, 1, 32, 1.0, 0, None, 0, 4096, None, 4096, 1,
             None) == 1
    assert f(None, None, 4096, 4096, ctypes.byref(d), None, 1, None, 1, 32, 1.0, 0, None, 0, 4096, 4100, 4096, 1,
             None) == 3
    # the attention's own checks run before anything is enqueued: no query
    assert f(None, None, 4096, 4096, ctypes.byref(d), 4096, 1, 4096, 1, 32, 1.0, 0, None, 0, 4096, 4096, 4096, 1,
             None) == 1


def test_selftest_bounded_wait_rejects_limits_outside_its_range():
    lib = pkv.lib()
    assert lib.pkv_selftest_bounded_wait(0, 0, None) == 2
    assert lib.pkv_selftest_bounded_wait(1000001, 0, None) == 2
