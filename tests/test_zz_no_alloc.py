"""pkv_paged_attention_static_workspace: the attention entry point for
callers that cannot allocate device memory (code inside a memory manager or
an allocation hook, frameworks that forbid allocation on the hot path, plain
C callers without a CUDA allocator).  It keeps split-KV partials in a scratch
array compiled into the library.

Checked here through the C ABI on three calls in a row, each split into more
than 8 ranges so that its partials really go through the array (fewer ranges
merge on chip and leave it untouched).  The second call has the first call's
shape but other context lengths, so rows that now have fewer ranges sit next
to stale partials of the first call; the third has another shape.  Every call
is compared with the ordinary entry point (which takes a caller workspace)
and with the FP64 oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, to_device

pytestmark = pytest.mark.gpu

PKV_ERR_WORKSPACE = 4


def _static_entry():
    import paged_kv_decode_attention_gb300 as pkv
    lib = ctypes.CDLL(pkv.library_path())
    f = lib.pkv_paged_attention_static_workspace
    p, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [p, p, p, p, ctypes.POINTER(pkv.CacheDesc), p, i32, p, i32, i32, i32, ctypes.c_float, i32, p]
    f.restype = ctypes.c_int
    return pkv, f


def _call_static(pkv, f, w, d, out, bps):
    desc = pkv.CacheDesc(w.num_blocks, 16, w.num_kv_heads, 128)
    return f(out.data_ptr(), d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
             ctypes.byref(desc), d["block_tables"].data_ptr(), w.max_blocks_per_seq, d["context_lens"].data_ptr(),
             w.num_seqs, w.q_len, w.num_q_heads, w.scale, bps, torch.cuda.current_stream().cuda_stream)


def _reference(pkv, w, d, bps):
    ws_bytes = pkv.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, w.max_blocks_per_seq, bps)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_attention(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], w.q_len,
                        w.scale, kv_blocks_per_split=bps, workspace=ws)
    return out


def test_static_workspace_entry_matches_workspace_entry_and_oracle_on_consecutive_calls():
    pkv, f = _static_entry()
    cases = [
        (W.build("first", [2300, 17, 700, 1, 0, 4100], 800, seed=21, max_blocks=257), 8),
        (W.build("second", [40, 4000, 1, 0, 2000, 300], 800, seed=24, max_blocks=257), 8),
        (W.build("third", [5, 300, 64, 1999], 400, q_len=3, seed=22), 10),
    ]
    for w, bps in cases:
        # more than 8 ranges: the partials go through the scratch array
        assert -(-w.max_blocks_per_seq // bps) > 8
        assert pkv.workspace_size(w.num_seqs, w.q_len, w.num_q_heads, w.max_blocks_per_seq, bps) > 0
        d = to_device(w)
        pkv.kv_append(d["k_cache"], d["v_cache"], d["slot_mapping"], d["k_new"], d["v_new"])
        out = torch.full_like(d["q"], float("nan"))
        st = _call_static(pkv, f, w, d, out, bps)
        assert st == 0, pkv.lib().pkv_status_string(st)
        ref = _reference(pkv, w, d, bps)
        torch.cuda.synchronize()
        got = bf16_to_f64(out)
        assert_close(got, bf16_to_f64(ref), what=f"static workspace vs workspace entry, {w.name}")
        assert_close(got, oracle.run_workload(w), what=f"static workspace vs oracle, {w.name}")
        assert not got[w.context_lens == 0].any(), f"{w.name}: padding rows must be zero"
    assert pkv.get_device_error(reset=True) == 0


def test_static_workspace_entry_rejects_requests_beyond_its_scratch():
    pkv, f = _static_entry()
    w = W.build("big", [16 * 528] * 64, 64 * 528 + 8, seed=23, fill_cache=False)
    need = pkv.workspace_size(w.num_seqs, 1, 32, w.max_blocks_per_seq, 1)
    assert need > (16 << 20)
    q = torch.zeros((w.num_seqs, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    d = {"q": q, "k_cache": cache, "v_cache": cache,
         "block_tables": torch.zeros((w.num_seqs, w.max_blocks_per_seq), dtype=torch.int32, device="cuda"),
         "context_lens": torch.zeros(w.num_seqs, dtype=torch.int32, device="cuda")}
    w.num_blocks = 1
    out = torch.zeros_like(q)
    assert _call_static(pkv, f, w, d, out, 1) == PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not out.any()
