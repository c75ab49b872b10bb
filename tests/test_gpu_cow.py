"""Copy-on-write on the device: pkv_copy_blocks is a bit copy, and two
branches that share a partly filled tail block (web textbook page "Chapter
8: Inference Optimization", §8.3.2 / Fig. 8-15) each append their own token
into a private copy, after which attention over each branch equals the FP64
oracle on the same operations."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, dev

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_decode_attention_gb300 as pkv
else:
    pkv = None


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_copy_blocks_bit_exact():
    rng = np.random.default_rng(60)
    kc = W.randn_bf16(rng, (40, 8, 16, 128))
    vc = W.randn_bf16(rng, (40, 8, 16, 128))
    src = np.array([3, 7, 11, 0], np.int32)
    dst = np.array([20, 21, 39, 5], np.int32)
    dk, dv = dev(kc), dev(vc)
    pkv.copy_blocks(dk, dv, dev(src), dev(dst))
    oracle.copy_blocks(kc, vc, src, dst)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(dk), kc) and np.array_equal(_u16(dv), vc)
    assert pkv.get_device_error(reset=True) == 0


def test_two_branches_append_into_private_copies_of_a_shared_tail():
    rng = np.random.default_rng(61)
    nb, ctx0 = 64, 40                          # common context: 2 full blocks + 8 tokens in a shared tail
    kc = W.randn_bf16(rng, (nb, 8, 16, 128))
    vc = W.randn_bf16(rng, (nb, 8, 16, 128))
    pool = pkv.BlockPool(nb, 16)
    base = []
    pool.reserve(base, 0, ctx0, 8)
    a, b = list(base), list(base)
    pool.share(base)
    copies = []
    for row in (a, b):
        copies += pool.reserve(row, ctx0, 1, 8)
    assert len(copies) == 1 and a[2] != b[2] and a[:2] == b[:2]
    src = np.array([c[0] for c in copies], np.int32)
    dst = np.array([c[1] for c in copies], np.int32)
    tables = np.array([a + [0] * (8 - len(a)), b + [0] * (8 - len(b))], np.int32)
    ctx = np.array([ctx0 + 1, ctx0 + 1], np.int32)
    slots = np.array([a[ctx0 // 16] * 16 + ctx0 % 16, b[ctx0 // 16] * 16 + ctx0 % 16], np.int64)
    k_new = W.randn_bf16(rng, (2, 8, 128))
    v_new = W.randn_bf16(rng, (2, 8, 128))
    q = W.randn_bf16(rng, (2, 1, 32, 128))
    # device: copy, append, attend
    dk, dv = dev(kc), dev(vc)
    pkv.copy_blocks(dk, dv, dev(src), dev(dst))
    pkv.kv_append(dk, dv, dev(slots), dev(k_new), dev(v_new))
    out = torch.empty((2, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention(out, dev(q), dk, dv, dev(tables), dev(ctx), 1, W.SCALE, kv_blocks_per_split=8)
    torch.cuda.synchronize()
    # oracle: the same operations on host copies
    ok, ov = kc.copy(), vc.copy()
    oracle.copy_blocks(ok, ov, src, dst)
    oracle.kv_append(ok, ov, slots, k_new, v_new)
    assert np.array_equal(_u16(dk), ok) and np.array_equal(_u16(dv), ov)
    ref = oracle.paged_attention(q, ok, ov, tables, ctx, 1, W.SCALE)
    assert_close(bf16_to_f64(out), ref, what="cow branches")
    # each branch sees its own new token and the shared first 40 tokens
    assert not np.array_equal(ok[a[2], :, 8], ok[b[2], :, 8])
    assert np.array_equal(ok[a[2], :, :8], ok[b[2], :, :8])
    assert pkv.get_device_error(reset=True) == 0
