"""Pins of the q8_0 oracle (quantised KV, web textbook page "Chapter 8:
Inference Optimization", §8.4.2 and Fig. 8-23) to things other than itself:
the sizes the page prints, closed forms of the quantiser (integer groups,
power-of-two scaling, the half-way rounding rule, the error bound), the
documented byte layout of a q8_0 tile, and -- for values q8_0 stores exactly
-- agreement with the pinned BF16 attention oracle."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W
from oracle import sizes

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ch8_printed_values.json")))


def _bf16(x) -> np.ndarray:
    """Float values that are exact in BF16 -> their bit patterns."""
    a = np.asarray(x, np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), a), "value not exact in BF16"
    return bits


def _fp16_bits(v: float) -> int:
    return int(np.array([v], np.float16).view(np.uint16)[0])


# ---------------------------------------------------------------- sizes --


def test_group_bytes_fig_8_23():
    g = GOLD["q8_0"]
    assert sizes.group_bytes(g["group"], 16, scale_bytes=0) == g["bf16_group_bytes"]
    assert sizes.group_bytes(g["group"], 8) == g["q8_group_bytes"]
    assert sizes.group_bytes(g["group"], 4) == g["q4_group_bytes"]
    assert sizes.bits_per_value(8) == g["q8_bits"] and sizes.bits_per_value(4) == g["q4_bits"]
    # a (block, kv head) tile of 16 tokens x 128 dims in q8_0: 64 groups of 34 bytes
    assert 16 * 128 // g["group"] * sizes.group_bytes(g["group"], 8) == oracle.Q8_TILE_BYTES


def test_q8_capacity_printed():
    g = GOLD["q8_0"]
    assert sizes.quantized_mib(g["bf16_8k_mib"], 8) == g["q8_8k_mib"]
    assert sizes.quantized_mib(g["bf16_8k_mib"], 4) == g["q4_8k_mib"]
    assert g["bf16_8k_mib"] - g["q8_8k_mib"] == g["q8_saved_mib"]
    assert g["bf16_8k_mib"] - g["q4_8k_mib"] == g["q4_saved_mib"]
    assert sizes.quantized_mib(g["long_bf16_mib"], 8) == g["long_q8_mib"]
    assert round(g["long_requests"] * g["long_q8_mib"] / 1024, 2) == g["long_q8_gib"]
    assert g["long_requests"] * g["long_q8_mib"] <= GOLD["capacity_table"]["pool_mib"]


def test_q8_read_time_example():
    g = GOLD["q8_0_read_time"]
    saved = sizes.saved_time_s(g["saved_mib"] * sizes.MIB, g["beta_tb_s"] * 1e12, 0.0) * 1e3
    # the page rounds its bandwidth (about 65% of 1792 GB/s); its 0.487 ms is within 0.5%
    assert saved == pytest.approx(g["saved_ms"], rel=5e-3)
    for conv, net in zip(g["convert_ms"], g["net_ms"]):
        assert round(g["saved_ms"] - conv, 3) == net


def test_q8_round_bytes_combined_example():
    g = GOLD["q8_0_round_bytes"]
    rb = GOLD["read_bytes"]
    k = GOLD["kv_bytes_per_token"]["value"]
    k_q8 = k * GOLD["q8_0"]["q8_group_bytes"] / GOLD["q8_0"]["bf16_group_bytes"]
    total = sizes.step_read_bytes(rb["weight_bytes"], g["batch"], g["context"], k_q8)
    assert round(total / 1e9, 2) == g["gb"]


# ------------------------------------------------------------ quantiser --


def test_integer_group_is_stored_exactly():
    """amax 127: scale 1, the codes are the values themselves."""
    x = np.arange(-127, 127 + 1, 8, dtype=np.float32)[:32]
    x[5] = 127.0
    codes, sb = oracle.quantize_q8_0_group(_bf16(x))
    assert sb == _fp16_bits(1.0)
    assert np.array_equal(codes.astype(np.float32), x)


@pytest.mark.parametrize("k", [-10, -3, -1, 1, 4, 8])
def test_power_of_two_scaling(k):
    """Scaling a group by 2^k scales d by 2^k exactly and leaves the codes."""
    rng = np.random.default_rng(100 + k)
    x = rng.integers(-127, 128, size=32).astype(np.float32)
    x[0] = -127.0
    codes0, sb0 = oracle.quantize_q8_0_group(_bf16(x))
    codes1, sb1 = oracle.quantize_q8_0_group(_bf16(x * np.float32(2.0 ** k)))
    assert np.array_equal(codes0, codes1)
    assert sb0 == _fp16_bits(1.0) and sb1 == _fp16_bits(2.0 ** k)


def test_zero_group():
    codes, sb = oracle.quantize_q8_0_group(np.zeros(32, np.uint16))
    assert sb == 0 and not codes.any()


def test_half_way_values_round_away_from_zero():
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1:9] = [0.5, 1.5, 2.5, -0.5, -2.5, 126.5, -3.5, 4.5]
    codes, _ = oracle.quantize_q8_0_group(_bf16(x))
    assert list(codes[:9]) == [127, 1, 2, 3, -1, -3, 127, -4, 5]


def test_error_bound_and_extreme_code():
    """|x - s*code| <= d/2 + 127*|s - d| with s = fp16(d); the group's
    largest magnitude gets code +-127."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        x32 = (rng.standard_normal(32) * 2.0 ** rng.integers(-8, 8)).astype(np.float32)
        bits = (x32.view(np.uint32) >> 16).astype(np.uint16)  # truncated to BF16
        x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        codes, sb = oracle.quantize_q8_0_group(bits)
        s = float(np.array([sb], np.uint16).view(np.float16)[0])
        d = np.float64(np.float32(np.abs(x).max()) / np.float32(127.0))
        err = np.abs(x - s * codes.astype(np.float64))
        assert err.max() <= d / 2 + 127 * abs(s - d) + 1e-12 * d
        i = int(np.abs(x).argmax())
        assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(x[i])


# -------------------------------------------------------- layout, append --


def test_tile_byte_layout():
    """The documented tile: codes int8 [16][128] (token-major), then FP16
    scales [16][4]; slot s lives in block s // 16 at offset s % 16."""
    nb, hkv = 3, 2
    kc = np.zeros((nb, hkv, oracle.Q8_TILE_BYTES), np.uint8)
    vc = np.zeros_like(kc)
    vals = np.zeros((1, hkv, 128), np.float32)
    for h in range(hkv):
        for g in range(4):
            grp = np.arange(32, dtype=np.float32) - 16.0  # max |x| 16 -> d = 16/127
            vals[0, h, 32 * g:32 * g + 32] = grp * np.float32(2.0 ** (g - h))
    slot = 1 * 16 + 5
    oracle.kv_append_q8_0(kc, vc, np.array([slot]), _bf16(vals), _bf16(-vals))
    for h in range(hkv):
        tile = kc[1, h]
        for g in range(4):
            codes_ref, sb_ref = oracle.quantize_q8_0_group(_bf16(vals[0, h, 32 * g:32 * g + 32]))
            assert np.array_equal(tile[5 * 128 + 32 * g:5 * 128 + 32 * g + 32].view(np.int8), codes_ref)
            off = 2048 + (5 * 4 + g) * 2
            assert int(tile[off]) | (int(tile[off + 1]) << 8) == sb_ref
        # nothing else of the pool was written
        mask = np.zeros(oracle.Q8_TILE_BYTES, bool)
        mask[5 * 128:6 * 128] = True
        mask[2048 + 40:2048 + 48] = True
        assert not tile[~mask].any()
    assert not kc[0].any() and not kc[2].any()
    assert np.array_equal(vc[1, :, 5 * 128:6 * 128].view(np.int8), -kc[1, :, 5 * 128:6 * 128].view(np.int8))


def _exact_tokens(rng, n, hkv):
    """BF16 K/V rows that q8_0 stores exactly: every 32-value group is an
    integer vector with max |x| = 127, times its own power of two."""
    x = rng.integers(-127, 128, size=(n, hkv, 4, 32)).astype(np.float32)
    x[..., 0] = np.where(rng.random((n, hkv, 4)) < 0.5, 127.0, -127.0)
    e = rng.integers(-12, -4, size=(n, hkv, 4, 1)).astype(np.float32)
    return _bf16((x * np.float32(2.0) ** e).reshape(n, hkv, 128))


def test_append_then_dequantize_matches_bf16_append():
    rng = np.random.default_rng(11)
    nb, hkv, n = 9, 2, 40
    slots = rng.permutation(nb * 16)[:n].astype(np.int64)
    slots[3] = -1  # padding entry: skipped
    k_new, v_new = _exact_tokens(rng, n, hkv), _exact_tokens(rng, n, hkv)
    kq = np.zeros((nb, hkv, oracle.Q8_TILE_BYTES), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_q8_0(kq, vq, slots, k_new, v_new)
    kb = np.zeros((nb, hkv, 16, 128), np.uint16)
    vb = np.zeros_like(kb)
    oracle.kv_append(kb, vb, slots, k_new, v_new)
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(oracle.dequantize_q8_0(kq), f(kb))
    assert np.array_equal(oracle.dequantize_q8_0(vq), f(vb))


@pytest.mark.parametrize("q_len", [1, 3])
def test_attention_on_exact_values_equals_bf16_oracle(q_len):
    rng = np.random.default_rng(5 + q_len)
    b, hkv, nb, mb = 3, 2, 24, 6
    ctx = np.array([70, 1, 96], np.int32)[:b]
    tables = rng.permutation(nb)[:b * mb].reshape(b, mb).astype(np.int32)
    slots = []
    for r in range(b):
        for t in range(ctx[r]):
            slots.append(tables[r, t // 16] * 16 + t % 16)
    slots = np.array(slots, np.int64)
    k_new, v_new = _exact_tokens(rng, len(slots), hkv), _exact_tokens(rng, len(slots), hkv)
    kq = np.zeros((nb, hkv, oracle.Q8_TILE_BYTES), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_q8_0(kq, vq, slots, k_new, v_new)
    kb = np.zeros((nb, hkv, 16, 128), np.uint16)
    vb = np.zeros_like(kb)
    oracle.kv_append(kb, vb, slots, k_new, v_new)
    q = W.randn_bf16(rng, (b, q_len, 4 * hkv, 128))
    ref = oracle.paged_attention(q, kb, vb, tables, ctx, q_len, 128 ** -0.5)
    got = oracle.paged_attention_f64(q, oracle.dequantize_q8_0(kq), oracle.dequantize_q8_0(vq), tables, ctx, q_len,
                                     128 ** -0.5)
    assert np.array_equal(got, ref)
