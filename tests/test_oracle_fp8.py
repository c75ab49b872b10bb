"""Pins of the FP8 (E4M3) KV oracle (web textbook page "Chapter 8: Inference
Optimization", §8.4.4: K and V stored in FP8, the query kept in BF16) to
things other than itself: values the E4M3 format fixes, an exhaustive check
of the encoder against a brute-force nearest-value search over every finite
BF16 input, the pool layout, and -- for values E4M3 stores exactly --
agreement with the pinned BF16 attention oracle."""
import numpy as np
import pytest

import oracle
import workloads as W


def _bf16(x) -> np.ndarray:
    a = np.asarray(x, np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), a), "value not exact in BF16"
    return bits


def _table():
    return np.array([oracle.e4m3_value(c) for c in range(256) if (c & 0x7F) != 0x7F])


def test_e4m3_values_fixed_by_the_format():
    # 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals below 2^-6
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0, 0x39: 1.125,
             0x3F: 1.875, 0x40: 2.0, 0x70: 128.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in known.items():
        assert oracle.e4m3_value(c) == v, hex(c)
    pos = [oracle.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(pos, pos[1:]))  # codes 0x00..0x7E increase strictly
    assert len(pos) == 127 and max(pos) == 448.0


def test_encoder_is_nearest_value_with_ties_to_even_for_every_bf16():
    """All 65536 BF16 patterns (the finite ones): the encoder's code must be the
    nearest E4M3 value, ties to the even code, saturating at +-448."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    vals = np.array([oracle.e4m3_value(c) for c in codes])
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(x)
    mism = []
    for xi in x[finite][::1]:
        got = oracle.e4m3_encode(xi)
        if abs(xi) >= 448.0:
            want_mag = 448.0
            ok = oracle.e4m3_value(got) == np.copysign(want_mag, xi)
        else:
            d = np.abs(vals - xi)
            best = d.min()
            cand = codes[d == best]
            # among equally near codes of the right sign (two at most, or +-0), the even one
            cand = [c for c in cand if (c >> 7) == (1 if np.signbit(xi) else 0)] or list(cand)
            want = min(cand, key=lambda c: (c & 1, c))
            ok = got == want or (oracle.e4m3_value(got) == oracle.e4m3_value(want) and best == 0.0)
        if not ok:
            mism.append(xi)
            if len(mism) > 5:
                break
    assert not mism, f"encoder differs from the nearest-value search at {mism}"


def test_round_trip_and_sign_of_zero():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c or oracle.e4m3_value(c) == 0.0
    assert oracle.e4m3_encode(-0.0) == 0x80 and oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(1e9) == 0x7E and oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00          # half the smallest subnormal: tie to even (zero)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02      # 1.5 subnormal steps: tie to even (2)


def _exact_fp8_tokens(rng, n, hkv):
    """BF16 rows that E4M3 stores exactly: small integers times powers of two."""
    m = rng.integers(-15, 16, size=(n, hkv, 128)).astype(np.float32)
    e = rng.integers(-6, 3, size=(n, hkv, 128)).astype(np.float32)
    return _bf16(m * np.float32(2.0) ** e)


def test_append_layout_and_exact_values():
    rng = np.random.default_rng(21)
    nb, hkv, n = 7, 2, 30
    slots = rng.permutation(nb * 16)[:n].astype(np.int64)
    slots[2] = -1
    k_new, v_new = _exact_fp8_tokens(rng, n, hkv), _exact_fp8_tokens(rng, n, hkv)
    kq = np.zeros((nb, hkv, 16, 128), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_fp8(kq, vq, slots, k_new, v_new)
    kb = np.zeros((nb, hkv, 16, 128), np.uint16)
    vb = np.zeros_like(kb)
    oracle.kv_append(kb, vb, slots, k_new, v_new)
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(oracle.dequantize_fp8(kq), f(kb))
    assert np.array_equal(oracle.dequantize_fp8(vq), f(vb))


def test_rounding_of_random_values():
    """Random BF16 values: E4M3 keeps 3 mantissa bits, so the relative error of a
    normal value is at most 2^-4, and subnormals are off by at most 2^-10."""
    rng = np.random.default_rng(22)
    x = (W.randn_bf16(rng, (4096,)).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.e4m3_value(oracle.e4m3_encode(v)) for v in x])
    err = np.abs(got - x)
    normal = np.abs(x) >= 2.0 ** -6
    assert (err[normal] <= np.abs(x[normal]) * 2.0 ** -4 + 1e-15).all()
    assert (err[~normal] <= 2.0 ** -10 + 1e-15).all()


@pytest.mark.parametrize("q_len", [1, 2])
def test_attention_on_exact_values_equals_bf16_oracle(q_len):
    rng = np.random.default_rng(30 + q_len)
    b, hkv, nb, mb = 3, 2, 20, 5
    ctx = np.array([33, 80, 7], np.int32)
    tables = rng.permutation(nb)[:b * mb].reshape(b, mb).astype(np.int32)
    slots = np.array([tables[r, t // 16] * 16 + t % 16 for r in range(b) for t in range(ctx[r])], np.int64)
    k_new, v_new = _exact_fp8_tokens(rng, len(slots), hkv), _exact_fp8_tokens(rng, len(slots), hkv)
    kq = np.zeros((nb, hkv, 16, 128), np.uint8)
    vq = np.zeros_like(kq)
    oracle.kv_append_fp8(kq, vq, slots, k_new, v_new)
    kb = np.zeros((nb, hkv, 16, 128), np.uint16)
    vb = np.zeros_like(kb)
    oracle.kv_append(kb, vb, slots, k_new, v_new)
    q = W.randn_bf16(rng, (b, q_len, 4 * hkv, 128))
    ref = oracle.paged_attention(q, kb, vb, tables, ctx, q_len, 128 ** -0.5)
    got = oracle.paged_attention_f64(q, oracle.dequantize_fp8(kq), oracle.dequantize_fp8(vq), tables, ctx, q_len,
                                     128 ** -0.5)
    assert np.array_equal(got, ref)
