"""Mistakes planted in a copy of the oracle must each break at least one pin.

Each mutant is a one-line edit of pkv_oracle.c of the kind a careless
restatement might make (a dropped scale, an off-by-one causal rule, a wrong
GQA group, a transposed cache index, a dropped normalisation, a wrong BF16
decode, a wrong slot split, the q8_0 quantiser's scale, rounding and layout,
and the FP8 encoder's rounding, bias, saturation and layout).  The copy is
compiled on the CPU and the pins of the oracle tests are run against it.
"""
import inspect

import pytest

import oracle
import test_oracle_attention as A
import test_oracle_fp8 as F
import test_oracle_q8 as Q
import test_oracle_sizes as S

MUTANTS = {
    "dropped_scale": ("logit[t] = scale * dot;", "logit[t] = dot;"),
    "causal_off_by_one": ("t <= (int64_t)ctx - q_len + i", "t < (int64_t)ctx - q_len + i"),
    "gqa_interleaved": ("int32_t kvh = h / group;", "int32_t kvh = h % num_kv_heads;"),
    "transposed_cache_index": ("return ((blk * num_kv_heads + kvh) * block_size + off)",
                               "return ((blk * block_size + off) * num_kv_heads + kvh)"),
    "unnormalised": ("double w = exp(logit[t] - m) / denom;", "double w = exp(logit[t] - m);"),
    "bf16_decode": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "slot_split": ("int32_t off = (int32_t)(slot % block_size);",
                   "int32_t off = (int32_t)((slot + 1) % block_size);"),
    # ignores the block table: logical block j read from physical block j
    "table_ignored": ("int64_t blk = block_tables[(int64_t)r * max_blocks_per_seq + t / block_size];",
                      "int64_t blk = t / block_size;"),
    # q8_0 (§8.4.2): wrong code range, round-half-even, scale stored in the
    # wrong slot, codes read unsigned, wrong group of a scale, groups stored
    # in reverse, V read from the K pool
    "q8_scale_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "q8_round_half_even": ("codes[i] = (int8_t)roundf(", "codes[i] = (int8_t)rintf("),
    "q8_scale_slot": ("memcpy(tile + 2048 + (off * 4 + g) * 2, &sb, 2);",
                      "memcpy(tile + 2048 + (g * 16 + off) * 2, &sb, 2);"),
    "q8_codes_unsigned": ("(double)(int8_t)tile[t * 128 + d]", "(double)tile[t * 128 + d]"),
    "q8_scale_group": ("(t * 4 + d / 32) * 2", "(t * 4 + d / 64) * 2"),
    "q8_groups_reversed": ("(int8_t*)(tile + off * 128 + 32 * g)", "(int8_t*)(tile + off * 128 + 32 * (3 - g))"),
    "q8_attention_reads_k_as_v": ("o[d] += w * v_cache[cache_index(", "o[d] += w * k_cache[cache_index("),
    # FP8 E4M3 (§8.4.4): ties away from zero, wrong exponent bias, overflow to
    # NaN instead of saturation, wrong subnormal step, transposed pool layout
    "fp8_ties_away": ("else pick = (lo & 1) ? hi : lo;", "else pick = hi;"),
    "fp8_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 6)"),
    "fp8_no_saturation": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 448.0) return sign | 0x7F;"),
    "fp8_subnormal_step": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "fp8_layout": ("int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * 128 + d;",
                   "int64_t dst = ((blk * block_size + off) * num_kv_heads + h) * 128 + d;"),
}


def _pins():
    fns = []
    for mod in (A, F, Q, S):
        for name, fn in inspect.getmembers(mod, inspect.isfunction):
            if name.startswith("test_") and fn.__module__ == mod.__name__:
                fns.append((name, fn))
    return fns


def _run_pin(fn):
    sig = inspect.signature(fn)
    if not sig.parameters:
        fn()
        return
    # parametrised pins: run each parameter set
    marks = getattr(fn, "pytestmark", [])
    params = [m for m in marks if m.name == "parametrize"]
    combos = [{}]
    for m in params:
        names = [n.strip() for n in m.args[0].split(",")]
        new = []
        for c in combos:
            for val in m.args[1]:
                vals = val if len(names) > 1 else (val,)
                new.append({**c, **dict(zip(names, vals))})
        combos = new
    for c in combos:
        fn(**c)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_breaks_a_pin(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation anchor not found: {old}"
    path = oracle.build_variant(src.replace(old, new), str(tmp_path / f"liboracle_{mutant}.so"))
    caught = []
    with oracle.swapped_library(path):
        for name, fn in _pins():
            try:
                _run_pin(fn)
            except (AssertionError, ValueError):
                caught.append(name)
    assert caught, f"no pin caught mutant {mutant}"


def test_unmutated_oracle_passes_every_pin():
    for name, fn in _pins():
        _run_pin(fn)
