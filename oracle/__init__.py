"""FP64 CPU oracle for paged KV decode attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference legs may import this package.  The library never does, and this
package imports nothing from the library: the two share only the seeded input
generator (``workloads``).

Contents:
  * ``pkv_oracle.c`` (built here into ``_build/liboracle.so``): the plain
    definition in C, FP64, OpenMP over output rows;
  * ``brute``: an independent dense NumPy restatement for tiny inputs;
  * ``sizes``: the pages' sizing arithmetic (bytes per token, blocks, waste,
    capacity), pinned by the printed values in the tests.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build", platform.machine())
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    c_p = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.oracle_kv_append.argtypes = [c_p, c_p, i32, i32, i32, i32, c_p, c_p, c_p, i32]
    lib.oracle_kv_append.restype = None
    lib.oracle_visible_pairs.argtypes = [c_p, i32, i32]
    lib.oracle_visible_pairs.restype = ctypes.c_int64
    lib.oracle_paged_attention.argtypes = [c_p, c_p, c_p, c_p, c_p, i32, i32, i32, i32, c_p, i32,
                                           c_p, i32, i32, i32, ctypes.c_double, c_p, i32, i32]
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    lib.oracle_quantize_q8_0_group.argtypes = [c_p, c_p, c_p]
    lib.oracle_quantize_q8_0_group.restype = None
    lib.oracle_kv_append_q8_0.argtypes = [c_p, c_p, i32, i32, i32, c_p, c_p, c_p, i32]
    lib.oracle_kv_append_q8_0.restype = None
    lib.oracle_dequantize_q8_0.argtypes = [c_p, c_p, i32, i32, i32]
    lib.oracle_dequantize_q8_0.restype = None
    lib.oracle_paged_attention_f64.argtypes = [c_p, c_p, c_p, c_p, c_p, i32, i32, i32, i32, c_p, i32, c_p, i32, i32,
                                               i32, ctypes.c_double, i32]
    lib.oracle_paged_attention_f64.restype = ctypes.c_int
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_kv_append_fp8.argtypes = [c_p, c_p, i32, i32, i32, c_p, c_p, c_p, i32]
    lib.oracle_kv_append_fp8.restype = None
    lib.oracle_dequantize_fp8.argtypes = [c_p, c_p, ctypes.c_int64]
    lib.oracle_dequantize_fp8.restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def swapped_library(path: str):
    """Run the Python entry points against another build of pkv_oracle.c
    (used by the tests that plant mistakes in the oracle to prove the pins
    catch them)."""
    global _lib
    saved = _load()
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def build_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of pkv_oracle.c (test use only)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp", src, "-o", out_path,
                    "-lm"],
                   check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping: np.ndarray,
              k_new: np.ndarray, v_new: np.ndarray) -> None:
    """In place: store new K/V rows in their slots (uint16 BF16 bit patterns)."""
    lib = _load()
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    nb, hkv, bs, d = k_cache.shape
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    t = slot_mapping.shape[0]
    assert k_new.shape == (t, hkv, d) and v_new.shape == (t, hkv, d)
    lib.oracle_kv_append(_ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d, _ptr(slot_mapping),
                         _ptr(k_new), _ptr(v_new), t)


def visible_pairs(context_lens, q_len: int) -> int:
    """(query, key) pairs admitted by the oracle's causal rule."""
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    return int(_load().oracle_visible_pairs(_ptr(ctx), ctx.shape[0], q_len))


def paged_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    block_tables: np.ndarray, context_lens: np.ndarray, q_len: int, scale: float,
                    seq_ids=None, num_threads: int = 0, with_lse: bool = False):
    """FP64 attention for every (selected) request; returns float64
    [n_sel][q_len][Hq][D] (and the natural-log lse [n_sel][q_len][Hq])."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    b, ql, hq, d = q.shape
    assert ql == q_len
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape and hq % hkv == 0
    ids = None
    n_sel = b
    if seq_ids is not None:
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        n_sel = ids.shape[0]
    out = np.zeros((n_sel, q_len, hq, d), dtype=np.float64)
    lse = np.zeros((n_sel, q_len, hq), dtype=np.float64)
    rc = lib.oracle_paged_attention(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    nb, bs, hkv, d, _ptr(tables), tables.shape[1], _ptr(ctx), b,
                                    q_len, hq, float(scale), _ptr(ids),
                                    0 if ids is None else n_sel, int(num_threads))
    if rc != 0:
        raise ValueError("block table entry outside the pool")
    return (out, lse) if with_lse else out


def run_workload(w, seq_ids=None, num_threads: int = 0, with_lse: bool = False, append: bool = True):
    """Apply the step's kv_append to copies of the pools, then attend."""
    kc = w.k_cache.copy()
    vc = w.v_cache.copy()
    if append:
        kv_append(kc, vc, w.slot_mapping, w.k_new, w.v_new)
    return paged_attention(w.q, kc, vc, w.block_tables, w.context_lens, w.q_len, w.scale,
                           seq_ids=seq_ids, num_threads=num_threads, with_lse=with_lse)


def attn_combine(partial_o: np.ndarray, partial_lse: np.ndarray):
    """Merge per-range attention results, FP64.

    partial_o [rows][S][D] holds each key range's own normalised softmax
    output and partial_lse [rows][S] its natural-log log-sum-exp (-inf for a
    range without keys).  A softmax over the union of disjoint ranges is the
    mix of the per-range ones weighted by exp(lse_s - lse), lse = log sum_s
    exp(lse_s).  Returns (out [rows][D], lse [rows]); rows without keys give
    zeros and -inf.
    """
    po = np.asarray(partial_o, dtype=np.float64)
    pl = np.asarray(partial_lse, dtype=np.float64)
    rows, s, d = po.shape
    out = np.zeros((rows, d))
    lse = np.full(rows, -np.inf)
    for r in range(rows):
        finite = np.isfinite(pl[r])
        if not finite.any():
            continue
        m = pl[r][finite].max()
        total = np.log(np.exp(pl[r][finite] - m).sum()) + m
        w = np.exp(pl[r][finite] - total)
        out[r] = (w[:, None] * po[r][finite]).sum(axis=0)
        lse[r] = total
    return out, lse


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, src_blocks, dst_blocks) -> None:
    """In place: physical block dst <- physical block src, all heads, K and V
    (the copy step of copy-on-write, §8.3.2 / Fig. 8-15)."""
    for s, d in zip(src_blocks, dst_blocks):
        k_cache[int(d)] = k_cache[int(s)]
        v_cache[int(d)] = v_cache[int(s)]


# ---------------------------------------------------------------------------
# q8_0 KV (§8.4.2, Fig. 8-23): 32 values share one FP16 scale; 8-bit codes.
# Pool per tensor: uint8 [num_blocks][Hkv][2176] = codes int8 [16][128] then
# scales fp16 [16][4] for each (block, kv head).
# ---------------------------------------------------------------------------
Q8_TILE_BYTES = 2176


def quantize_q8_0_group(x_bits: np.ndarray):
    """32 BF16 bit patterns -> (int8 codes[32], uint16 FP16 scale bits)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert x.size == 32
    codes = np.zeros(32, np.int8)
    sb = np.zeros(1, np.uint16)
    _load().oracle_quantize_q8_0_group(_ptr(x), _ptr(codes), _ptr(sb))
    return codes, int(sb[0])


def kv_append_q8_0(k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping, k_new, v_new, block_size: int = 16):
    """In place: quantize and store new K/V rows in q8_0 pools (uint8 [nb][Hkv][2176])."""
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    nb, hkv, tb = k_cache.shape
    assert tb == Q8_TILE_BYTES
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    _load().oracle_kv_append_q8_0(_ptr(k_cache), _ptr(v_cache), nb, block_size, hkv, _ptr(slot_mapping), _ptr(k_new),
                                  _ptr(v_new), slot_mapping.shape[0])


def dequantize_q8_0(cache: np.ndarray, block_size: int = 16) -> np.ndarray:
    """q8_0 pool -> float64 [nb][Hkv][16][128] of scale * code."""
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    nb, hkv, _ = cache.shape
    out = np.zeros((nb, hkv, block_size, 128), np.float64)
    _load().oracle_dequantize_q8_0(_ptr(cache), _ptr(out), nb, hkv, block_size)
    return out


def paged_attention_f64(q, k_cache_f64, v_cache_f64, block_tables, context_lens, q_len: int, scale: float,
                        num_threads: int = 0, with_lse: bool = False):
    """Attention over float64 pools [nb][Hkv][16][D] (e.g. dequantized q8_0)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(k_cache_f64, dtype=np.float64)
    vc = np.ascontiguousarray(v_cache_f64, dtype=np.float64)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    b, ql, hq, d = q.shape
    nb, hkv, bs, _ = kc.shape
    out = np.zeros((b, q_len, hq, d), np.float64)
    lse = np.zeros((b, q_len, hq), np.float64)
    rc = _load().oracle_paged_attention_f64(_ptr(out), _ptr(lse), _ptr(q), _ptr(kc), _ptr(vc), nb, bs, hkv, d,
                                            _ptr(tables), tables.shape[1], _ptr(ctx), b, q_len, hq, float(scale),
                                            int(num_threads))
    if rc != 0:
        raise ValueError("block table entry outside the pool")
    return (out, lse) if with_lse else out


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV (§8.4.4): uint8 pools [num_blocks][Hkv][16][128] of E4M3 codes.
# ---------------------------------------------------------------------------
FP8_TILE_BYTES = 2048


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(int(code)))


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def kv_append_fp8(k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping, k_new, v_new, block_size: int = 16):
    """In place: round new BF16 K/V rows to E4M3 and store them (pools uint8 [nb][Hkv][16][128])."""
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    nb, hkv, bs, d = k_cache.shape
    assert bs == block_size and d == 128
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    _load().oracle_kv_append_fp8(_ptr(k_cache), _ptr(v_cache), nb, block_size, hkv, _ptr(slot_mapping), _ptr(k_new),
                                 _ptr(v_new), slot_mapping.shape[0])


def dequantize_fp8(cache: np.ndarray) -> np.ndarray:
    """E4M3 pool -> float64 pool of the same shape."""
    cache = np.ascontiguousarray(cache, dtype=np.uint8)
    out = np.zeros(cache.shape, np.float64)
    _load().oracle_dequantize_fp8(_ptr(cache), _ptr(out), cache.size)
    return out
