"""paged_kv_decode_attention_gb300 -- Python binding of libpkv (C ABI in include/pkv.h).

Argument marshalling only: each function checks tensor dtypes/devices/shapes,
passes raw device pointers and the current CUDA stream to the exported C
function of the same name, and turns a non-zero status into PkvError.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and importing this module fails loudly when the shared
library cannot be built or loaded.

PyTorch provides device memory and streams only.  BF16 tensors are passed as
torch.bfloat16 (or int16/uint16 holding BF16 bit patterns).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "PkvError", "BlockPool", "copy_blocks", "kv_append", "paged_attention", "paged_attention_append",
    "paged_attention_cascade", "paged_attention_cascade_append", "cascade_plan",
    "cascade_workspace_size", "attn_combine", "workspace_size",
    "choose_kv_blocks_per_split", "get_device_error", "library_path", "lib", "DEVERR_BLOCK_ID",
    "DEVERR_SLOT", "DEVERR_CONTEXT", "DEVERR_TIMEOUT", "Q8_TILE_BYTES", "kv_append_q8_0", "paged_attention_q8_0",
    "choose_kv_blocks_per_split_q8_0", "choose_kv_blocks_per_split_fp8_e4m3", "workspace_size_q8_0", "copy_blocks_q8_0", "FP8_TILE_BYTES",
    "kv_append_fp8_e4m3", "paged_attention_fp8_e4m3", "paged_attention_fp8_e4m3_append",
    "paged_attention_q8_0_append", "copy_blocks_fp8_e4m3",
    "DecodeGraph", "KV_BF16", "KV_Q8_0", "KV_FP8_E4M3", "selftest_bounded_wait",
]

DEVERR_BLOCK_ID = 1
DEVERR_SLOT = 2
DEVERR_CONTEXT = 4
DEVERR_TIMEOUT = 8

BLOCK_SIZE = 16
HEAD_DIM = 128


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.pkv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


KV_BF16, KV_Q8_0, KV_FP8_E4M3 = 0, 1, 2


class DecodeGraphBuffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens",
                                               "out", "group_seqs", "group_blocks", "seq_prefix_blocks")]


class DecodeGraphDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("kv_format", ctypes.c_int32), ("cache", CacheDesc),
                ("k_caches", ctypes.POINTER(ctypes.c_void_p)), ("v_caches", ctypes.POINTER(ctypes.c_void_p)),
                ("num_seqs", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("num_tokens", ctypes.c_int32), ("scale", ctypes.c_float),
                ("kv_blocks_per_split", ctypes.c_int32), ("num_groups", ctypes.c_int32),
                ("max_prefix_blocks", ctypes.c_int32), ("max_suffix_blocks", ctypes.c_int32),
                ("prefix_blocks_per_split", ctypes.c_int32), ("suffix_blocks_per_split", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("set", DecodeGraphBuffers * 2)]


def _load():
    path = _build.build()
    lib = ctypes.CDLL(path)
    p, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.pkv_kv_append.argtypes = [p, p, ctypes.POINTER(CacheDesc), p, p, p, i32, p]
    lib.pkv_kv_append.restype = ctypes.c_int
    lib.pkv_choose_kv_blocks_per_split.argtypes = [i32, i32, i32, i32, i32]
    lib.pkv_choose_kv_blocks_per_split.restype = i32
    lib.pkv_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pkv_workspace_size.restype = sz
    lib.pkv_paged_attention.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32, i32, f32,
                                        i32, p, sz, p]
    lib.pkv_paged_attention.restype = ctypes.c_int
    lib.pkv_attn_combine.argtypes = [p, p, p, p, i32, i32, i32, p]
    lib.pkv_attn_combine.restype = ctypes.c_int
    lib.pkv_cascade_plan.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.pkv_cascade_plan.restype = None
    lib.pkv_cascade_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.pkv_cascade_workspace_size.restype = sz
    lib.pkv_paged_attention_cascade.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32, f32,
                                                p, p, p, i32, i32, i32, i32, i32, p, sz, p]
    lib.pkv_paged_attention_cascade.restype = ctypes.c_int
    pp = ctypes.POINTER(i32)
    lib.pkv_block_pool_create.argtypes = [i32, i32, ctypes.POINTER(p)]
    lib.pkv_block_pool_create.restype = ctypes.c_int
    lib.pkv_block_pool_destroy.argtypes = [p]
    lib.pkv_block_pool_destroy.restype = None
    lib.pkv_block_pool_num_free.argtypes = [p]
    lib.pkv_block_pool_num_free.restype = i32
    lib.pkv_block_pool_refcount.argtypes = [p, i32]
    lib.pkv_block_pool_refcount.restype = i32
    lib.pkv_block_pool_alloc.argtypes = [p, i32, pp]
    lib.pkv_block_pool_alloc.restype = ctypes.c_int
    lib.pkv_block_pool_share.argtypes = [p, pp, i32]
    lib.pkv_block_pool_share.restype = ctypes.c_int
    lib.pkv_block_pool_release.argtypes = [p, pp, i32]
    lib.pkv_block_pool_release.restype = ctypes.c_int
    lib.pkv_block_pool_reserve.argtypes = [p, pp, pp, i32, i32, i32, pp, pp, pp]
    lib.pkv_block_pool_reserve.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [p, p, ctypes.POINTER(CacheDesc), p, p, i32, p]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    lib.pkv_kv_append_q8_0.argtypes = [p, p, ctypes.POINTER(CacheDesc), p, p, p, i32, p]
    lib.pkv_kv_append_q8_0.restype = ctypes.c_int
    lib.pkv_choose_kv_blocks_per_split_q8_0.argtypes = [i32, i32, i32, i32]
    lib.pkv_choose_kv_blocks_per_split_q8_0.restype = i32
    lib.pkv_choose_kv_blocks_per_split_fp8_e4m3.argtypes = [i32, i32, i32, i32]
    lib.pkv_choose_kv_blocks_per_split_fp8_e4m3.restype = i32
    lib.pkv_workspace_size_q8_0.argtypes = [i32, i32, i32, i32]
    lib.pkv_workspace_size_q8_0.restype = sz
    lib.pkv_paged_attention_q8_0.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32, f32, i32,
                                             p, sz, p]
    lib.pkv_paged_attention_q8_0.restype = ctypes.c_int
    lib.pkv_copy_blocks_q8_0.argtypes = [p, p, ctypes.POINTER(CacheDesc), p, p, i32, p]
    lib.pkv_copy_blocks_q8_0.restype = ctypes.c_int
    lib.pkv_kv_append_fp8_e4m3.argtypes = [p, p, ctypes.POINTER(CacheDesc), p, p, p, i32, p]
    lib.pkv_kv_append_fp8_e4m3.restype = ctypes.c_int
    lib.pkv_paged_attention_fp8_e4m3.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32, f32, i32,
                                                 p, sz, p]
    lib.pkv_paged_attention_fp8_e4m3.restype = ctypes.c_int
    lib.pkv_copy_blocks_fp8_e4m3.argtypes = [p, p, ctypes.POINTER(CacheDesc), p, p, i32, p]
    lib.pkv_copy_blocks_fp8_e4m3.restype = ctypes.c_int
    lib.pkv_paged_attention_append.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32, i32, f32,
                                               i32, p, sz, p, p, p, i32, p]
    lib.pkv_paged_attention_append.restype = ctypes.c_int
    lib.pkv_paged_attention_cascade_append.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32,
                                                       f32, p, p, p, i32, i32, i32, i32, i32, p, sz, p, p, p, i32, p]
    lib.pkv_paged_attention_cascade_append.restype = ctypes.c_int
    lib.pkv_paged_attention_fp8_e4m3_append.argtypes = [p, p, p, p, ctypes.POINTER(CacheDesc), p, i32, p, i32, i32,
                                                        f32, i32, p, sz, p, p, p, i32, p]
    lib.pkv_paged_attention_fp8_e4m3_append.restype = ctypes.c_int
    lib.pkv_paged_attention_q8_0_append.argtypes = lib.pkv_paged_attention_fp8_e4m3_append.argtypes
    lib.pkv_paged_attention_q8_0_append.restype = ctypes.c_int
    lib.pkv_decode_graph_create.argtypes = [ctypes.POINTER(DecodeGraphDesc), ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_decode_graph_create.restype = ctypes.c_int
    lib.pkv_decode_graph_launch.argtypes = [p, i32, p]
    lib.pkv_decode_graph_launch.restype = ctypes.c_int
    lib.pkv_decode_graph_destroy.argtypes = [p]
    lib.pkv_decode_graph_destroy.restype = None
    lib.pkv_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.pkv_get_device_error.restype = ctypes.c_int
    lib.pkv_selftest_bounded_wait.argtypes = [ctypes.c_uint32, i32, p]
    lib.pkv_selftest_bounded_wait.restype = ctypes.c_int
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    del i64
    return lib, path


_lib, _path = _load()


def library_path() -> str:
    return _path


def lib():
    """The ctypes handle of libpkv.so (for callers that marshal themselves)."""
    return _lib


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _bf16(t: torch.Tensor, name: str):
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must hold BF16 values (bfloat16 or 16-bit bit patterns), got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")


def _desc(cache: torch.Tensor) -> CacheDesc:
    if cache.dim() != 4:
        raise ValueError("cache must be [num_blocks][num_kv_heads][16][128]")
    nb, hkv, bs, d = cache.shape
    return CacheDesc(nb, bs, hkv, d)


def _check(status: int, where: str):
    if status != 0:
        raise PkvError(status, where)


def kv_append(k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor,
              k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Store k_new/v_new [T][Hkv][D] into the caches at slot_mapping[T] (int64, <0 skips)."""
    _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"), _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    t = slot_mapping.numel()
    hkv, d = k_cache.shape[1], k_cache.shape[3]
    if tuple(k_new.shape) != (t, hkv, d) or tuple(v_new.shape) != (t, hkv, d):
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    desc = _desc(k_cache)
    _check(_lib.pkv_kv_append(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc), slot_mapping.data_ptr(),
                              k_new.data_ptr(), v_new.data_ptr(), t, _stream_ptr(stream)), "pkv_kv_append")


def choose_kv_blocks_per_split(num_seqs: int, num_kv_heads: int, q_len: int, max_blocks_per_seq: int,
                               sm_count: int = 0) -> int:
    return int(_lib.pkv_choose_kv_blocks_per_split(num_seqs, num_kv_heads, q_len, max_blocks_per_seq, sm_count))


def workspace_size(num_seqs: int, q_len: int, num_q_heads: int, max_blocks_per_seq: int,
                   kv_blocks_per_split: int, head_dim: int = HEAD_DIM) -> int:
    return int(_lib.pkv_workspace_size(num_seqs, q_len, num_q_heads, head_dim, max_blocks_per_seq,
                                       kv_blocks_per_split))


def paged_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    block_tables: torch.Tensor, context_lens: torch.Tensor, q_len: int, scale: float,
                    kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None, stream=None) -> None:
    """out[B][q_len][Hq][D] = causal softmax(q K^T * scale) V through the block tables.

    kv_blocks_per_split: 0 = library heuristic; >= max_blocks_per_seq = no
    split.  When a split is made, `workspace` must be a CUDA tensor of at
    least workspace_size(...) bytes (256-byte aligned, as torch allocations are).
    """
    _bf16(out, "out"), _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != q_len or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][q_len][num_q_heads][head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be [num_seqs][max_blocks_per_seq]")
    hq = q.shape[2]
    maxb = block_tables.shape[1]
    desc = _desc(k_cache)
    bps = kv_blocks_per_split
    if bps == 0:
        bps = choose_kv_blocks_per_split(b, desc.num_kv_heads, q_len, maxb)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(_lib.pkv_paged_attention(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                    ctypes.byref(desc), block_tables.data_ptr(), maxb, context_lens.data_ptr(),
                                    b, q_len, hq, float(scale), bps, ws_ptr, ws_bytes, _stream_ptr(stream)),
           "pkv_paged_attention")


def paged_attention_append(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, q_len: int, scale: float,
                           slot_mapping: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                           kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None, stream=None) -> None:
    """kv_append(k_cache, v_cache, slot_mapping, k_new, v_new), then paged_attention(...), as one call
    (one launch for a decode step that appends each request's new token; see include/pkv.h)."""
    _bf16(out, "out"), _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != q_len or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][q_len][num_q_heads][head_dim]")
    desc = _desc(k_cache)
    t = slot_mapping.numel()
    if tuple(k_new.shape) != (t, desc.num_kv_heads, HEAD_DIM) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None \
        else (0, 0)
    _check(_lib.pkv_paged_attention_append(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), b, q_len, q.shape[2], float(scale),
        int(kv_blocks_per_split), ws_ptr, ws_bytes, slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t,
        _stream_ptr(stream)), "pkv_paged_attention_append")


def cascade_plan(num_seqs: int, num_kv_heads: int, num_groups: int, max_prefix_blocks: int,
                 max_suffix_blocks: int, sm_count: int = 0):
    """(prefix_blocks_per_split, suffix_blocks_per_split) the cascade call would choose."""
    pb, sb = ctypes.c_int32(0), ctypes.c_int32(0)
    _lib.pkv_cascade_plan(num_seqs, num_kv_heads, num_groups, max_prefix_blocks, max_suffix_blocks, sm_count,
                          ctypes.byref(pb), ctypes.byref(sb))
    return int(pb.value), int(sb.value)


def cascade_workspace_size(num_seqs: int, num_q_heads: int, max_prefix_blocks: int, max_suffix_blocks: int,
                           prefix_blocks_per_split: int, suffix_blocks_per_split: int) -> int:
    return int(_lib.pkv_cascade_workspace_size(num_seqs, num_q_heads, max_prefix_blocks, max_suffix_blocks,
                                               prefix_blocks_per_split, suffix_blocks_per_split))


def paged_attention_cascade(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                            group_seqs: torch.Tensor, group_blocks: torch.Tensor, seq_prefix_blocks: torch.Tensor,
                            max_prefix_blocks: int, max_suffix_blocks: int, workspace: torch.Tensor,
                            prefix_blocks_per_split: int = 0, suffix_blocks_per_split: int = 0,
                            stream=None) -> None:
    """Decode attention (q_len 1) with shared prefixes contracted once per group of <= 16 sharers.

    group_seqs int32 [G][16] (-1 = unused), group_blocks int32 [G], seq_prefix_blocks int32 [B];
    workspace >= cascade_workspace_size(...) bytes."""
    _bf16(out, "out"), _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    for t, n in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                 (seq_prefix_blocks, "seq_prefix_blocks")):
        _i32(t, n)
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != 1 or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][1][num_q_heads][head_dim]")
    g = group_seqs.shape[0] if group_seqs is not None else 0
    if g:
        _i32(group_seqs, "group_seqs"), _i32(group_blocks, "group_blocks")
        if group_seqs.dim() != 2 or group_seqs.shape[1] != 16 or group_blocks.numel() != g:
            raise ValueError("group_seqs must be [num_groups][16] and group_blocks [num_groups]")
    desc = _desc(k_cache)
    ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(_lib.pkv_paged_attention_cascade(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), b, q.shape[2], float(scale),
        group_seqs.data_ptr() if g else 0, group_blocks.data_ptr() if g else 0, seq_prefix_blocks.data_ptr(), g,
        int(max_prefix_blocks), int(max_suffix_blocks), int(prefix_blocks_per_split), int(suffix_blocks_per_split),
        ws_ptr, ws_bytes, _stream_ptr(stream)), "pkv_paged_attention_cascade")


def paged_attention_cascade_append(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   scale: float, group_seqs: torch.Tensor, group_blocks: torch.Tensor,
                                   seq_prefix_blocks: torch.Tensor, max_prefix_blocks: int, max_suffix_blocks: int,
                                   workspace: torch.Tensor, slot_mapping: torch.Tensor, k_new: torch.Tensor,
                                   v_new: torch.Tensor, prefix_blocks_per_split: int = 0,
                                   suffix_blocks_per_split: int = 0, stream=None) -> None:
    """kv_append, then paged_attention_cascade, as one call (the suffix pass stores the new tokens)."""
    _bf16(out, "out"), _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    for t, n in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                 (seq_prefix_blocks, "seq_prefix_blocks")):
        _i32(t, n)
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != 1 or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][1][num_q_heads][head_dim]")
    g = group_seqs.shape[0] if group_seqs is not None else 0
    if g:
        _i32(group_seqs, "group_seqs"), _i32(group_blocks, "group_blocks")
    desc = _desc(k_cache)
    t = slot_mapping.numel()
    if tuple(k_new.shape) != (t, desc.num_kv_heads, HEAD_DIM) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    _check(_lib.pkv_paged_attention_cascade_append(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), b, q.shape[2], float(scale),
        group_seqs.data_ptr() if g else 0, group_blocks.data_ptr() if g else 0, seq_prefix_blocks.data_ptr(), g,
        int(max_prefix_blocks), int(max_suffix_blocks), int(prefix_blocks_per_split), int(suffix_blocks_per_split),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), slot_mapping.data_ptr(),
        k_new.data_ptr(), v_new.data_ptr(), t, _stream_ptr(stream)), "pkv_paged_attention_cascade_append")


def attn_combine(out: torch.Tensor, partial_o: torch.Tensor, partial_lse: torch.Tensor,
                 out_lse: torch.Tensor | None = None, stream=None) -> None:
    """out[rows][D] (BF16) from partial_o[rows][S][D] and partial_lse[rows][S] (FP32)."""
    _bf16(out, "out")
    if partial_o.dtype != torch.float32 or partial_lse.dtype != torch.float32:
        raise TypeError("partials must be float32")
    if not (partial_o.is_cuda and partial_lse.is_cuda and partial_o.is_contiguous() and partial_lse.is_contiguous()):
        raise ValueError("partials must be contiguous CUDA tensors")
    rows, s, d = partial_o.shape
    if tuple(partial_lse.shape) != (rows, s) or out.numel() != rows * d:
        raise ValueError("shape mismatch between out, partial_o and partial_lse")
    lse_ptr = 0
    if out_lse is not None:
        if out_lse.dtype != torch.float32 or out_lse.numel() != rows or not out_lse.is_cuda:
            raise ValueError("out_lse must be a float32 CUDA tensor of num_rows elements")
        lse_ptr = out_lse.data_ptr()
    _check(_lib.pkv_attn_combine(out.data_ptr(), lse_ptr, partial_o.data_ptr(), partial_lse.data_ptr(), rows, d, s,
                                 _stream_ptr(stream)), "pkv_attn_combine")


class BlockPool:
    """Refcounted physical-block pool (host memory) with copy-on-write reservation.

    Wraps pkv_block_pool_*: alloc / share / release blocks, and `reserve`
    a request's table row for new tokens (fresh blocks appended, shared
    partly-filled blocks replaced by private copies to be made with
    copy_blocks)."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        self._p = ctypes.c_void_p(0)
        _check(_lib.pkv_block_pool_create(num_blocks, block_size, ctypes.byref(self._p)), "pkv_block_pool_create")
        self.block_size = block_size

    def close(self):
        if self._p:
            _lib.pkv_block_pool_destroy(self._p)
            self._p = ctypes.c_void_p(0)

    def __del__(self):
        self.close()

    @staticmethod
    def _arr(values):
        return (ctypes.c_int32 * max(1, len(values)))(*values)

    @property
    def num_free(self) -> int:
        return int(_lib.pkv_block_pool_num_free(self._p))

    def refcount(self, block: int) -> int:
        return int(_lib.pkv_block_pool_refcount(self._p, block))

    def alloc(self, n: int) -> list:
        out = (ctypes.c_int32 * max(1, n))()
        _check(_lib.pkv_block_pool_alloc(self._p, n, out), "pkv_block_pool_alloc")
        return list(out[:n])

    def share(self, blocks) -> None:
        _check(_lib.pkv_block_pool_share(self._p, self._arr(blocks), len(blocks)), "pkv_block_pool_share")

    def release(self, blocks) -> None:
        _check(_lib.pkv_block_pool_release(self._p, self._arr(blocks), len(blocks)), "pkv_block_pool_release")

    def reserve(self, table_row: list, ctx_before: int, num_new: int, max_blocks: int):
        """Extend/privatise `table_row` (list, modified in place) for num_new tokens
        after ctx_before; returns the list of (src, dst) block copies to make."""
        row = (ctypes.c_int32 * max(1, max_blocks))(*table_row)
        n = ctypes.c_int32(len(table_row))
        cap = -(-num_new // self.block_size) + 1
        src, dst = (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)()
        nc = ctypes.c_int32(0)
        _check(_lib.pkv_block_pool_reserve(self._p, row, ctypes.byref(n), max_blocks, ctx_before, num_new, src, dst,
                                           ctypes.byref(nc)), "pkv_block_pool_reserve")
        table_row[:] = list(row[:n.value])
        return [(src[i], dst[i]) for i in range(nc.value)]


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_blocks: torch.Tensor, dst_blocks: torch.Tensor,
                stream=None) -> None:
    """Copy physical blocks src -> dst (all heads, K and V), bit for bit."""
    _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(src_blocks, "src_blocks"), _i32(dst_blocks, "dst_blocks")
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks differ in length")
    desc = _desc(k_cache)
    _check(_lib.pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc), src_blocks.data_ptr(),
                                dst_blocks.data_ptr(), src_blocks.numel(), _stream_ptr(stream)), "pkv_copy_blocks")


# ---------------------------------------------------------------------------
# q8_0 KV pools: uint8 [num_blocks][num_kv_heads][Q8_TILE_BYTES] per tensor
# (codes int8 [16][128], then FP16 scales [16][4] per (block, kv head)).
# ---------------------------------------------------------------------------
Q8_TILE_BYTES = 2176


def _q8_pool(t: torch.Tensor, name: str) -> CacheDesc:
    if t.dtype not in (torch.uint8, torch.int8) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor")
    if t.dim() != 3 or t.shape[2] != Q8_TILE_BYTES:
        raise ValueError(f"{name} must be [num_blocks][num_kv_heads][{Q8_TILE_BYTES}]")
    return CacheDesc(t.shape[0], BLOCK_SIZE, t.shape[1], HEAD_DIM)


def kv_append_q8_0(k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                   k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Quantise k_new/v_new [T][Hkv][128] (BF16) to q8_0 and store them at slot_mapping[T]."""
    desc = _q8_pool(k_cache, "k_cache")
    _q8_pool(v_cache, "v_cache")
    _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    t = slot_mapping.numel()
    if tuple(k_new.shape) != (t, desc.num_kv_heads, HEAD_DIM) or tuple(v_new.shape) != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][128]")
    _check(_lib.pkv_kv_append_q8_0(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                                   slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t,
                                   _stream_ptr(stream)), "pkv_kv_append_q8_0")


def choose_kv_blocks_per_split_q8_0(num_seqs: int, num_kv_heads: int, max_blocks_per_seq: int,
                                    sm_count: int = 0) -> int:
    return int(_lib.pkv_choose_kv_blocks_per_split_q8_0(num_seqs, num_kv_heads, max_blocks_per_seq, sm_count))


def choose_kv_blocks_per_split_fp8_e4m3(num_seqs: int, num_kv_heads: int, max_blocks_per_seq: int,
                                        sm_count: int = 0) -> int:
    return int(_lib.pkv_choose_kv_blocks_per_split_fp8_e4m3(num_seqs, num_kv_heads, max_blocks_per_seq, sm_count))


def workspace_size_q8_0(num_seqs: int, num_q_heads: int, max_blocks_per_seq: int, kv_blocks_per_split: int) -> int:
    return int(_lib.pkv_workspace_size_q8_0(num_seqs, num_q_heads, max_blocks_per_seq, kv_blocks_per_split))


def paged_attention_q8_0(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                         kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None, stream=None) -> None:
    """Decode step (q_len 1) over q8_0 pools: out[B][1][Hq][128] = softmax(q K^T * scale) V."""
    desc = _q8_pool(k_cache, "k_cache")
    _q8_pool(v_cache, "v_cache")
    _bf16(out, "out"), _bf16(q, "q")
    _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != 1 or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][1][num_q_heads][128]")
    if block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be [num_seqs][max_blocks_per_seq]")
    maxb = block_tables.shape[1]
    bps = kv_blocks_per_split or choose_kv_blocks_per_split_q8_0(b, desc.num_kv_heads, maxb)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(_lib.pkv_paged_attention_q8_0(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                         ctypes.byref(desc), block_tables.data_ptr(), maxb, context_lens.data_ptr(),
                                         b, q.shape[2], float(scale), bps, ws_ptr, ws_bytes, _stream_ptr(stream)),
           "pkv_paged_attention_q8_0")


def paged_attention_q8_0_append(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                slot_mapping: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None,
                                stream=None) -> None:
    """kv_append_q8_0, then paged_attention_q8_0, as one call (one launch when each request appends its one new
    token)."""
    desc = _q8_pool(k_cache, "k_cache")
    _q8_pool(v_cache, "v_cache")
    _bf16(out, "out"), _bf16(q, "q"), _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != 1 or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][1][num_q_heads][head_dim]")
    t = slot_mapping.numel()
    if tuple(k_new.shape) != (t, desc.num_kv_heads, HEAD_DIM) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None \
        else (0, 0)
    _check(_lib.pkv_paged_attention_q8_0_append(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), b, q.shape[2], float(scale),
        int(kv_blocks_per_split), ws_ptr, ws_bytes, slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t,
        _stream_ptr(stream)), "pkv_paged_attention_q8_0_append")


def copy_blocks_q8_0(k_cache: torch.Tensor, v_cache: torch.Tensor, src_blocks: torch.Tensor,
                     dst_blocks: torch.Tensor, stream=None) -> None:
    """copy_blocks for q8_0 pools."""
    desc = _q8_pool(k_cache, "k_cache")
    _q8_pool(v_cache, "v_cache")
    _i32(src_blocks, "src_blocks"), _i32(dst_blocks, "dst_blocks")
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks differ in length")
    _check(_lib.pkv_copy_blocks_q8_0(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                                     src_blocks.data_ptr(), dst_blocks.data_ptr(), src_blocks.numel(),
                                     _stream_ptr(stream)), "pkv_copy_blocks_q8_0")


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV pools: uint8 [num_blocks][num_kv_heads][16][128] codes.
# ---------------------------------------------------------------------------
FP8_TILE_BYTES = 2048


def _fp8_pool(t: torch.Tensor, name: str) -> CacheDesc:
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 (or float8_e4m3fn) tensor")
    if t.dim() != 4 or t.shape[2] != BLOCK_SIZE or t.shape[3] != HEAD_DIM:
        raise ValueError(f"{name} must be [num_blocks][num_kv_heads][16][128]")
    return CacheDesc(t.shape[0], BLOCK_SIZE, t.shape[1], HEAD_DIM)


def kv_append_fp8_e4m3(k_cache: torch.Tensor, v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                       k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Round k_new/v_new [T][Hkv][128] (BF16) to E4M3 and store them at slot_mapping[T]."""
    desc = _fp8_pool(k_cache, "k_cache")
    _fp8_pool(v_cache, "v_cache")
    _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    t = slot_mapping.numel()
    if tuple(k_new.shape) != (t, desc.num_kv_heads, HEAD_DIM) or tuple(v_new.shape) != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][128]")
    _check(_lib.pkv_kv_append_fp8_e4m3(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                                       slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t,
                                       _stream_ptr(stream)), "pkv_kv_append_fp8_e4m3")


def paged_attention_fp8_e4m3(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                             kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None,
                             stream=None) -> None:
    """Decode step (q_len 1) over E4M3 pools with a BF16 query: out[B][1][Hq][128]."""
    desc = _fp8_pool(k_cache, "k_cache")
    _fp8_pool(v_cache, "v_cache")
    _bf16(out, "out"), _bf16(q, "q")
    _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != 1 or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][1][num_q_heads][128]")
    if block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be [num_seqs][max_blocks_per_seq]")
    maxb = block_tables.shape[1]
    bps = kv_blocks_per_split or choose_kv_blocks_per_split_q8_0(b, desc.num_kv_heads, maxb)
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(_lib.pkv_paged_attention_fp8_e4m3(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                             ctypes.byref(desc), block_tables.data_ptr(), maxb,
                                             context_lens.data_ptr(), b, q.shape[2], float(scale), bps, ws_ptr,
                                             ws_bytes, _stream_ptr(stream)), "pkv_paged_attention_fp8_e4m3")


def paged_attention_fp8_e4m3_append(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                    v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                    scale: float, slot_mapping: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                    kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None,
                                    stream=None) -> None:
    """kv_append_fp8_e4m3, then paged_attention_fp8_e4m3, as one call (one launch when each request appends its
    one new token)."""
    desc = _fp8_pool(k_cache, "k_cache")
    _fp8_pool(v_cache, "v_cache")
    _bf16(out, "out"), _bf16(q, "q"), _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    _i32(block_tables, "block_tables"), _i32(context_lens, "context_lens")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous CUDA int64 tensor")
    b = context_lens.numel()
    if q.dim() != 4 or q.shape[0] != b or q.shape[1] != 1 or out.shape != q.shape:
        raise ValueError("q/out must be [num_seqs][1][num_q_heads][head_dim]")
    t = slot_mapping.numel()
    if tuple(k_new.shape) != (t, desc.num_kv_heads, HEAD_DIM) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new/v_new must be [num_tokens][num_kv_heads][head_dim]")
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) if workspace is not None \
        else (0, 0)
    _check(_lib.pkv_paged_attention_fp8_e4m3_append(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), b, q.shape[2], float(scale),
        int(kv_blocks_per_split), ws_ptr, ws_bytes, slot_mapping.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), t,
        _stream_ptr(stream)), "pkv_paged_attention_fp8_e4m3_append")


def copy_blocks_fp8_e4m3(k_cache: torch.Tensor, v_cache: torch.Tensor, src_blocks: torch.Tensor,
                         dst_blocks: torch.Tensor, stream=None) -> None:
    """copy_blocks for E4M3 pools."""
    desc = _fp8_pool(k_cache, "k_cache")
    _fp8_pool(v_cache, "v_cache")
    _i32(src_blocks, "src_blocks"), _i32(dst_blocks, "dst_blocks")
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks differ in length")
    _check(_lib.pkv_copy_blocks_fp8_e4m3(k_cache.data_ptr(), v_cache.data_ptr(), ctypes.byref(desc),
                                         src_blocks.data_ptr(), dst_blocks.data_ptr(), src_blocks.numel(),
                                         _stream_ptr(stream)), "pkv_copy_blocks_fp8_e4m3")


def _addr(x) -> int:
    return int(x) if isinstance(x, int) else int(x.data_ptr())


class DecodeGraph:
    """A decode step of `num_layers` layers -- per layer, the append of the
    step's new tokens into that layer's pools, then the attention over them --
    captured once per buffer set as a CUDA graph (pkv_decode_graph_create);
    launch(s) replays set s with one launch.  Fill one set while the other
    runs ("ping-pong" buffers).

    k_caches, v_caches: per-layer pools (tensors or device addresses) of
    format `kv_format` and geometry `cache` (a CacheDesc).  sets: two dicts of
    contiguous CUDA tensors: q, out (BF16 [num_layers][num_seqs][q_len][Hq][128]),
    k_new, v_new (BF16 [num_layers][num_tokens][Hkv][128]), slot_mapping
    (int64), block_tables, context_lens (int32), and for a cascade
    group_seqs, group_blocks, seq_prefix_blocks (int32).  cascade: None or a
    dict of num_groups, max_prefix_blocks, max_suffix_blocks and optionally
    prefix_blocks_per_split, suffix_blocks_per_split.  Buffer extents are
    the caller's to get right, as for the direct calls."""

    def __init__(self, k_caches, v_caches, cache: CacheDesc, sets, *, num_seqs: int, q_len: int, num_q_heads: int,
                 max_blocks_per_seq: int, num_tokens: int, scale: float, kv_format: int = KV_BF16,
                 kv_blocks_per_split: int = 0, workspace: torch.Tensor | None = None, cascade: dict | None = None):
        self._handle = None
        if len(sets) != 2 or len(k_caches) != len(v_caches):
            raise ValueError("two buffer sets and one K and one V pool per layer are required")
        n = len(k_caches)
        kc = (ctypes.c_void_p * n)(*[_addr(t) for t in k_caches])
        vc = (ctypes.c_void_p * n)(*[_addr(t) for t in v_caches])
        d = DecodeGraphDesc()
        d.num_layers, d.kv_format, d.cache = n, kv_format, cache
        d.k_caches = ctypes.cast(kc, ctypes.POINTER(ctypes.c_void_p))
        d.v_caches = ctypes.cast(vc, ctypes.POINTER(ctypes.c_void_p))
        d.num_seqs, d.q_len, d.num_q_heads = num_seqs, q_len, num_q_heads
        d.max_blocks_per_seq, d.num_tokens, d.scale = max_blocks_per_seq, num_tokens, scale
        d.kv_blocks_per_split = kv_blocks_per_split
        if cascade:
            d.num_groups = cascade["num_groups"]
            d.max_prefix_blocks = cascade["max_prefix_blocks"]
            d.max_suffix_blocks = cascade["max_suffix_blocks"]
            d.prefix_blocks_per_split = cascade.get("prefix_blocks_per_split", 0)
            d.suffix_blocks_per_split = cascade.get("suffix_blocks_per_split", 0)
        if workspace is not None:
            d.workspace, d.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
        self._keep = [kc, vc, workspace, sets]
        for i, st in enumerate(sets):
            b = d.set[i]
            for name in ("q", "out"):
                _bf16(st[name], f"sets[{i}].{name}")
            for name in ("block_tables", "context_lens") + (
                    ("group_seqs", "group_blocks", "seq_prefix_blocks") if cascade else ()):
                _i32(st[name], f"sets[{i}].{name}")
            if num_tokens > 0:
                _bf16(st["k_new"], f"sets[{i}].k_new")
                _bf16(st["v_new"], f"sets[{i}].v_new")
                if st["slot_mapping"].dtype != torch.int64 or not st["slot_mapping"].is_cuda:
                    raise ValueError(f"sets[{i}].slot_mapping must be a CUDA int64 tensor")
            for name, _ in DecodeGraphBuffers._fields_:
                t = st.get(name)
                if t is not None:
                    setattr(b, name, t.data_ptr())
        h = ctypes.c_void_p()
        _check(_lib.pkv_decode_graph_create(ctypes.byref(d), ctypes.byref(h)), "pkv_decode_graph_create")
        self._handle = h

    def launch(self, buffer_set: int, stream=None) -> None:
        _check(_lib.pkv_decode_graph_launch(self._handle, buffer_set, _stream_ptr(stream)), "pkv_decode_graph_launch")

    def close(self) -> None:
        if self._handle is not None:
            _lib.pkv_decode_graph_destroy(self._handle)
            self._handle = None

    def __del__(self):
        self.close()


def get_device_error(reset: bool = True) -> int:
    """Device error word (DEVERR_* bits) of the current device; synchronises."""
    word = ctypes.c_uint32(0)
    _check(_lib.pkv_get_device_error(ctypes.byref(word), 1 if reset else 0), "pkv_get_device_error")
    return int(word.value)


def selftest_bounded_wait(wait_limit_us: int, arm_all: bool = False, stream=None) -> None:
    """Run the kernels' bounded wait on a barrier that nothing arms (or, with
    arm_all, on armed ones): with nothing arming it the wait gives up after
    wait_limit_us and sets DEVERR_TIMEOUT; read it with get_device_error."""
    _check(_lib.pkv_selftest_bounded_wait(int(wait_limit_us), 1 if arm_all else 0, _stream_ptr(stream)),
           "pkv_selftest_bounded_wait")
