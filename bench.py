#!/usr/bin/env python3
"""Benchmark of paged KV decode attention on GB300.

One step = one decode step of the attention part of a 36-layer model: for
every layer, kv_append of the batch's new tokens, then paged_attention over
the whole batch (split-KV + combine when the library's heuristic splits).
Every layer has its own KV pool, so consecutive layer-calls never find their
KV in L2 (the 36 pools together are far larger than the 129 MB L2).

Prints ONE JSON line (rank 0).  `value` is achieved HBM throughput in GB/s on
the algorithmic bytes: the unique physical KV slots read (a shared-prefix
block counts once), Q and output, the block-table entries and context
lengths read, plus the append's read and write of the new tokens' K/V.

  python bench.py [--workload short|long|mixed|chunk|tiny] [--steps K] [--warmup W]
                  [--kv bf16|q8_0] [--kv-blocks-per-split S] [--graph] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged decode attention µs/layer & achieved HBM GB/s (% of GB300 peak), 1 GPU"
KV_BYTES_PER_TOKEN = 2 * W.NUM_KV_HEADS * W.HEAD_DIM * 2  # K and V of one token in one layer


# ---------------------------------------------------------------------------
# workload selection
# ---------------------------------------------------------------------------

def make_workload(name: str, seed: int, num_seqs: int = 0):
    if name == "short":
        return W.short_chat(seed=seed, fill_cache=False), W.NUM_LAYERS
    if name == "long":
        return W.long_shared(seed=seed, fill_cache=False), W.NUM_LAYERS
    if name == "mixed":
        return W.mixed(seed=seed, fill_cache=False), W.NUM_LAYERS
    if name == "chunk":
        return W.chunk(seed=seed, fill_cache=False, **({"num_seqs": num_seqs} if num_seqs else {})), 1
    if name == "tiny":
        return W.tiny(seed=seed, fill_cache=False), W.NUM_LAYERS
    raise SystemExit(f"unknown workload {name}")


WORKLOAD_TEXT = {
    "short": "short-chat decode: 37 requests x (2048 + U{0..255}) tokens, 36 layers, 12 GiB pool",
    "long": "long-context decode: 16 requests x (8192 + U{0..255}) tokens, 6144-token shared prefix, 36 layers",
    "mixed": "mixed batch: 48 short + 16 long (shared prefix) + 8 requests of 1..15 tokens, 36 layers",
    "chunk": "streaming chunks: 128 requests, q_len 16 causal, history logU[1K,32K], 1 layer (4.8 GB)",
    "tiny": "tiny: 4 requests, contexts {17,64,100,256}, 36 layers",
}


# q8_0 (§8.4.2): 34 bytes per 32 values instead of 64; FP8 (§8.4.4): one byte per value
KV_BYTES_PER_TOKEN_Q8 = KV_BYTES_PER_TOKEN * 34 // 64
KV_BYTES_PER_TOKEN_FP8 = KV_BYTES_PER_TOKEN // 2


def bytes_per_layer(w, kv: str = "bf16"):
    """(attention algorithmic bytes, append bytes) of one layer-call."""
    stored = {"q8_0": KV_BYTES_PER_TOKEN_Q8, "fp8_e4m3": KV_BYTES_PER_TOKEN_FP8}.get(kv, KV_BYTES_PER_TOKEN)
    uniq = w.unique_tokens()
    qo = 2 * w.num_seqs * w.q_len * w.num_q_heads * w.head_dim * 2
    table = sum(-(-int(c) // 16) for c in w.context_lens) * 4 + w.num_seqs * 4
    attn = uniq * stored + qo + table
    t = int((w.slot_mapping >= 0).sum())
    # read the new BF16 K/V, write them in the pool's format, read the slot ids
    append = t * (KV_BYTES_PER_TOKEN + stored) + w.slot_mapping.size * 8
    return attn, append


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        # PKV_CLOCKS_CSV keeps the raw samples where the caller wants them
        self.path = os.environ.get("PKV_CLOCKS_CSV") or f"/tmp/pkv_clocks_{gpu_index}_{os.getpid()}.csv"
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no collective on the data path)
# ---------------------------------------------------------------------------

def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_gbs(world: int, step_bytes: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes one replica of the step; time is the max over ranks."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


def all_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    on_gpu = torch.cuda.is_available() and dist.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, kc_dev, vc_dev, max_seqs: int):
    """Host copies of the blocks `max_seqs` requests read (layer 0), tables remapped."""
    seq_ids = list(range(min(max_seqs, w.num_seqs)))
    need = {}
    for r in seq_ids:
        for b in w.block_tables[r, :-(-int(w.context_lens[r]) // 16)]:
            need.setdefault(int(b), len(need))
    ids = torch.tensor(sorted(need, key=need.get), dtype=torch.long, device=kc_dev.device)
    kc = kc_dev.index_select(0, ids).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    vc = vc_dev.index_select(0, ids).cpu().view(torch.int16).numpy().view(np.uint16).copy()
    tables = np.vectorize(lambda b: need.get(int(b), 0))(w.block_tables[seq_ids]).astype(np.int32)
    sl = w.slot_mapping.reshape(w.num_seqs, w.q_len)[seq_ids].reshape(-1)
    sl = np.array([need[int(s) // 16] * 16 + int(s) % 16 if s >= 0 else -1 for s in sl], np.int64)
    sub = W.Workload(**{**w.__dict__, "k_cache": kc, "v_cache": vc, "block_tables": tables,
                        "context_lens": w.context_lens[seq_ids].copy(), "q": w.q[seq_ids].copy(),
                        "k_new": w.k_new.reshape(w.num_seqs, w.q_len, -1, 128)[seq_ids].reshape(-1, w.num_kv_heads, 128),
                        "v_new": w.v_new.reshape(w.num_seqs, w.q_len, -1, 128)[seq_ids].reshape(-1, w.num_kv_heads, 128),
                        "slot_mapping": sl})
    return sub


def oracle_sample_q8(w, kq_dev, vq_dev, max_seqs: int):
    """oracle_sample for quantised pools: host copies of the tiles the sampled requests read."""
    seq_ids = list(range(min(max_seqs, w.num_seqs)))
    need = {}
    for r in seq_ids:
        for b in w.block_tables[r, :-(-int(w.context_lens[r]) // 16)]:
            need.setdefault(int(b), len(need))
    ids = torch.tensor(sorted(need, key=need.get), dtype=torch.long, device=kq_dev.device)
    kq = kq_dev.index_select(0, ids).cpu().numpy().copy()
    vq = vq_dev.index_select(0, ids).cpu().numpy().copy()
    tables = np.vectorize(lambda b: need.get(int(b), 0))(w.block_tables[seq_ids]).astype(np.int32)
    sl = w.slot_mapping.reshape(w.num_seqs, w.q_len)[seq_ids].reshape(-1)
    sl = np.array([need[int(s) // 16] * 16 + int(s) % 16 if s >= 0 else -1 for s in sl], np.int64)
    sub = W.Workload(**{**w.__dict__, "k_cache": None, "v_cache": None, "block_tables": tables,
                        "context_lens": w.context_lens[seq_ids].copy(), "q": w.q[seq_ids].copy(),
                        "k_new": w.k_new.reshape(w.num_seqs, w.q_len, -1, 128)[seq_ids].reshape(-1, w.num_kv_heads, 128),
                        "v_new": w.v_new.reshape(w.num_seqs, w.q_len, -1, 128)[seq_ids].reshape(-1, w.num_kv_heads, 128),
                        "slot_mapping": sl})
    return sub, kq, vq


def time_oracle_q8(sub, kq, vq, budget_s: float = 12.0, max_reps: int = 200, kv: str = "q8_0",
                   num_threads: int = 0):
    """The oracle's quantising append, dequantisation and FP64 attention on the sample."""
    import oracle
    attn_b, app_b = bytes_per_layer(sub, kv)
    append = oracle.kv_append_q8_0 if kv == "q8_0" else oracle.kv_append_fp8
    deq = oracle.dequantize_q8_0 if kv == "q8_0" else oracle.dequantize_fp8
    reps, t0 = 0, time.perf_counter()
    while True:
        append(kq, vq, sub.slot_mapping, sub.k_new, sub.v_new)
        oracle.paged_attention_f64(sub.q, deq(kq), deq(vq), sub.block_tables, sub.context_lens, 1, sub.scale,
                                   num_threads=num_threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    per = el / reps
    return {"gbs": (attn_b + app_b) / per / 1e9, "s_per_layer_call": per, "reps": reps,
            "cores": num_threads or oracle.max_threads(), "seqs": sub.num_seqs}


def time_oracle(sub, budget_s: float = 12.0, max_reps: int = 200, num_threads: int = 0):
    """Run the oracle's append + attention on the sample until ~budget_s; GB/s
    of algorithmic bytes.  num_threads 0 = all host cores."""
    import oracle
    attn_b, app_b = bytes_per_layer(sub)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.kv_append(sub.k_cache, sub.v_cache, sub.slot_mapping, sub.k_new, sub.v_new)
        oracle.paged_attention(sub.q, sub.k_cache, sub.v_cache, sub.block_tables, sub.context_lens, sub.q_len,
                               sub.scale, num_threads=num_threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    per = el / reps
    return {"gbs": (attn_b + app_b) / per / 1e9, "s_per_layer_call": per, "reps": reps,
            "cores": num_threads or oracle.max_threads(), "seqs": sub.num_seqs}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="short", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-blocks-per-split", type=int, default=0)
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=True,
                    help="replay each 36-layer step as one CUDA graph (default on)")
    ap.add_argument("--prefix-blocks-per-split", type=int, default=0, help="cascade prefix pass split (0 = plan)")
    ap.add_argument("--suffix-blocks-per-split", type=int, default=0, help="cascade suffix pass split (0 = plan)")
    ap.add_argument("--no-cascade", action="store_true",
                    help="shared-prefix workloads: plain paged attention instead of the cascade call")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "q8_0", "fp8_e4m3"],
                    help="KV pool format: bf16, q8_0 or fp8_e4m3 (the last two: decode only)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--oracle-budget-s", type=float, default=12.0)
    ap.add_argument("--kernel-pass-s", type=float, default=1.0,
                    help="GPU seconds of the sustained kernel-timing pass (at least --steps replays)")
    ap.add_argument("--per-config", action=argparse.BooleanOptionalAction, default=True,
                    help="default short-chat run: also time the long, mixed and chunk workloads")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--num-seqs", type=int, default=0, help="chunk workload: fewer requests (small profiling cases)")
    ap.add_argument("--sweep", action="store_true", help="q_len-1 batch x context sweep instead of a step benchmark")
    ap.add_argument("--sweep-batches", default="", help="comma list (default 1..512, powers of two)")
    ap.add_argument("--sweep-contexts", default="", help="comma list (default 128..65536, powers of two)")
    ap.add_argument("--sweep-reps", type=int, default=10)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.sweep:
        return run_sweep(args)
    world, rank, local = dist_init(args.gpus)
    if args.impl == "reference":
        w, layers = make_workload(args.workload, args.seed, args.num_seqs)
        if args.layers > 0:
            layers = args.layers
        attn_b, app_b = bytes_per_layer(w, args.kv)
        return run_reference(args, world, rank, w, layers, layers * (attn_b + app_b))
    line = bench_one(args, args.workload, world, rank, local, headline=True)
    # the other decode targets in the same run (the default run only): the
    # long shared-prefix batch, the mixed batch and the streaming chunks,
    # each with its own timing, roofline and clocks
    if args.per_config and args.workload == "short" and args.kv == "bf16" and args.layers == 0:
        per = {}
        for name in PER_CONFIG:
            gc.collect()  # the previous workload's pools
            torch.cuda.empty_cache()
            r = bench_one(args, name, world, rank, local, headline=False)
            if r is not None:
                per[name] = {k: r[k] for k in ("ms_per_step", "us_per_layer_call", "us_per_layer_call_isolated",
                                               "value", "bytes_per_step", "attention_tokens_layers_per_s",
                                               "decode_steps_per_s", "roofline", "clocks", "clocks_kernel_pass",
                                               "launch")}
                per[name]["workload"] = r["config"]["workload"]
                per[name]["unit"] = "GB/s"
        if line is not None:
            line["per_config"] = per
    if line is not None:
        print(json.dumps(line), flush=True)


# the other configurations the default run measures beside the headline
PER_CONFIG = ("long", "mixed", "chunk")


def l2_text(w, layers: int, kv: str) -> str:
    """How the timed loop keeps KV out of L2 (the same text for both arms)."""
    tile = {"q8_0": 2176, "fp8_e4m3": 2048}.get(kv, 4096)
    return "inputs larger than L2: one KV pool per layer, %.1f GB total" % (
        2 * layers * w.num_blocks * W.NUM_KV_HEADS * tile / 1e9)


def bench_one(args, name: str, world: int, rank: int, local: int, headline: bool):
    """Benchmark one workload; returns the JSON line's dict on rank 0 (None
    elsewhere).  headline: also the end-to-end leg and the CPU baseline."""
    w, layers = make_workload(name, args.seed, args.num_seqs if headline else 0)
    if args.layers > 0 and headline:
        layers = args.layers
    q8 = args.kv in ("q8_0", "fp8_e4m3")  # a quantised pool (q8_0 or E4M3)
    fp8 = args.kv == "fp8_e4m3"
    if q8 and w.q_len != 1:
        raise SystemExit(f"--kv {args.kv} is a decode (q_len 1) path")
    attn_b, app_b = bytes_per_layer(w, args.kv)
    step_bytes = layers * (attn_b + app_b)
    tokens_layers = int(w.context_lens.sum()) * w.q_len * layers if w.q_len > 1 else int(w.context_lens.sum()) * layers

    import paged_kv_decode_attention_gb300 as pkv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = pkv.lib()
    b, ql, hq, hkv, d = w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim
    maxb = w.max_blocks_per_seq
    if q8:
        choose = pkv.choose_kv_blocks_per_split_fp8_e4m3 if fp8 else pkv.choose_kv_blocks_per_split_q8_0
        bps = args.kv_blocks_per_split or choose(b, hkv, maxb)
    else:
        bps = args.kv_blocks_per_split or pkv.choose_kv_blocks_per_split(b, hkv, ql, maxb)
    bps = min(bps, maxb)
    splits = -(-maxb // bps)

    # device state: per-layer pools (filled on the device), per-layer step inputs/outputs
    if q8:
        # BF16 values drawn on the device, quantised into each layer's q8_0 pool by the library's append
        tile_shape = (16, d) if fp8 else (pkv.Q8_TILE_BYTES,)
        k_pool = torch.empty((layers, w.num_blocks, hkv) + tile_shape, dtype=torch.uint8, device=dev)
        v_pool = torch.empty_like(k_pool)
        tmp_k = torch.empty((w.num_blocks, hkv, 16, d), dtype=torch.bfloat16, device=dev)
        tmp_v = torch.empty_like(tmp_k)
        all_slots = torch.arange(w.num_blocks * 16, dtype=torch.int64, device=dev)
        tok = lambda p: p.permute(0, 2, 1, 3).contiguous().view(w.num_blocks * 16, hkv, d)
        for l in range(layers):
            W.fill_pool_device(tmp_k, 1000 + 2 * l + args.seed * 7919)
            W.fill_pool_device(tmp_v, 1001 + 2 * l + args.seed * 7919)
            (pkv.kv_append_fp8_e4m3 if fp8 else pkv.kv_append_q8_0)(k_pool[l], v_pool[l], all_slots, tok(tmp_k),
                                                                    tok(tmp_v))
        del tmp_k, tmp_v, all_slots
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    else:
        pool_shape = (layers, w.num_blocks, hkv, 16, d)
        k_pool = torch.empty(pool_shape, dtype=torch.bfloat16, device=dev)
        v_pool = torch.empty(pool_shape, dtype=torch.bfloat16, device=dev)
        for l in range(layers):
            W.fill_pool_device(k_pool[l], 1000 + 2 * l + args.seed * 7919)
            W.fill_pool_device(v_pool[l], 1001 + 2 * l + args.seed * 7919)
    rng = np.random.Generator(np.random.PCG64(args.seed + 17))
    t_tok = w.slot_mapping.size
    h_q = torch.from_numpy(W.randn_bf16(rng, (layers, b, ql, hq, d))).view(torch.bfloat16)
    h_kn = torch.from_numpy(W.randn_bf16(rng, (layers, t_tok, hkv, d))).view(torch.bfloat16)
    h_vn = torch.from_numpy(W.randn_bf16(rng, (layers, t_tok, hkv, d))).view(torch.bfloat16)
    h_q[0] = torch.from_numpy(w.q).view(torch.bfloat16)
    h_kn[0] = torch.from_numpy(w.k_new).view(torch.bfloat16)
    h_vn[0] = torch.from_numpy(w.v_new).view(torch.bfloat16)
    h_tables = torch.from_numpy(w.block_tables)
    h_ctx = torch.from_numpy(w.context_lens)
    h_slots = torch.from_numpy(w.slot_mapping)
    q = h_q.to(dev)
    kn, vn = h_kn.to(dev), h_vn.to(dev)
    tables, ctx, slots = h_tables.to(dev), h_ctx.to(dev), h_slots.to(dev)
    out = torch.empty_like(q)
    ws_bytes = pkv.workspace_size_q8_0(b, hq, maxb, bps) if q8 else pkv.workspace_size(b, ql, hq, maxb, bps)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    desc = pkv.CacheDesc(w.num_blocks, 16, hkv, d)
    stream = torch.cuda.Stream(dev)  # non-default: CUDA graphs can be captured on it
    torch.cuda.set_stream(stream)
    sp = stream.cuda_stream
    pool_stride = w.num_blocks * hkv * (pkv.FP8_TILE_BYTES if fp8 else pkv.Q8_TILE_BYTES if q8 else 16 * d * 2)
    kp0, vp0 = k_pool.data_ptr(), v_pool.data_ptr()
    q_stride, kn_stride = b * ql * hq * d * 2, t_tok * hkv * d * 2
    # append + attention (+ the combine pass when splits go through the workspace: more than 8
    # splits, or any split on the tensor-core paths -- chunks, quantised pools and q_len-1 batches
    # of at least 2 (request, KV head) rows per SM)
    tc_decode = decode_on_tensor_cores(b, hkv, ql, maxb, torch.cuda.get_device_properties(dev).multi_processor_count)
    launches_per_layer = 1 + 1 + (1 if (splits > 8 or (splits > 1 and (ql >= 16 or q8 or tc_decode))) else 0)
    # shared prefixes: the caller states the groups and the cascade call reads each prefix once per group
    gs_h, gb_h, sp_h = W.prefix_groups(w)
    cascade = (not args.no_cascade) and gs_h.shape[0] > 0 and ql == 1 and not q8
    if cascade:
        maxp = int(gb_h.max())
        maxs = W.max_suffix_blocks(w, sp_h)
        pbps, sbps = pkv.cascade_plan(b, hkv, gs_h.shape[0], maxp, maxs)
        pbps = args.prefix_blocks_per_split or pbps
        sbps = args.suffix_blocks_per_split or sbps
        cws = torch.empty(max(256, pkv.cascade_workspace_size(b, hq, maxp, maxs, pbps, sbps)), dtype=torch.uint8,
                          device=dev)
        gs_d, gb_d, sp_d = (torch.from_numpy(x).to(dev) for x in (gs_h, gb_h, sp_h))
        splits = -(-maxp // pbps) + -(-maxs // sbps)
        # append, prefix pass, suffix decode (+ the combine pass past 8 suffix splits)
        launches_per_layer = 1 + 2 + (1 if -(-maxs // sbps) > 8 else 0)

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {lib.pkv_status_string(st).decode()}")

    def layer_call(l, ev=None):
        append = lib.pkv_kv_append_fp8_e4m3 if fp8 else lib.pkv_kv_append_q8_0 if q8 else lib.pkv_kv_append
        check(append(kp0 + l * pool_stride, vp0 + l * pool_stride, ctypes.byref(desc), slots.data_ptr(),
                     kn.data_ptr() + l * kn_stride, vn.data_ptr() + l * kn_stride, t_tok, sp), "kv_append")
        if ev is not None:
            ev[0].record(stream)
        attention_call(l)
        if ev is not None:
            ev[1].record(stream)

    def attention_call(l):
        if q8:
            attn = lib.pkv_paged_attention_fp8_e4m3 if fp8 else lib.pkv_paged_attention_q8_0
            check(attn(out.data_ptr() + l * q_stride, q.data_ptr() + l * q_stride, kp0 + l * pool_stride,
                       vp0 + l * pool_stride, ctypes.byref(desc), tables.data_ptr(), maxb, ctx.data_ptr(), b, hq,
                       w.scale, bps, ws.data_ptr(), ws.numel(), sp), "paged_attention_" + args.kv)
        elif cascade:
            check(lib.pkv_paged_attention_cascade(
                out.data_ptr() + l * q_stride, q.data_ptr() + l * q_stride, kp0 + l * pool_stride,
                vp0 + l * pool_stride, ctypes.byref(desc), tables.data_ptr(), maxb, ctx.data_ptr(), b, hq, w.scale,
                gs_d.data_ptr(), gb_d.data_ptr(), sp_d.data_ptr(), gs_h.shape[0], maxp, maxs, pbps, sbps, cws.data_ptr(),
                cws.numel(), sp), "paged_attention_cascade")
        else:
            check(lib.pkv_paged_attention(out.data_ptr() + l * q_stride, q.data_ptr() + l * q_stride,
                                          kp0 + l * pool_stride, vp0 + l * pool_stride, ctypes.byref(desc),
                                          tables.data_ptr(), maxb, ctx.data_ptr(), b, ql, hq, w.scale, bps,
                                          ws.data_ptr(), ws.numel(), sp), "paged_attention")

    def step(events=None):
        for l in range(layers):
            layer_call(l, None if events is None else events[l])

    # the step as the library's decode graph: one CUDA graph per buffer set
    # (set 0 = the buffers above, set 1 = a second copy for the end-to-end
    # leg's ping-pong), each the layers' append + attention calls
    graph = None
    sets_dev = None
    if args.graph:
        sets_dev = [dict(q=q, k_new=kn, v_new=vn, slot_mapping=slots, block_tables=tables, context_lens=ctx, out=out)]
        sets_dev.append({k: v.clone() for k, v in sets_dev[0].items()})
        if cascade:
            for st_ in sets_dev:
                st_.update(group_seqs=gs_d.clone(), group_blocks=gb_d.clone(), seq_prefix_blocks=sp_d.clone())
        graph = pkv.DecodeGraph(
            [kp0 + l * pool_stride for l in range(layers)], [vp0 + l * pool_stride for l in range(layers)], desc,
            sets_dev, num_seqs=b, q_len=ql, num_q_heads=hq, max_blocks_per_seq=maxb, num_tokens=t_tok,
            scale=w.scale, kv_format=pkv.KV_FP8_E4M3 if fp8 else pkv.KV_Q8_0 if q8 else pkv.KV_BF16,
            kv_blocks_per_split=bps, workspace=cws if cascade else ws,
            cascade={"num_groups": int(gs_h.shape[0]), "max_prefix_blocks": maxp, "max_suffix_blocks": maxs,
                     "prefix_blocks_per_split": pbps, "suffix_blocks_per_split": sbps} if cascade else None)
        run_step = lambda events=None: graph.launch(0, stream)
        if ql == 1 and t_tok == b and (q8 or cascade or not tc_decode):
            launches_per_layer -= 1  # the graph's decode layers fuse the append into the attention
    else:
        run_step = step

    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    if pkv.get_device_error(reset=True) != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- timed region: whole steps, device events on the launching stream ----
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        run_step()
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms_total = all_max(t_start.elapsed_time(t_end), world)
    ms_per_step = ms_total / args.steps
    if pkv.get_device_error(reset=True) != 0:
        raise RuntimeError("device error word set during the timed region")

    # ---- kernel timing: a second timed pass with an event pair around every attention call ----
    # (kept apart from the step timing above: events between launches cost the
    # overlap programmatic dependent launch gives, so they would lower `value`)
    attn_events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(layers)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s in range(args.steps):
        step(attn_events[s])
    torch.cuda.synchronize()
    attn_ms = [e[0].elapsed_time(e[1]) for st in attn_events for e in st]
    attn_us_isolated = statistics.mean(attn_ms) * 1e3
    if pkv.get_device_error(reset=True) != 0:
        raise RuntimeError("device error word set during the kernel-timing pass")

    # ---- kernel timing, sustained: the layers' attention calls alone, back to
    # back in one CUDA graph as in the step (launch gaps hidden by programmatic
    # dependent launch; each call still waits for the previous one before it
    # reads its inputs), timed with one event pair over K replays ----
    attn_us = attn_us_isolated
    clk_kernel = None
    sustained = graph is not None
    if sustained:
        def attention_layers():
            for l in range(layers):
                attention_call(l)
        attention_layers()
        torch.cuda.synchronize()
        attn_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(attn_graph, stream=stream):
            attention_layers()
        for _ in range(args.warmup):
            attn_graph.replay()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        # as many replays as fill about args.kernel_pass_s of GPU time (K at
        # least), so that the clock samples taken meanwhile carry weight
        a0.record(stream)
        for _ in range(3):
            attn_graph.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        reps = max(args.steps, int(math.ceil(args.kernel_pass_s * 1e3 / max(a0.elapsed_time(a1) / 3, 1e-3))))
        kclocks = ClockSampler(local)
        kclocks.start()
        a0.record(stream)
        for _ in range(reps):
            attn_graph.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        clk_kernel = kclocks.stop()
        if clk_kernel is not None:
            clk_kernel["replays"] = reps
        attn_us = a0.elapsed_time(a1) * 1e3 / (reps * layers)
        if pkv.get_device_error(reset=True) != 0:
            raise RuntimeError("device error word set during the sustained kernel-timing pass")

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if headline and not args.no_e2e:
        p_q, p_kn, p_vn = h_q.pin_memory(), h_kn.pin_memory(), h_vn.pin_memory()
        p_tables, p_ctx, p_slots = h_tables.pin_memory(), h_ctx.pin_memory(), h_slots.pin_memory()
        p_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (p_q, p_kn, p_vn, p_tables, p_ctx, p_slots))
        d2h = p_out.numel() * p_out.element_size()

        def e2e_run_graph(n_steps):
            """The decode loop with the two buffer sets: step n runs set n % 2
            while the copy stream uploads step n + 1's inputs into the other
            set and reads step n's output back; the host waits for step n - 1's
            output before enqueueing step n + 1 (at most two steps in flight)."""
            copy = e2e_copy_stream
            copy.wait_stream(stream)
            for n in range(n_steps):
                s_ = n & 1
                st_ = sets_dev[s_]
                if n == 0:
                    with torch.cuda.stream(copy):
                        for name, src in pinned_in:
                            st_[name].copy_(src, non_blocking=True)
                        ev_in[0].record(copy)
                stream.wait_event(ev_in[s_])
                graph.launch(s_, stream)
                ev_done[s_].record(stream)
                with torch.cuda.stream(copy):
                    if n + 1 < n_steps:
                        if n >= 1:
                            copy.wait_event(ev_done[1 - s_])  # the other set's last step is done
                        for name, src in pinned_in:
                            sets_dev[1 - s_][name].copy_(src, non_blocking=True)
                        ev_in[1 - s_].record(copy)
                    copy.wait_event(ev_done[s_])
                    p_outs[s_].copy_(st_["out"], non_blocking=True)
                    ev_out[s_].record(copy)
                if n >= 1:
                    ev_out[1 - s_].synchronize()  # step n - 1's result is on the host
            ev_out[(n_steps - 1) & 1].synchronize()

        def e2e_step():
            for dst, src in ((q, p_q), (kn, p_kn), (vn, p_vn), (tables, p_tables), (ctx, p_ctx), (slots, p_slots)):
                dst.copy_(src, non_blocking=True)
            for l in range(layers):
                if q8:
                    (pkv.kv_append_fp8_e4m3 if fp8 else pkv.kv_append_q8_0)(k_pool[l], v_pool[l], slots, kn[l], vn[l])
                    (pkv.paged_attention_fp8_e4m3 if fp8 else pkv.paged_attention_q8_0)(
                        out[l], q[l], k_pool[l], v_pool[l], tables, ctx, w.scale, kv_blocks_per_split=bps,
                        workspace=ws)
                    continue
                pkv.kv_append(k_pool[l], v_pool[l], slots, kn[l], vn[l])
                if cascade:
                    pkv.paged_attention_cascade(out[l], q[l], k_pool[l], v_pool[l], tables, ctx, w.scale, gs_d, gb_d,
                                                sp_d, maxp, maxs, cws, pbps, sbps)
                else:
                    pkv.paged_attention(out[l], q[l], k_pool[l], v_pool[l], tables, ctx, ql, w.scale,
                                        kv_blocks_per_split=bps, workspace=ws)
            p_out.copy_(out, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        if graph is not None:
            e2e_copy_stream = torch.cuda.Stream(dev)
            pinned_in = [("q", p_q), ("k_new", p_kn), ("v_new", p_vn), ("block_tables", p_tables),
                         ("context_lens", p_ctx), ("slot_mapping", p_slots)]
            p_outs = [p_out, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
            ev_in = [torch.cuda.Event(), torch.cuda.Event()]
            ev_done = [torch.cuda.Event(), torch.cuda.Event()]
            ev_out = [torch.cuda.Event(), torch.cuda.Event()]
            e2e_run_graph(2)
            torch.cuda.synchronize()
            barrier(world)
            t0 = time.perf_counter()
            e2e_run_graph(args.steps)
            torch.cuda.synchronize()
            el = all_max(time.perf_counter() - t0, world)
        else:
            for _ in range(2):
                e2e_step()
            barrier(world)
            t0 = time.perf_counter()
            for _ in range(args.steps):
                e2e_step()
            el = all_max(time.perf_counter() - t0, world)
        e2e = {"value": round(world * step_bytes / (el / args.steps) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(el / args.steps * 1e3, 4), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h)}

    # ---- CPU oracle baseline (rank 0 at N=1 only) ----
    cpu = None
    if headline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        if q8:
            sub, kq_h, vq_h = oracle_sample_q8(w, k_pool[0], v_pool[0], max_seqs=w.num_seqs)
            r = time_oracle_q8(sub, kq_h, vq_h, budget_s=args.oracle_budget_s, kv=args.kv)
            sub1, kq1, vq1 = oracle_sample_q8(w, k_pool[0], v_pool[0], max_seqs=2)
            r1 = time_oracle_q8(sub1, kq1, vq1, budget_s=args.oracle_budget_s / 2, kv=args.kv, num_threads=1)
        else:
            sub = oracle_sample(w, k_pool[0], v_pool[0], max_seqs=w.num_seqs)
            r = time_oracle(sub, budget_s=args.oracle_budget_s)
            sub1 = oracle_sample(w, k_pool[0], v_pool[0], max_seqs=2)
            r1 = time_oracle(sub1, budget_s=args.oracle_budget_s / 2, num_threads=1)
        cpu = {"value": round(r["gbs"], 4), "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
               "sample": f"layer 0 of this workload ({r['seqs']} requests, append + attention), FP64 C oracle, "
                         f"{r['reps']} repetitions, {r['s_per_layer_call'] * 1e3:.1f} ms per layer-call",
               "single_core": {"value": round(r1["gbs"], 4), "unit": "GB/s", "cores": 1,
                               "sample": f"layer 0, requests 0-{r1['seqs'] - 1} of this workload (append + "
                                         f"attention), FP64 C oracle on one thread, {r1['reps']} repetitions, "
                                         f"{r1['s_per_layer_call'] * 1e3:.1f} ms per sample"}}

    if graph is not None:
        graph.close()
    if rank != 0:
        return None
    peaks = {}
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        peaks = json.load(open(pp))
    peak = peaks.get("hbm_gbs")
    peak_src = "measured"
    if not peak:
        peak, peak_src = 6800.0, "fallback"
    achieved = attn_b / (attn_us * 1e-6) / 1e9
    value = aggregate_gbs(world, step_bytes, ms_per_step)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath)).get(name + ("_" + args.kv if q8 else ""))
        if tj and tj.get("kernel_build") == kernel_build_id():
            traffic = tj.get("bytes_per_launch")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("fp8_e4m3 KV, e4m3 tensor-core Q.K and P.V (query and weights as e4m3 high + low parts), "
                  "f32 accumulation and softmax" if fp8 else
                  f"{args.kv} KV, f16 tensor-core Q.K, f32 softmax and P.V" if q8 else "bf16"),
        "data": "synthetic",
        "config": workload_config(name, w, layers, args.kv, world),
        "launch": {"kv_blocks_per_split": bps, "splits": splits, "cuda_graph": bool(graph is not None),
                   "cascade": ({"groups": int(gs_h.shape[0]), "prefix_blocks": maxp, "max_suffix_blocks": maxs,
                                "prefix_blocks_per_split": pbps,
                                "suffix_blocks_per_split": sbps} if cascade else None)},
        "us_per_layer_call": round(attn_us, 3),
        "us_per_layer_call_isolated": round(attn_us_isolated, 3),
        "attention_tokens_layers_per_s": round(world * tokens_layers / (ms_per_step * 1e-3), 1),
        "decode_steps_per_s": round(1e3 / ms_per_step, 2),
        "bytes_per_step": int(step_bytes),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_src,
                     "kernel": ("paged_attention_%s call (%s%s)" % (
                                    args.kv, "8-bit tensor-core decode" if fp8 else "tensor-core dequantising decode",
                                    " + combine" if splits > 1 else "") if q8 else
                                "paged_attention_cascade call (prefix tensor-core pass + suffix decode + combine)"
                                if cascade else "paged_attention call (%s%s)" % (
                                    "tensor-core chunk" if ql >= 16 else "decode",
                                    " + combine" if (splits > 8 or (ql >= 16 and splits > 1)) else "")),
                     "algorithmic_bytes_per_launch": int(attn_b),
                     "timing": ("sustained: one CUDA event pair over K replays of a graph of the %d layers' "
                                "attention calls alone, divided by the calls; us_per_layer_call_isolated = mean "
                                "event time of each call with events around it, launch gaps included" % layers)
                     if sustained else "mean CUDA-event time of the call over a second timed pass of the same steps"},
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(launches_per_layer * layers * args.steps),
        "clocks": clk,
        "clocks_kernel_pass": clk_kernel,
    }
    return line


def workload_config(name: str, w, layers: int, kv: str, world: int) -> dict:
    """The JSON line's `config`: the workload alone (both arms report the same)."""
    return {"workload": WORKLOAD_TEXT[name], "name": name, "num_seqs": w.num_seqs, "q_len": w.q_len,
            "layers": layers, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": 16, "ctx_min": int(w.context_lens.min()), "ctx_max": int(w.context_lens.max()),
            "kv_format": kv, "l2": l2_text(w, layers, kv), "parallelism": f"replicas x{world}"}


def quantised_pools(pkv, kv: str, nb: int, seed: int, dev, chunk: int = 4096):
    """K and V pools of `nb` blocks in the q8_0 or E4M3 format, every slot
    holding N(0,1) BF16 values stored through the format's append, filled
    `chunk` blocks at a time so the BF16 staging stays small."""
    fp8 = kv == "fp8_e4m3"
    tile = (16, 128) if fp8 else (pkv.Q8_TILE_BYTES,)
    kq = torch.empty((nb, 8) + tile, dtype=torch.uint8, device=dev)
    vq = torch.empty_like(kq)
    append = pkv.kv_append_fp8_e4m3 if fp8 else pkv.kv_append_q8_0
    tk = torch.empty((min(chunk, nb), 8, 16, 128), dtype=torch.bfloat16, device=dev)
    tv = torch.empty_like(tk)
    for c0 in range(0, nb, chunk):
        n = min(chunk, nb - c0)
        W.fill_pool_device(tk[:n], seed * 7919 + 2 * c0)
        W.fill_pool_device(tv[:n], seed * 7919 + 2 * c0 + 1)
        slots = torch.arange(c0 * 16, (c0 + n) * 16, dtype=torch.int64, device=dev)
        append(kq, vq, slots, tk[:n].permute(0, 2, 1, 3).contiguous().view(n * 16, 8, 128),
               tv[:n].permute(0, 2, 1, 3).contiguous().view(n * 16, 8, 128))
    return kq, vq


def decode_on_tensor_cores(num_seqs: int, num_kv_heads: int, q_len: int, max_blocks: int, sms: int) -> bool:
    """The library's choice of the persistent tensor-core decode (pkv_api.cu),
    restated to count the step's launches: from 2 (request, KV head) rows per
    SM, or from 3/4 of a row per SM with requests of >= 128 blocks when the
    CTA-per-row kernel's one wave of 2 CTAs per SM would fill < 90 % of it."""
    if q_len != 1:
        return False
    rows, slots = num_seqs * num_kv_heads, 2 * sms
    if rows >= 2 * sms:
        return True
    if 4 * rows < 3 * sms or max_blocks < 128:
        return False
    splits = slots // rows
    bps = max_blocks if (max_blocks <= 16 or splits <= 1) else min(max(16, -(-max_blocks // splits)), max_blocks)
    return 10 * rows * (-(-max_blocks // bps)) < 9 * slots


def run_sweep(args):
    """q_len-1 stress sweep: batch x context grid, one layer, default split;
    L2 flushed (a 256 MiB write) before every timed call so small points are
    read from HBM too, then a 256 MiB read evicts the flush's dirty lines so
    their write-back is not charged to the call, and a device-side delay
    covers the host's launch of the call so the events time the device work.
    Prints one JSON line with every point."""
    import paged_kv_decode_attention_gb300 as pkv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    drain = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MiB read after the flush
    free, _ = torch.cuda.mem_get_info(dev)
    quant = args.kv in ("q8_0", "fp8_e4m3")
    fp8 = args.kv == "fp8_e4m3"
    batches = [int(x) for x in args.sweep_batches.split(",")] if args.sweep_batches else W.SWEEP_BATCHES
    contexts = [int(x) for x in args.sweep_contexts.split(",")] if args.sweep_contexts else W.SWEEP_CONTEXTS
    peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("hbm_gbs", 6800.0) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else 6800.0
    points = []
    for b in batches:
        for c in contexts:
            nb = b * (-(-c // 16)) + 8
            pool_bytes = 2 * nb * 8 * 16 * 128 * 2
            if pool_bytes > 0.8 * free:
                points.append({"batch": b, "ctx": c, "skipped": "pool larger than free device memory"})
                continue
            w = W.build(f"sweep", [c] * b, nb, seed=b * 7919 + c, fill_cache=False)
            if quant:  # N(0,1) values through the format's append, a chunk of blocks at a time
                kc, vc = quantised_pools(pkv, args.kv, nb, 2 * b + 1, dev)
            else:
                kc = torch.empty((nb, 8, 16, 128), dtype=torch.bfloat16, device=dev)
                vc = torch.empty_like(kc)
                W.fill_pool_device(kc, 2 * b + 1)
                W.fill_pool_device(vc, 2 * b + 2)
            q = torch.from_numpy(w.q).view(torch.bfloat16).to(dev)
            tables = torch.from_numpy(w.block_tables).to(dev)
            ctx = torch.from_numpy(w.context_lens).to(dev)
            out = torch.empty_like(q)
            maxb = w.max_blocks_per_seq
            if quant:
                choose = pkv.choose_kv_blocks_per_split_fp8_e4m3 if fp8 else pkv.choose_kv_blocks_per_split_q8_0
                bps = choose(b, 8, maxb)
                ws = torch.empty(max(256, pkv.workspace_size_q8_0(b, 32, maxb, bps)), dtype=torch.uint8, device=dev)
            else:
                bps = pkv.choose_kv_blocks_per_split(b, 8, 1, maxb)
                ws = torch.empty(max(256, pkv.workspace_size(b, 1, 32, maxb, bps)), dtype=torch.uint8, device=dev)
            times = []
            for it in range(args.warmup + args.sweep_reps):
                flush.fill_(it & 0xFF)
                drain.sum()
                torch.cuda._sleep(200000)  # ~100 us: the call below is enqueued before the GPU reaches it
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if quant:
                    (pkv.paged_attention_fp8_e4m3 if fp8 else pkv.paged_attention_q8_0)(
                        out, q, kc, vc, tables, ctx, w.scale, kv_blocks_per_split=bps, workspace=ws)
                else:
                    pkv.paged_attention(out, q, kc, vc, tables, ctx, 1, w.scale, kv_blocks_per_split=bps,
                                        workspace=ws)
                e1.record(stream)
                e1.synchronize()
                if it >= args.warmup:
                    times.append(e0.elapsed_time(e1))
            us = statistics.median(times) * 1e3
            attn_b, _ = bytes_per_layer(w, args.kv)
            points.append({"batch": b, "ctx": c, "us": round(us, 2), "gbs": round(attn_b / (us * 1e-6) / 1e9, 1),
                           "frac": round(attn_b / (us * 1e-6) / 1e9 / peak, 4), "splits": -(-maxb // bps)})
            del kc, vc, q, out, ws
            torch.cuda.empty_cache()
    if pkv.get_device_error(reset=True) != 0:
        raise RuntimeError("device error word set during the sweep")
    print(json.dumps({"metric": "paged decode attention sweep (q_len 1, one layer, L2 flushed)", "kv_format": args.kv,
                      "peak_gbs": peak,
                      "reps": args.sweep_reps, "points": points}), flush=True)


def kernel_build_id() -> str:
    """Hash of the CUDA sources' code (comments and blank space left out):
    traffic numbers are valid only for the code they were taken on."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_attention_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, fn), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(fn.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def run_reference(args, world, rank, w, layers, step_bytes):
    """Reference arm: the FP64 CPU oracle, as it stands, on the host cores;
    each step is a bounded sample (some requests of one layer) of the workload."""
    if rank != 0:
        return
    import oracle
    # build a host pool for a bounded sample of requests
    max_seqs = max(1, min(w.num_seqs, 8))
    sub = W.build("sample", w.context_lens[:max_seqs], int(sum(-(-int(c) // 16) for c in w.context_lens[:max_seqs])) + 8,
                  q_len=w.q_len, seed=args.seed)
    attn_b, app_b = bytes_per_layer(sub)
    for _ in range(args.warmup):
        oracle.kv_append(sub.k_cache, sub.v_cache, sub.slot_mapping, sub.k_new, sub.v_new)
        oracle.paged_attention(sub.q, sub.k_cache, sub.v_cache, sub.block_tables, sub.context_lens, sub.q_len,
                               sub.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kv_append(sub.k_cache, sub.v_cache, sub.slot_mapping, sub.k_new, sub.v_new)
        oracle.paged_attention(sub.q, sub.k_cache, sub.v_cache, sub.block_tables, sub.context_lens, sub.q_len,
                               sub.scale)
    el = (time.perf_counter() - t0) / args.steps
    value = (attn_b + app_b) / el / 1e9
    sample = (f"{max_seqs} of {w.num_seqs} requests of one layer of the {args.workload} workload "
              f"(append + attention) per step, FP64 C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, w, layers, args.kv, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.max_threads(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
