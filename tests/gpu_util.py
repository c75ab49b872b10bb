"""Helpers shared by the GPU tests: move a workloads.Workload to the device
and compare results with the oracle's FP64 output."""
import numpy as np
import torch

MAX_ABS = 1e-2   # attention tolerance against the FP64 oracle (BF16 inputs, FP32 math)
REL_L2 = 5e-3


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def to_device(w):
    d = {
        "q": dev(w.q),
        "block_tables": dev(w.block_tables),
        "context_lens": dev(w.context_lens),
        "slot_mapping": dev(w.slot_mapping),
        "k_new": dev(w.k_new),
        "v_new": dev(w.v_new),
    }
    if w.k_cache is not None:
        d["k_cache"] = dev(w.k_cache)
        d["v_cache"] = dev(w.v_cache)
    return d


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, max_abs=MAX_ABS, rel_l2=REL_L2, what=""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / denom) if denom > 0 else float(np.linalg.norm(got - ref))
    assert mx <= max_abs, f"{what}: max abs err {mx:.3e} > {max_abs}"
    assert rel <= rel_l2, f"{what}: rel L2 err {rel:.3e} > {rel_l2}"
    return mx, rel
