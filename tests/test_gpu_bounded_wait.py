"""The kernels' fail-fast path: a pipeline wait that cannot complete gives up
after its limit, sets PKV_DEVERR_TIMEOUT and lets the kernel return, and the
stream stays usable (the PhyAI deployment page "Parallel serving", failure
handling: fail fast on a timeout).  pkv_selftest_bounded_wait runs the
kernels' bounded wait on a ring stage that nothing arms; no copy is in flight
when it gives up."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_close, bf16_to_f64, to_device

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import paged_kv_decode_attention_gb300 as pkv
else:  # collected on CPU-only machines, every test skipped
    pkv = None


def _ordinary_step_matches_oracle():
    w = W.tiny(seed=5)
    d = to_device(w)
    out = torch.full_like(d["q"], float("nan"))
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    pkv.paged_attention_append(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], 1,
                               w.scale, d["slot_mapping"], d["k_new"], d["v_new"], workspace=ws)
    torch.cuda.synchronize()
    assert_close(bf16_to_f64(out), oracle.run_workload(w), what="call after the expired wait")


def test_armed_waits_complete_without_error():
    pkv.get_device_error(reset=True)
    pkv.selftest_bounded_wait(5000, arm_all=True)
    assert pkv.get_device_error(reset=True) == 0


def test_unarmed_wait_expires_reports_timeout_and_the_stream_stays_usable():
    pkv.get_device_error(reset=True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    pkv.selftest_bounded_wait(5000)
    ev1.record()
    assert pkv.get_device_error(reset=True) == pkv.DEVERR_TIMEOUT
    # the wait gave up after its limit (5 ms), not at once and not much later
    ms = ev0.elapsed_time(ev1)
    assert 4.5 <= ms < 1000.0, ms
    # the next ordinary call on the same stream runs and is right
    _ordinary_step_matches_oracle()
    assert pkv.get_device_error(reset=True) == 0
