"""Failure detection on the GPU without a GPU fault ("vla.cpp: A Unified
Inference Runtime for Vision-Language-Action Models", §III-C: a response
carries the action chunk or an error).

* Abort: the host sets the handle's abort flag (host-mapped memory); the
  solver latches VLA_ERR_ABORTED, the launch runs to completion, the status
  is reported and cleared by vla_expert_poll_status, and after clearing the
  flag the same handle serves a correct request.
* Timeout: with a 1 ms wait limit, a kernel whose bounded wait can never be
  satisfied gives up, latches VLA_ERR_TIMEOUT and returns (no trap, no hang);
  the handle then serves a correct request.
Neither test faults, traps or hangs the GPU: every wait is bounded.
"""

import time

import numpy as np
import pytest

import oracle as O
from _harness import gpu_run
from workloads import CONFIGS

pytestmark = pytest.mark.gpu

ABORTED, TIMEOUT = 7, 6


def _rerun_ok(run):
    import torch
    ex = run["expert"]
    c = run["cfg"]
    Kc, Vc = ex.alloc_cache(c.B, c.P)
    ex.prefix_kv_build(torch.from_numpy(run["Z"]).to(torch.bfloat16).cuda(), Kc, Vc)
    act = ex.denoise(Kc, Vc, torch.from_numpy(run["noise"]).cuda())
    torch.cuda.synchronize()
    assert ex.poll_status() == 0
    Kr, Vr = O.prefix_kv(run["Z"].astype(np.float64), run["w"], c)
    xr, _ = O.denoise(run["noise"].astype(np.float64), Kr, Vr, run["w"], c)
    assert O.parity_metrics(act.cpu().numpy(), xr)["e_inf"] <= 1e-2


def test_abort_flag_latches_and_handle_recovers():
    import torch
    run = gpu_run(CONFIGS["small_bf16"])
    assert run["status"] == 0
    ex, c = run["expert"], run["cfg"]
    Kc, Vc = ex.alloc_cache(c.B, c.P)
    ex.prefix_kv_build(torch.from_numpy(run["Z"]).to(torch.bfloat16).cuda(), Kc, Vc)
    ex.set_abort(True)
    ex.denoise(Kc, Vc, torch.from_numpy(run["noise"]).cuda())
    torch.cuda.synchronize()
    assert ex.poll_status() == ABORTED
    assert ex.poll_status() == 0  # polling cleared it
    ex.set_abort(False)
    _rerun_ok(run)


def test_bounded_wait_times_out_and_handle_recovers():
    import torch
    run = gpu_run(CONFIGS["small_bf16"])
    ex = run["expert"]
    ex.set_wait_limit(1_000_000)  # 1 ms
    t0 = time.perf_counter()
    ex.check_wait_timeout()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert ex.poll_status() == TIMEOUT
    assert waited < 1.0  # the wait gave up after its limit, not the 2 s default
    ex.set_wait_limit(0)
    _rerun_ok(run)
