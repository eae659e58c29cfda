"""Failure detection on the device without a fault: every pipeline wait of
the library is bounded, and a wait that runs out records
DFLASH_DEV_WAIT_TIMEOUT and returns instead of spinning.  The probe waits on
an mbarrier that nothing completes, with a limit of a few milliseconds, and
the host reads the code; the context stays usable afterwards."""
import time

import pytest
import torch

from block_diffusion_draft_gb300 import workloads as W

import helpers as T

pytestmark = pytest.mark.gpu

DFLASH_DEV_WAIT_TIMEOUT = 1


def _layer():
    sp = W.spec("qwen3_8b_single", hidden=1024, n_heads=8, n_kv_heads=2, batch=1,
                n_target_layers=2, max_position=4096)
    return sp, T.Scenario(sp, seed=21, capacity=256)


def test_completed_barrier_records_nothing():
    _, sc = _layer()
    sc.attn.wait_probe(2_000_000, arrive=True)
    assert sc.attn.device_error() == 0


def test_wait_that_runs_out_reports_timeout_and_returns():
    sp, sc = _layer()
    t0 = time.perf_counter()
    sc.attn.wait_probe(3_000_000, arrive=False)  # 3 ms, a barrier nobody completes
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert dt < 2.0, f"the bounded wait took {dt:.3f} s"
    assert sc.attn.device_error() == DFLASH_DEV_WAIT_TIMEOUT
    assert sc.attn.device_error() == 0  # read and cleared
    # the context is still usable: a forward step matches the oracle
    got, ref = sc.step([40])
    T.assert_close(got, ref, "bf16", "step after a timed-out wait")
    assert sc.attn.device_error() == 0


def test_probe_rejects_limits_outside_its_range():
    _, sc = _layer()
    for bad in (0, 999, 100_000_001):
        with pytest.raises(Exception, match="ARG"):
            sc.attn.wait_probe(bad, arrive=False)
    assert sc.attn.device_error() == 0
