"""Failure detection without a GPU fault: the bounded wait every kernel pipeline uses is
made to run out (an mbarrier nothing arrives on) with a short limit; the kernel must set
STATUS_TIMEOUT in the status word and return, and the device must stay usable."""
import numpy as np
import pytest
import torch

import workloads as W
from pa_harness import TOL, StepRun, oracle_step, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_53_gb300 as pa
    pa.get_status()
    return pa


def test_wait_gives_up_and_flags_timeout(pa):
    pa.selftest_wait_timeout(2000)  # 2 ms
    assert pa.get_status() == pa.STATUS_TIMEOUT
    assert pa.get_status() == 0  # read once, then cleared


def test_device_stays_usable_after_a_timeout(pa):
    pa.selftest_wait_timeout(500)
    torch.cuda.synchronize()
    assert pa.get_status() & pa.STATUS_TIMEOUT
    step = W.decode_step("after_timeout", W.Shape(32, 8, 128, 16, "bf16"), [1, 40, 700],
                         seed=61)
    run = StepRun(step)
    kc, vc = run.host_pool()
    vals = run.host_values()
    res = run.run()
    ref = oracle_step(step, kc, vc, vals)
    err = np.abs(to_f64(res["out_decode"]) - ref["out_decode"])
    assert np.all(err <= TOL["bf16"])
    assert pa.get_status() == 0


def test_timeouts_on_several_streams(pa):
    streams = [torch.cuda.Stream() for _ in range(3)]
    for s in streams:
        pa.selftest_wait_timeout(300, s)
    torch.cuda.synchronize()
    assert pa.get_status() == pa.STATUS_TIMEOUT
