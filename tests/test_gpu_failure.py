"""Failure detection without a GPU fault: every pipeline wait in the kernels
is bounded; when it runs out the kernel records PA_DEV_TIMEOUT and returns.
The self-test makes a wait run out (a barrier that nothing arrives on) and
checks the status, then that the context still works."""
import numpy as np
import pytest
import torch

import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import assert_close, gpu_decode, gpu_pool, oracle_full
from workloads import Geometry, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_bounded_wait_gives_up_and_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_wait_selftest(status, limit_us=2000)
    torch.cuda.synchronize()
    assert pa.pa_status_from_device(int(status.item())) == -10  # PA_ERR_TIMEOUT


def test_context_is_usable_after_a_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(3):
        pa.pa_wait_selftest(status, limit_us=500)
    torch.cuda.synchronize()
    w = make_workload("after_timeout", Geometry(8, 2, 64), [40, 7, 300], seed=23)
    out, st = gpu_decode(w, gpu_pool(w, DEV), DEV)
    assert st == 0
    ref, _ = oracle_full(w)
    assert_close(out.float().cpu().numpy(), ref, "decode after a timed-out wait")


def test_selftest_argument_checks():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for bad in (0, -5, 2_000_000):
        with pytest.raises(pa.PAError):
            pa.pa_wait_selftest(status, limit_us=bad)
