"""Failure handling on the GPU without a fault: a bounded device wait that
runs out reports GBO_STATUS_TIMEOUT and leaves the context usable."""

import time

import pytest
import torch

from adamw_optimizer_step_gb300 import _binding as B
from tests.parity import random_entries, run_muon_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from adamw_optimizer_step_gb300 import build
    build.build()
    B.lib()


def test_bounded_wait_times_out_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    B.gbo_testing_wait_timeout(status, 20000)  # 20 ms on a barrier nothing arrives on
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) & B.GBO_STATUS_TIMEOUT
    assert 0.018 < dt < 2.0
    # the context is still usable: a normal step runs and reports no condition
    entries = random_entries([(64, 96, None, None)], seed=3)
    _, st, _ = run_muon_gpu(entries, lr=0.02, precision="bf16")
    assert st == 0
    with pytest.raises(B.GboError):
        B.gbo_testing_wait_timeout(status, 0)
