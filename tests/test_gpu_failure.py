"""Failure detection on the GPU without a fault: a bounded wait runs out.

asp_selftest_wait_timeout launches one warp whose thread waits, through the
library's bounded mbarrier wait, on a barrier that nothing completes. After
the 2 s limit the wait gives up, the kernel sets ASP_DEVERR_TIMEOUT in the
workspace's error word and returns; the host reads the bit, and the same
context then runs a normal decode step that matches the oracle.
"""

from __future__ import annotations

import time

import pytest
import torch

from adaptive_sparse_paged_gb300 import binding as B
from tests.test_gpu_parity import SMALL, Case, check_case

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(cuda_device):
    ws = torch.empty(4096, dtype=torch.uint8, device=cuda_device)
    B.asp_workspace_init(ws)
    assert B.asp_get_device_error(ws) == 0
    t0 = time.perf_counter()
    B.asp_selftest_wait_timeout(ws)
    code = B.asp_get_device_error(ws)  # synchronises
    elapsed = time.perf_counter() - t0
    assert code == B.ASP_DEVERR_TIMEOUT, hex(code)
    assert 1.5 < elapsed < 30.0, elapsed  # the 2 s limit, not an instant failure
    assert B.asp_get_device_error(ws) == 0  # read and cleared
    # the context is intact: a normal step still matches the oracle
    case = Case(SMALL[0], seed=71, device=cuda_device)
    res = case.run(0, 0.9)
    check_case(case, 0, 0.9, 0, *res)
