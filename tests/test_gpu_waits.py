"""Bounded waits end in a status, not a hang.

Every on-chip wait of the scoring kernels gives up after a time limit, sets
a bit in the device status word and lets the kernel finish. This test makes
one such wait run out -- on a barrier that nothing completes -- with a short
limit, reads the status bit from the host, and checks that the context is
still usable by scoring a batch afterwards.
"""
from __future__ import annotations

import time

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import assert_parity, oracle_probs

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_sets_status_and_returns(cuda_lib):
    lib = cuda_lib
    torch.cuda.synchronize()
    assert binding.cs_device_status(clear=True) == 0
    t0 = time.perf_counter()
    assert lib.cs_selftest_bounded_wait(2000, None) == binding.CS_OK  # 2 ms limit
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0
    assert binding.cs_device_status(clear=True) == 1  # CS_DEVERR_WAIT_TIMEOUT
    # the context is still usable
    wl = workloads.random_case(4, 255, 512, 1, workloads.CLM_SCALE, 17, "cuda:0")
    p = binding.cs_score_candidates_batch(wl.Q, wl.C, 1, wl.scale, 1.0)
    torch.cuda.synchronize()
    assert_parity(p, oracle_probs(wl.Q, wl.C, 1, wl.scale, 1.0), "after a given-up wait")
    assert binding.cs_device_status() == 0


def test_selftest_rejects_bad_limit(cuda_lib):
    assert cuda_lib.cs_selftest_bounded_wait(0, None) == binding.CS_ERR_BAD_PLAN
    assert cuda_lib.cs_selftest_bounded_wait(2_000_000, None) == binding.CS_ERR_BAD_PLAN
