"""The no-allocation entry point, cs_score_candidates_batch_unfused_noalloc.

Some callers cannot call cudaMalloc: code running under a host framework
that owns every byte of device memory through its own pool, or
latency-critical code that cannot pay for cudaMalloc's implicit device-wide
synchronization. For them the unfused baseline has a variant whose staged
array is a buffer built into the library, so the call allocates nothing.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test. It calls the entry point through
the C ABI with raw device pointers, twice in a row (the second call reuses
the buffer the first left filled), and checks each result against the
existing unfused entry point (caller-owned staged buffer) within the 1e-4
the other GPU tests use.
"""
from __future__ import annotations

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import ATOL, assert_parity, oracle_probs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _call_noalloc(lib, wl, out, stream):
    return lib.cs_score_candidates_batch_unfused_noalloc(
        wl.Q.data_ptr(), wl.C.data_ptr(), wl.B, wl.K, wl.D, wl.normalize, wl.scale, wl.temperature,
        out.data_ptr(), stream)


def _call_unfused(lib, wl, staged, out, stream):
    return lib.cs_score_candidates_batch_unfused(
        wl.Q.data_ptr(), wl.C.data_ptr(), wl.B, wl.K, wl.D, wl.normalize, wl.scale, wl.temperature,
        staged.data_ptr(), out.data_ptr(), stream)


def test_no_alloc_matches_unfused_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib
    stream = torch.cuda.current_stream().cuda_stream
    cases = [workloads.random_case(8, 255, 512, 1, workloads.CLM_SCALE, 901, DEV),
             workloads.random_case(300, 255, 512, 0, workloads.KEV_SCALE, 902, DEV)]
    outs = [torch.full((wl.B, wl.K), -1.0, device=DEV) for wl in cases]
    for wl, out in zip(cases, outs):  # two calls in a row, nothing in between
        assert _call_noalloc(lib, wl, out, stream) == binding.CS_OK
    torch.cuda.synchronize()
    for wl, out in zip(cases, outs):
        staged = torch.empty((wl.B, wl.K), device=DEV)
        ref = torch.empty((wl.B, wl.K), device=DEV)
        assert _call_unfused(lib, wl, staged, ref, stream) == binding.CS_OK
        torch.cuda.synchronize()
        assert torch.max(torch.abs(out - ref)).item() <= ATOL
        assert_parity(out, oracle_probs(wl.Q, wl.C, wl.normalize, wl.scale, wl.temperature), "no-alloc")


def test_no_alloc_rejects_more_rows_than_its_buffer(cuda_lib):
    lib = cuda_lib
    # B*K one row over the built-in buffer. The sizes are refused before any
    # CUDA call, so the (far apart, never dereferenced) addresses need no
    # memory behind them.
    B, K, D = binding.CS_NOALLOC_MAX_ROWS // 255 + 1, 255, 4
    s = lib.cs_score_candidates_batch_unfused_noalloc(0x7F0000000000, 0x7F1000000000, B, K, D, 1, 1.0, 1.0,
                                                      0x7F2000000000, None)
    assert s == binding.CS_ERR_SCRATCH_TOO_SMALL
    assert "no-allocation" in binding.cs_status_string(s)


def test_no_alloc_at_exactly_its_row_limit(cuda_lib):
    """B*K equal to the built-in buffer's size (8192 questions of K=128, D=4:
    1,048,576 rows, every float of the buffer used) is accepted and scored
    like the caller-buffer form and the oracle, on two calls in a row."""
    lib = cuda_lib
    stream = torch.cuda.current_stream().cuda_stream
    B, K = 8192, 128
    assert B * K == binding.CS_NOALLOC_MAX_ROWS
    wl = workloads.random_case(B, K, 4, 1, workloads.CLM_SCALE, 903, DEV)
    outs = [torch.full((B, K), -1.0, device=DEV) for _ in range(2)]
    for out in outs:
        assert _call_noalloc(lib, wl, out, stream) == binding.CS_OK
    staged = torch.empty((B, K), device=DEV)
    ref = torch.empty((B, K), device=DEV)
    assert _call_unfused(lib, wl, staged, ref, stream) == binding.CS_OK
    torch.cuda.synchronize()
    expected = oracle_probs(wl.Q, wl.C, wl.normalize, wl.scale, wl.temperature)
    for out in outs:
        assert torch.max(torch.abs(out - ref)).item() <= ATOL
        assert_parity(out, expected, "no-alloc at the row limit")
