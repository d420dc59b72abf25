"""The bounds-checked build in place of a memory checker.

The library compiled with -DCS_DEBUG_BOUNDS checks, before every global
access its kernels make, that the range lies inside its buffer; a failing
check skips the access, records its site number and sets CS_DEVERR_BOUNDS.
These tests run every entry point on valid inputs of many shapes (all
plans, ragged, bfloat16, unfused, projections) through that build and
require that no check fails and that the results equal the release build's.
The detection itself is shown by a self-test kernel that checks a range one
past a buffer's end without touching memory. Nothing here reads or writes
outside a buffer.
"""
from __future__ import annotations

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import assert_parity, oracle_probs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def dbg(cuda_lib):
    lib = binding.debug_library()
    assert lib.cs_debug_bounds_build() == 1
    with binding.using(lib):
        binding.cs_device_status(clear=True)
        binding.cs_bounds_violation(clear=True)
    return lib


def _both(dbg, fn):
    """fn() with the release build, then with the bounds-checked build;
    returns both results and the debug build's status and bounds words."""
    ref = fn()
    torch.cuda.synchronize()
    with binding.using(dbg):
        got = fn()
        torch.cuda.synchronize()
        status = binding.cs_device_status(clear=True)
        site = binding.cs_bounds_violation(clear=True)
    return ref, got, status, site


def _same(ref, got, what):
    assert ref.shape == got.shape
    diff = torch.max(torch.abs(ref.float() - got.float())).item() if ref.numel() else 0.0
    assert diff <= 1e-6, f"{what}: release and bounds-checked builds differ by {diff:.3e}"


def test_release_build_has_no_checks(cuda_lib):
    assert cuda_lib.cs_debug_bounds_build() == 0
    assert cuda_lib.cs_selftest_bounds(None) == binding.CS_ERR_BAD_PLAN
    assert binding.cs_bounds_violation() == 0


def test_selftest_records_the_site(dbg):
    with binding.using(dbg):
        binding.cs_selftest_bounds()
        torch.cuda.synchronize()
        assert binding.cs_bounds_violation(clear=True) == 99
        assert binding.cs_device_status(clear=True) == binding.CS_DEVERR_BOUNDS
        assert binding.cs_bounds_violation() == 0


SHAPES = [  # B, K, D, normalize: STREAM, CLUSTER (2..16), GENERIC (D % 4 != 0), large D
    (300, 255, 512, 1), (300, 255, 512, 0), (1, 255, 512, 1), (8, 255, 512, 1), (1, 5, 512, 1),
    (1, 64, 512, 1), (1, 255, 2560, 0), (3, 17, 511, 1), (2, 9, 12288, 0), (157, 3, 64, 1),
]


@pytest.mark.parametrize("B,K,D,normalize", SHAPES)
def test_batch_within_bounds(dbg, B, K, D, normalize):
    wl = workloads.random_case(B, K, D, normalize, 3.0, 50 + B + K, DEV)
    ref, got, status, site = _both(dbg, lambda: binding.cs_score_candidates_batch(wl.Q, wl.C, normalize, 3.0, 1.0))
    assert site == 0 and status == 0, f"bounds site {site}, status {status}"
    _same(ref, got, f"B={B} K={K} D={D}")
    if B * K * D <= 3_000_000:
        assert_parity(got, oracle_probs(wl.Q.cpu(), wl.C.cpu(), normalize, 3.0, 1.0), "bounds-checked build")


def test_single_bf16_unfused_within_bounds(dbg):
    wl = workloads.random_case(40, 255, 512, 1, 3.0, 61, DEV)
    Cb = wl.C.to(torch.bfloat16)
    calls = {
        "single": lambda: binding.cs_score_candidates(wl.Q[0], wl.C[0], 1, 3.0, 1.0),
        "bf16": lambda: binding.cs_score_candidates_batch_bf16(wl.Q, Cb, 1, 3.0, 1.0),
        "bf16_dot": lambda: binding.cs_score_candidates_batch_bf16(wl.Q, Cb, 0, 3.0, 1.0),
        "unfused_cos": lambda: binding.cs_score_candidates_batch_unfused(wl.Q, wl.C, 1, 3.0, 1.0),
        "unfused_dot": lambda: binding.cs_score_candidates_batch_unfused(wl.Q, wl.C, 0, 3.0, 1.0),
        "unfused_noalloc": lambda: binding.cs_score_candidates_batch_unfused_noalloc(
            wl.Q, wl.C, 1, 3.0, 1.0, out=torch.empty(40, 255, device=DEV)),
    }
    for name, fn in calls.items():
        ref, got, status, site = _both(dbg, fn)
        assert site == 0 and status == 0, f"{name}: bounds site {site}, status {status}"
        _same(ref, got, name)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_within_bounds(dbg, dtype):
    rw = workloads.ragged(700, 512, 1, 3.0, 62, DEV, kmin=1, kmax=255)
    C = rw.C.to(dtype)
    ref, got, status, site = _both(dbg, lambda: binding.cs_score_candidates_ragged(rw.Q, C, rw.offsets, 1, 3.0, 1.0))
    assert site == 0 and status == 0, f"bounds site {site}, status {status}"
    _same(ref, got, f"ragged {dtype}")


def test_ragged_bad_offsets_are_the_kernels_own_check(dbg):
    """A question with invalid offsets is skipped by the kernel's own check
    (CS_DEVERR_BAD_OFFSETS), before any access: no bounds check fails."""
    rw = workloads.ragged(50, 512, 1, 3.0, 63, DEV, kmin=1, kmax=255)
    off = rw.offsets.clone()
    off[10] = off[11] + 5  # question 9 too long, question 10 negative: both skipped
    out = torch.full((int(rw.C.shape[0]),), -7.0, device=DEV)
    with binding.using(dbg):
        binding.cs_score_candidates_ragged(rw.Q, rw.C, off, 1, 3.0, 1.0, out=out)
        torch.cuda.synchronize()
        status = binding.cs_device_status(clear=True)
        site = binding.cs_bounds_violation(clear=True)
    assert site == 0
    assert status == 4  # CS_DEVERR_BAD_OFFSETS


def test_projections_within_bounds(dbg):
    g = torch.Generator(device="cpu")
    g.manual_seed(64)
    B, K, Din, D = 200, 255, 256, 512
    Hq = torch.randn(B, Din, generator=g).to(torch.bfloat16).to(DEV)
    Hc = torch.randn(B, K, Din, generator=g).to(torch.bfloat16).to(DEV)
    Wq = (torch.randn(D, Din, generator=g) * Din ** -0.5).to(torch.bfloat16).to(DEV)
    Wc = (torch.randn(D, Din, generator=g) * Din ** -0.5).to(torch.bfloat16).to(DEV)
    for name, fn in {"rows": lambda: binding.cs_project_rows(Hc.view(B * K, Din), Wc),
                     "score": lambda: binding.cs_project_score_batch(Hq, Wq, Hc, Wc, 1, 3.0, 1.0)}.items():
        ref, got, status, site = _both(dbg, fn)
        assert site == 0 and status == 0, f"{name}: bounds site {site}, status {status}"
        _same(ref, got, name)


def _placed(t, offset_elems):
    flat = torch.empty(t.numel() + offset_elems + 64, dtype=t.dtype, device=DEV)
    v = flat[offset_elems:offset_elems + t.numel()].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("B,K,D,oq,oc,bf16", [(300, 255, 510, 0, 0, False), (200, 64, 512, 1, 3, False),
                                                (160, 33, 13, 0, 1, False), (170, 37, 21, 2, 5, True),
                                                (3, 64, 509, 0, 3, False), (150, 255, 1025, 1, 3, True),
                                                (200, 64, 512, 1, 1, True), (100, 31, 258, 0, 7, True),
                                                (120, 255, 511, 3, 3, False), (60, 40, 2562, 1, 1, True),
                                                (50, 40, 2563, 0, 2, True), (60, 40, 1030, 1, 3, False),
                                                (2, 255, 512, 1, 1, True), (3, 40, 258, 0, 2, True),
                                                (1, 255, 511, 2, 1, False)])
def test_unaligned_rows_within_bounds(dbg, B, K, D, oq, oc, bf16):
    """Unaligned plans copy each stage's 16-byte aligned span; what the
    kernels check and use is the rows' own range, which must stay inside C,
    and the span must fit its ring slot. A few questions take the DIRECT
    plan's 4-byte units instead, checked the same way."""
    wl = workloads.random_case(B, K, D, 1, 3.0, 70 + B + D, DEV)
    Q = _placed(wl.Q, oq)
    C = _placed(wl.C.to(torch.bfloat16) if bf16 else wl.C, oc)
    fn = binding.cs_score_candidates_batch_bf16 if bf16 else binding.cs_score_candidates_batch
    for normalize in (1, 0):
        ref, got, status, site = _both(dbg, lambda: fn(Q, C, normalize, 3.0, 1.0))
        assert site == 0 and status == 0, f"bounds site {site}, status {status}"
        _same(ref, got, f"unaligned B={B} K={K} D={D} q+{oq} c+{oc} bf16={bf16}")
