"""The C ABI on a machine without a GPU: the library loads, exports every
function its header declares, and rejects bad arguments before any CUDA call
(so nothing is launched and the output is untouched).

Source of the rejected arguments: PR #69 "cuda: add a fused candidate-scoring
kernel for CLM and Kev", section "Verified on hardware" (K above 255, K of
zero, D of zero, a zero scale, a negative temperature, a null query).
"""
from __future__ import annotations

import ctypes
import glob
import math
import os
import re

import numpy as np
import pytest

from similarity_softmax_candidate_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Fake device addresses: validation must never dereference them.
Q_ADDR, C_ADDR, OUT_ADDR = 0x7F0000000000, 0x7F1000000000, 0x7F2000000000


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(cs_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("cs_abi_version", "cs_status_string", "cs_score_candidates", "cs_score_candidates_batch"):
        assert n in names


def test_header_limits_match_binding():
    text = open(os.path.join(ROOT, "include", "candidate_scoring.h")).read()
    m = re.search(r"#define CS_PROJ_MAX_ROWS (\d+)LL", text)
    assert m and int(m.group(1)) == binding.CS_PROJ_MAX_ROWS == (1 << 31) - 256
    m = re.search(r"#define CS_NOALLOC_MAX_ROWS (\d+)", text)
    assert m and int(m.group(1)) == binding.CS_NOALLOC_MAX_ROWS


@pytest.mark.parametrize("name", _declared_functions())
def test_library_exports_declared_symbol(host_lib, name):
    assert hasattr(host_lib, name), f"{name} declared in include/*.h but not exported"


def test_abi_version(host_lib):
    assert host_lib.cs_abi_version() == 1


def test_status_strings(host_lib):
    for code in range(15):
        s = host_lib.cs_status_string(code).decode()
        assert s and s != "unknown status"
    assert host_lib.cs_status_string(999).decode() == "unknown status"


def _batch(lib, Q=Q_ADDR, C=C_ADDR, B=1, K=5, D=512, normalize=1, scale=14.2857, temperature=1.0, out=OUT_ADDR):
    return lib.cs_score_candidates_batch(Q, C, B, K, D, normalize, scale, temperature, out, None)


def _single(lib, q=Q_ADDR, C=C_ADDR, K=5, D=512, normalize=1, scale=14.2857, temperature=1.0, out=OUT_ADDR):
    return lib.cs_score_candidates(q, C, K, D, normalize, scale, temperature, out, None)


REJECTS = [
    ("k_above_255", dict(K=256), binding.CS_ERR_K_TOO_LARGE),
    ("k_far_above", dict(K=100000), binding.CS_ERR_K_TOO_LARGE),
    ("k_zero", dict(K=0), binding.CS_ERR_K_ZERO),
    ("k_negative", dict(K=-3), binding.CS_ERR_K_ZERO),
    ("d_zero", dict(D=0), binding.CS_ERR_D_ZERO),
    ("d_negative", dict(D=-1), binding.CS_ERR_D_ZERO),
    ("scale_zero", dict(scale=0.0), binding.CS_ERR_BAD_SCALE),
    ("scale_neg_zero", dict(scale=-0.0), binding.CS_ERR_BAD_SCALE),
    ("scale_nan", dict(scale=math.nan), binding.CS_ERR_BAD_SCALE),
    ("scale_inf", dict(scale=math.inf), binding.CS_ERR_BAD_SCALE),
    ("temperature_negative", dict(temperature=-1.0), binding.CS_ERR_BAD_TEMPERATURE),
    ("temperature_zero", dict(temperature=0.0), binding.CS_ERR_BAD_TEMPERATURE),
    ("temperature_nan", dict(temperature=math.nan), binding.CS_ERR_BAD_TEMPERATURE),
    ("temperature_inf", dict(temperature=math.inf), binding.CS_ERR_BAD_TEMPERATURE),
    # |scale / temperature| above 2^126: the kernels need the logit factor
    # times log2(e) finite, and the exact softmax of such logits is an
    # argmax that float32 similarities cannot settle reliably
    ("factor_tiny_temperature", dict(scale=14.2857, temperature=1e-37), binding.CS_ERR_RANGE),
    ("factor_huge_scale", dict(scale=3e38, temperature=0.5), binding.CS_ERR_RANGE),
    ("factor_negative", dict(scale=-1e30, temperature=1e-10), binding.CS_ERR_RANGE),
    ("null_query", dict(Q=None), binding.CS_ERR_NULL_POINTER),
    ("null_candidates", dict(C=None), binding.CS_ERR_NULL_POINTER),
    ("null_out", dict(out=None), binding.CS_ERR_NULL_POINTER),
    ("similarity_2", dict(normalize=2), binding.CS_ERR_BAD_SIMILARITY),
    ("similarity_neg", dict(normalize=-1), binding.CS_ERR_BAD_SIMILARITY),
]


@pytest.mark.parametrize("name,kw,status", REJECTS, ids=[r[0] for r in REJECTS])
def test_batch_rejects(host_lib, name, kw, status):
    assert _batch(host_lib, **kw) == status


@pytest.mark.parametrize("name,kw,status", REJECTS, ids=[r[0] for r in REJECTS])
def test_single_rejects(host_lib, name, kw, status):
    kw = {("q" if k == "Q" else k): v for k, v in kw.items()}
    assert _single(host_lib, **kw) == status


@pytest.mark.parametrize("B", [0, -1, -(2 ** 31)])
def test_batch_rejects_bad_batch(host_lib, B):
    assert _batch(host_lib, B=B) == binding.CS_ERR_BAD_BATCH


def test_rejects_out_overlapping_inputs(host_lib):
    B, K, D = 4, 8, 16
    # out starting inside C, and out starting inside Q
    assert _batch(host_lib, B=B, K=K, D=D, out=C_ADDR + 4 * 100) == binding.CS_ERR_ALIAS
    assert _batch(host_lib, B=B, K=K, D=D, out=Q_ADDR + 4 * (B * D - 1)) == binding.CS_ERR_ALIAS
    # out ending exactly where Q starts does not overlap (would go on to CUDA, so not called here)


def test_rejects_oversized_problem(host_lib):
    assert _batch(host_lib, B=2 ** 31 - 1, K=255, D=2 ** 31 - 1) == binding.CS_ERR_TOO_LARGE


def test_largest_factor_is_checked_in_double_precision(host_lib):
    """The factor is scale / temperature formed in double precision and
    refused above 2^126. A factor of exactly 2^126 passes the scalar
    checks: with an overlapping out, the call then stops at the overlap
    check, which validation makes after the scalars; so does a factor too
    small for float32."""
    top = 2.0 ** 126
    assert _batch(host_lib, scale=top, temperature=0.999) == binding.CS_ERR_RANGE
    assert _batch(host_lib, scale=-top, temperature=0.5) == binding.CS_ERR_RANGE
    assert _batch(host_lib, scale=float(np.finfo(np.float32).max), temperature=1.0) == binding.CS_ERR_RANGE
    B, K, D = 4, 8, 16
    for scale, T in ((top, 1.0), (-top, 1.0), (1e-30, 1e30)):
        assert _batch(host_lib, B=B, K=K, D=D, scale=scale, temperature=T, out=C_ADDR + 400) == binding.CS_ERR_ALIAS


def test_rejects_pointers_off_their_element_size(host_lib):
    """Elements are read as float32 (bfloat16 for the _bf16 candidates): a
    pointer off its element size is refused before any CUDA call. Offsets
    from a 16-byte boundary that keep the element alignment are accepted by
    validation (an aliasing out then stops those calls at the later overlap
    check)."""
    E = binding
    assert _batch(host_lib, Q=Q_ADDR + 2) == E.CS_ERR_MISALIGNED
    assert _batch(host_lib, C=C_ADDR + 1) == E.CS_ERR_MISALIGNED
    assert _batch(host_lib, out=OUT_ADDR + 3) == E.CS_ERR_MISALIGNED
    assert _single(host_lib, q=Q_ADDR + 6) == E.CS_ERR_MISALIGNED
    bf = host_lib.cs_score_candidates_batch_bf16
    assert bf(Q_ADDR, C_ADDR + 1, 1, 5, 512, 1, 1.0, 1.0, OUT_ADDR, None) == E.CS_ERR_MISALIGNED
    B, K, D = 4, 8, 16
    assert bf(Q_ADDR, C_ADDR + 2, B, K, D, 1, 1.0, 1.0, C_ADDR + 400, None) == E.CS_ERR_ALIAS
    assert _batch(host_lib, B=B, K=K, D=D, Q=Q_ADDR + 4, C=C_ADDR + 12, out=C_ADDR + 400) == E.CS_ERR_ALIAS
    assert _ragged(host_lib, offsets=OFF_ADDR + 4) == E.CS_ERR_MISALIGNED
    assert _unfused(host_lib, staged=STAGED_ADDR + 2) == E.CS_ERR_MISALIGNED


def test_first_failing_check_wins(host_lib):
    # the page lists each reject on its own; with several bad arguments the
    # library reports pointers, then B, K, D, similarity, scale, temperature
    assert _batch(host_lib, Q=None, K=0) == binding.CS_ERR_NULL_POINTER
    assert _batch(host_lib, K=0, D=0) == binding.CS_ERR_K_ZERO
    assert _batch(host_lib, D=0, scale=0.0) == binding.CS_ERR_D_ZERO
    assert _batch(host_lib, scale=0.0, temperature=-1.0) == binding.CS_ERR_BAD_SCALE


def test_rejected_call_leaves_output_untouched(host_lib):
    """Validation returns before any CUDA call, so even a host buffer passed
    as out is never written by a rejected call."""
    out = np.full(64, 12345.0, dtype=np.float32)
    before = out.copy()
    for _, kw, status in REJECTS:
        if "out" in kw:
            continue
        assert _batch(host_lib, out=out.ctypes.data, **kw) == status
    np.testing.assert_array_equal(out, before)


def test_plan_entry_rejects_unknown_plan(host_lib):
    f = host_lib.cs_score_candidates_batch_plan
    assert f(Q_ADDR, C_ADDR, 1, 5, 512, 1, 1.0, 1.0, OUT_ADDR, None, 7, 0, 0) == binding.CS_ERR_BAD_PLAN
    assert f(Q_ADDR, C_ADDR, 1, 5, 512, 1, 1.0, 1.0, OUT_ADDR, None, -1, 0, 0) == binding.CS_ERR_BAD_PLAN
    assert f(Q_ADDR, C_ADDR, 1, 0, 512, 1, 1.0, 1.0, OUT_ADDR, None, 1, 0, 0) == binding.CS_ERR_K_ZERO


def test_query_plan_validates(host_lib):
    i = ctypes.c_int()
    r = ctypes.byref(i)
    assert host_lib.cs_query_plan(Q_ADDR, C_ADDR, 1, 256, 512, 1, r, r, r, r) == binding.CS_ERR_K_TOO_LARGE
    assert host_lib.cs_query_plan(None, C_ADDR, 1, 5, 512, 1, r, r, r, r) == binding.CS_ERR_NULL_POINTER


def test_device_status_null(host_lib):
    assert host_lib.cs_device_status(None, 0) == binding.CS_ERR_NULL_POINTER


def test_binding_refuses_host_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(8)
    C = torch.zeros(3, 8)
    with pytest.raises(ValueError, match="CUDA device"):
        binding.cs_score_candidates(q, C, 1, 1.0, 1.0)


STAGED_ADDR = 0x7F3000000000


def _unfused(lib, Q=Q_ADDR, C=C_ADDR, B=1, K=5, D=512, normalize=1, scale=14.2857, temperature=1.0,
             staged=STAGED_ADDR, out=OUT_ADDR):
    return lib.cs_score_candidates_batch_unfused(Q, C, B, K, D, normalize, scale, temperature, staged, out, None)


@pytest.mark.parametrize("name,kw,status", REJECTS, ids=[r[0] for r in REJECTS])
def test_unfused_rejects(host_lib, name, kw, status):
    assert _unfused(host_lib, **kw) == status


def test_unfused_rejects_null_or_overlapping_staged(host_lib):
    assert _unfused(host_lib, staged=None) == binding.CS_ERR_NULL_POINTER
    B, K, D = 4, 8, 16
    assert _unfused(host_lib, B=B, K=K, D=D, staged=C_ADDR + 64) == binding.CS_ERR_ALIAS
    assert _unfused(host_lib, B=B, K=K, D=D, staged=OUT_ADDR + 4 * (B * K - 1)) == binding.CS_ERR_ALIAS
    assert _unfused(host_lib, B=B, K=K, D=D, staged=Q_ADDR) == binding.CS_ERR_ALIAS


@pytest.mark.parametrize("name,kw,status", REJECTS, ids=[r[0] for r in REJECTS])
def test_bf16_batch_rejects(host_lib, name, kw, status):
    kw = {**dict(Q=Q_ADDR, C=C_ADDR, B=1, K=5, D=512, normalize=1, scale=14.2857, temperature=1.0, out=OUT_ADDR), **kw}
    assert host_lib.cs_score_candidates_batch_bf16(kw["Q"], kw["C"], kw["B"], kw["K"], kw["D"], kw["normalize"],
                                                   kw["scale"], kw["temperature"], kw["out"], None) == status


def test_bf16_alias_uses_two_byte_elements(host_lib):
    B, K, D = 4, 8, 16
    # C holds B*K*D*2 = 1 KB: an out 1100 bytes past C's start does not
    # overlap it, one 1000 bytes past does
    assert host_lib.cs_score_candidates_batch_bf16(Q_ADDR, C_ADDR, B, K, D, 1, 1.0, 1.0, C_ADDR + 1000,
                                                   None) == binding.CS_ERR_ALIAS


OFF_ADDR = 0x7F4000000000


def _ragged(lib, Q=Q_ADDR, C=C_ADDR, offsets=OFF_ADDR, B=4, total=40, D=512, normalize=1, scale=2.0,
            temperature=1.0, out=OUT_ADDR):
    return lib.cs_score_candidates_ragged(Q, C, offsets, B, total, D, normalize, scale, temperature, out, None)


def test_ragged_rejects(host_lib):
    E = binding
    assert _ragged(host_lib, offsets=None) == E.CS_ERR_NULL_POINTER
    assert _ragged(host_lib, Q=None) == E.CS_ERR_NULL_POINTER
    assert _ragged(host_lib, B=0) == E.CS_ERR_BAD_BATCH
    assert _ragged(host_lib, B=4, total=3) == E.CS_ERR_K_ZERO          # some question would have no row
    assert _ragged(host_lib, B=4, total=4 * 255 + 1) == E.CS_ERR_K_TOO_LARGE
    assert _ragged(host_lib, D=0) == E.CS_ERR_D_ZERO
    assert _ragged(host_lib, normalize=3) == E.CS_ERR_BAD_SIMILARITY
    assert _ragged(host_lib, scale=0.0) == E.CS_ERR_BAD_SCALE
    assert _ragged(host_lib, temperature=-2.0) == E.CS_ERR_BAD_TEMPERATURE
    assert _ragged(host_lib, scale=14.2857, temperature=1e-37) == E.CS_ERR_RANGE
    assert _ragged(host_lib, out=OFF_ADDR + 8) == E.CS_ERR_ALIAS         # out over the offsets
    assert _ragged(host_lib, out=C_ADDR + 4 * 512 * 39) == E.CS_ERR_ALIAS
    assert host_lib.cs_score_candidates_ragged_bf16(Q_ADDR, C_ADDR, OFF_ADDR, 4, 40, 512, 1, 2.0, 1.0,
                                                    C_ADDR + 2 * 512 * 39, None) == E.CS_ERR_ALIAS


W_ADDR, P_ADDR = 0x7F5000000000, 0x7F6000000000


def test_project_rejects(host_lib):
    E = binding
    f = host_lib.cs_project_rows
    assert f(None, W_ADDR, 10, 64, 256, P_ADDR, None) == E.CS_ERR_NULL_POINTER
    assert f(Q_ADDR, W_ADDR, 0, 64, 256, P_ADDR, None) == E.CS_ERR_BAD_BATCH
    assert f(Q_ADDR, W_ADDR, (1 << 31) - 255, 64, 256, P_ADDR, None) == E.CS_ERR_BAD_BATCH  # > CS_PROJ_MAX_ROWS
    assert f(Q_ADDR, W_ADDR, 10, 0, 256, P_ADDR, None) == E.CS_ERR_D_ZERO
    assert f(Q_ADDR, W_ADDR, 10, 96, 256, P_ADDR, None) == E.CS_ERR_BAD_PLAN     # Din not a multiple of 64
    assert f(Q_ADDR, W_ADDR, 10, 64, 384, P_ADDR, None) == E.CS_ERR_BAD_PLAN     # D not 256 or 512
    assert f(Q_ADDR + 8, W_ADDR, 10, 64, 256, P_ADDR, None) == E.CS_ERR_BAD_PLAN  # unaligned
    assert f(Q_ADDR, W_ADDR, 10, 64, 256, Q_ADDR + 64, None) == E.CS_ERR_ALIAS
    g = host_lib.cs_project_score_batch
    args = dict(Hq=Q_ADDR, Wq=W_ADDR, Hc=C_ADDR, Wc=W_ADDR + (1 << 24), B=2, K=5, Din=64, D=256, n=1, s=2.0, t=1.0,
                qp=P_ADDR, out=OUT_ADDR)

    def call(**kw):
        a = {**args, **kw}
        return g(a["Hq"], a["Wq"], a["Hc"], a["Wc"], a["B"], a["K"], a["Din"], a["D"], a["n"], a["s"], a["t"],
                 a["qp"], a["out"], None)
    assert call(Hc=None) == E.CS_ERR_NULL_POINTER
    assert call(K=256) == E.CS_ERR_K_TOO_LARGE
    assert call(K=0) == E.CS_ERR_K_ZERO
    assert call(B=0) == E.CS_ERR_BAD_BATCH
    assert call(B=(1 << 31) // 200, K=255) == E.CS_ERR_BAD_BATCH  # B*K > CS_PROJ_MAX_ROWS
    assert call(s=0.0) == E.CS_ERR_BAD_SCALE
    assert call(t=-1.0) == E.CS_ERR_BAD_TEMPERATURE
    assert call(s=14.2857, t=1e-37) == E.CS_ERR_RANGE
    assert call(n=5) == E.CS_ERR_BAD_SIMILARITY
    assert call(D=128) == E.CS_ERR_BAD_PLAN
    assert call(out=C_ADDR) == E.CS_ERR_ALIAS
    assert call(qp=OUT_ADDR) == E.CS_ERR_ALIAS


def test_bounds_checked_build_compiles_and_reports_itself(host_lib):
    """The -DCS_DEBUG_BOUNDS variant builds from the same sources and says
    so; the release library does not (neither call touches a GPU)."""
    import ctypes

    from similarity_softmax_candidate_gb300 import _build
    dbg = ctypes.CDLL(_build.build_library(debug_bounds=True))
    assert dbg.cs_debug_bounds_build() == 1
    assert host_lib.cs_debug_bounds_build() == 0
    for name in _declared_functions():
        assert hasattr(dbg, name), f"{name} missing from the bounds-checked build"
