"""Planted mistakes in the oracle must fail its pins.

Each case below copies oracle/oracle.c, plants one plausible mistake in the
copy (a dropped or inverted term, a wrong index or operand, a missing
square root, the page's own second defect of a query norm summed over
eight warps, ...), builds it with gcc and runs tests/test_oracle_pins.py
against that build in a child process. The pins must fail every mutant; an
unaltered copy must pass them, so the harness itself is checked too. Every
planted edit must match the source exactly once, so that a change to
oracle.c that moves a target makes this test fail instead of checking
nothing. CPU only: nothing here touches a GPU or the CUDA library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# name -> [(text in oracle.c, replacement), ...]
MUTANTS = {
    "temperature_multiplies": [("scale * sim / temperature", "scale * sim * temperature")],
    "temperature_dropped": [("scale * sim / temperature", "scale * sim")],
    "scale_dropped": [("scale * sim / temperature", "sim / temperature")],
    "query_norm_summed_over_8_warps": [("double qnorm = sqrt(qq);", "double qnorm = sqrt(8.0 * qq);")],
    "eps_added_not_clamped": [("double a = qnorm > eps ? qnorm : eps;", "double a = qnorm + eps;"),
                              ("double c_ = cnorm > eps ? cnorm : eps;", "double c_ = cnorm + eps;")],
    "eps_clamps_the_product": [("sim = t / (a * c_);",
                                "sim = t / ((qnorm * cnorm) > eps ? (qnorm * cnorm) : eps); (void)a; (void)c_;")],
    "candidate_norm_from_dot": [("cc += (double)c[d] * (double)c[d];", "cc += (double)c[d] * (double)q[d];")],
    "candidate_norm_without_sqrt": [("double cnorm = sqrt(cc);", "double cnorm = cc;")],
    "dot_uses_query_twice": [("t += (double)c[d] * (double)q[d];", "t += (double)q[d] * (double)q[d];")],
    "dot_skips_first_feature": [("for (long d = 0; d < D; ++d) t +=", "for (long d = 1; d < D; ++d) t +=")],
    "candidate_index_shifted": [("((size_t)b * (size_t)K + (size_t)k) * (size_t)D",
                                 "((size_t)b * (size_t)K + (size_t)((k + 1) % K)) * (size_t)D")],
    "questions_reversed": [("const float *q = Q + (size_t)b * (size_t)D;",
                            "const float *q = Q + (size_t)(B - 1 - b) * (size_t)D;")],
    "no_max_subtraction": [("pr[k] = exp(zr[k] - m);", "pr[k] = exp(zr[k]);")],
    "min_subtracted_not_max": [("if (zr[k] > m) m = zr[k];", "if (zr[k] < m) m = zr[k];")],
    "exponent_sign_flipped": [("pr[k] = exp(zr[k] - m);", "pr[k] = exp(m - zr[k]);")],
    "wrong_normaliser": [("pr[k] = pr[k] / s;", "pr[k] = pr[k] / (s + 1.0);")],
    "projection_features_reversed": [("const float *w = W + (size_t)n * (size_t)Din;",
                                      "const float *w = W + (size_t)(D - 1 - n) * (size_t)Din;")],
    "projection_drops_last_input": [("for (long i = 0; i < Din; ++i) acc +=", "for (long i = 0; i < Din - 1; ++i) acc +=")],
}


def _have_gcc():
    return shutil.which("gcc") is not None


def _run_pins(tmp_path, name, edits):
    """Build oracle.c with `edits` applied and run the pins against it;
    returns (exit code, tail of the output)."""
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, f"{name}: target {old!r} found {src.count(old)} times in oracle.c"
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    c_path, so_path = d / "oracle.c", d / "liboracle.so"
    c_path.write_text(src)
    env = dict(os.environ, CS_ORACLE_SRC=str(c_path), CS_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert so_path.exists(), f"{name}: the altered oracle was not built:\n{r.stdout[-2000:]}\n{r.stderr[-2000:]}"
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.mark.skipif(not _have_gcc(), reason="gcc not available: could not check (skipped, not passed)")
def test_unaltered_copy_passes_the_pins(tmp_path):
    rc, out = _run_pins(tmp_path, "unaltered", [])
    assert rc == 0, f"the pins fail an unaltered copy of the oracle:\n{out}"


@pytest.mark.skipif(not _have_gcc(), reason="gcc not available: could not check (skipped, not passed)")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    rc, out = _run_pins(tmp_path, name, MUTANTS[name])
    assert rc == 1, f"no pin caught the planted mistake {name!r} (pytest exit {rc}):\n{out}"
