"""Helpers shared by the GPU tests: run the fp64 oracle on the very inputs
the kernel saw, and compare.

Tolerances (PR #69 "cuda: add a fused candidate-scoring kernel for CLM and
Kev", "The manifest, and CI": max_abs 1e-4): each probability within 1e-4
of the oracle, and each row of probabilities summing to 1 within 1e-5.
"""
from __future__ import annotations

import numpy as np

import oracle

ATOL = 1e-4
ROWSUM_TOL = 1e-5


def oracle_probs(Q, C, normalize, scale, temperature):
    """Oracle probabilities for torch tensors (any device) or numpy arrays."""
    Qh = Q.detach().cpu().numpy() if hasattr(Q, "detach") else np.asarray(Q)
    Ch = C.detach().cpu().numpy() if hasattr(C, "detach") else np.asarray(C)
    return oracle.score_batch(Qh, Ch, normalize, scale, temperature)


def assert_parity(p_gpu, p_ref, what=""):
    """Element-wise |p_gpu - p_ref| <= ATOL and GPU rows summing to 1."""
    p = p_gpu.detach().cpu().numpy().astype(np.float64) if hasattr(p_gpu, "detach") else np.asarray(p_gpu, np.float64)
    p = p.reshape(p_ref.shape)
    assert np.all(np.isfinite(p)), f"{what}: non-finite probabilities"
    err = np.max(np.abs(p - p_ref)) if p.size else 0.0
    assert err <= ATOL, f"{what}: max |gpu - oracle| = {err:.3e} > {ATOL}"
    sums = p.reshape(-1, p.shape[-1]).sum(axis=1)
    serr = np.max(np.abs(sums - 1.0)) if sums.size else 0.0
    assert serr <= ROWSUM_TOL, f"{what}: max |row sum - 1| = {serr:.3e} > {ROWSUM_TOL}"
    return err
