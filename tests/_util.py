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


# Scale and temperature pairs that put a temperature other than 1 and a
# negative scale through a path (PR #69 lists the temperature among the
# call's arguments, "Verified on hardware"; the logits are scale * sim / T).
# Cosine logits are bounded by |scale| / T, so the pairs keep that at most
# about 20: the float32 error of a logit grows with its size, and these
# pairs keep it near 1e-5, far inside the 1e-4 bar, while a dropped,
# multiplied or sign-flipped factor still moves the probabilities by far
# more than the bar. Dot logits grow with the data, so `tempered_case`
# rescales the candidates to keep them of a few units.
TEMPERED = {
    1: [(14.2857, 0.7), (-14.2857, 3.0), (0.5, 0.05), (-0.5, 0.05)],
    0: [(0.0625, 0.7), (-0.0625, 3.0), (0.0625, 0.05), (-0.0625, 0.05)],
}


def plain_pair(normalize):
    """The page's own scale at temperature 1."""
    return (14.2857, 1.0) if normalize else (0.0625, 1.0)


def pairs_in_rotation(normalize):
    """The plain pair first, then every tempered pair: index i of a list of
    shapes takes pair i % 5, so a plan run over several shapes meets them all."""
    return [plain_pair(normalize)] + TEMPERED[normalize]


def tempered_case(B, K, D, normalize, pair, seed, device="cpu"):
    """A random_case with the given (scale, temperature). For the dot, the
    candidates of a tempered pair are rescaled so that the logits' spread is
    at most about 3 whatever D, scale and temperature are (q and C are
    N(0,1), so c.q has spread sqrt(D)); the plain pair keeps N(0,1) data."""
    from similarity_softmax_candidate_gb300 import workloads
    scale, temperature = pair
    wl = workloads.random_case(B, K, D, normalize, scale, seed, device, temperature=temperature)
    if not normalize and pair != plain_pair(0):
        f = 3.0 * temperature / (abs(scale) * D ** 0.5)
        if f < 1.0:
            wl.C.mul_(f)
    return wl
