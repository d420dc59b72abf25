"""Pins of the fp64 oracle against facts fixed by the page and by mathematics.

Source of the method: PR #69 "cuda: add a fused candidate-scoring kernel for
CLM and Kev" -- the opening table (CLM: exp(logit_scale) * cosine; Kev:
1/sqrt(256) * dot; each softmaxed over the question's candidates), "What is
fused, precisely" and the fixed cases of "Verified on hardware" (a single
candidate, identical candidates, a zero candidate, raw logits that overflow a
naive softmax).

None of these tests re-types the oracle's formula. Each one checks a value or
property that a plausible mistake in the oracle would break:
  hand cases (tests/golden)   wrong similarity, sign, eps reading, scale or
                              temperature placement
  library cross-check         transposed operand, wrong index, dropped term
                              (numpy matmul, scipy cosine distance, scipy softmax)
  closed forms (K=1, K=2)     softmax normalisation and sign
  invariances                 max-subtraction, norm computed once, order
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax
from scipy.spatial.distance import cdist

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, *shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


# ---------------------------------------------------------------- hand cases

@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_case_logits(case):
    q = np.array(case["q"], dtype=np.float32)
    C = np.array(case["C"], dtype=np.float32)
    # every fixture value must be exact in float32, or the derivation is off
    assert np.array_equal(q.astype(np.float64), np.array(case["q"], dtype=np.float64))
    assert np.array_equal(C.astype(np.float64), np.array(case["C"], dtype=np.float64))
    z = oracle.logits(q, C, case["normalize"], case["scale"], case["temperature"])[0]
    np.testing.assert_allclose(z, case["expected_logits"], rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_case_probabilities(case):
    q = np.array(case["q"], dtype=np.float32)
    C = np.array(case["C"], dtype=np.float32)
    p = oracle.score_batch(q, C, case["normalize"], case["scale"], case["temperature"])[0]
    expected = sp_softmax(np.array(case["expected_logits"], dtype=np.float64))
    assert np.all(np.isfinite(p))
    np.testing.assert_allclose(p, expected, rtol=1e-13, atol=1e-15)


def test_axes_closed_form():
    """q = e1, C = {e1, e2, -e1}, cosine, scale s: p = (e^s, 1, e^-s) / sum."""
    s = 3.5
    q = np.array([1, 0, 0], np.float32)
    C = np.array([[1, 0, 0], [0, 1, 0], [-1, 0, 0]], np.float32)
    p = oracle.score_batch(q, C, 1, s, 1.0)[0]
    den = math.exp(s) + 1.0 + math.exp(-s)
    np.testing.assert_allclose(p, [math.exp(s) / den, 1 / den, math.exp(-s) / den], rtol=1e-14)


def test_overflow_case_finite_and_logistic():
    """Raw logits of 1000 and 998.046875: exp overflows, the result must not.
    p0 = 1 / (1 + e^-1.953125 + e^-2000)."""
    case = next(c for c in _cases() if c["name"] == "dot_overflow")
    assert math.isinf(math.exp(700) * math.exp(300))  # a naive softmax overflows here
    p = oracle.score_batch(np.array(case["q"], np.float32), np.array(case["C"], np.float32),
                           0, 1.0, 1.0)[0]
    assert np.all(np.isfinite(p))
    g = 1000.0 - 998.046875
    np.testing.assert_allclose(p[0], 1.0 / (1.0 + math.exp(-g)), rtol=1e-15)
    np.testing.assert_allclose(p[1], math.exp(-g) / (1.0 + math.exp(-g)), rtol=1e-14)
    assert p[2] == 0.0  # e^-2000 underflows to exactly zero in double


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("normalize", [0, 1])
def test_single_candidate_is_one(normalize):
    rng = _rng(1)
    for D in (1, 3, 512, 2560):
        p = oracle.score_batch(_rand(rng, D), _rand(rng, 1, D), normalize, 14.2857, 0.7)
        assert p.shape == (1, 1) and p[0, 0] == 1.0


@pytest.mark.parametrize("normalize", [0, 1])
def test_k2_is_logistic(normalize):
    """Two candidates: p0 = 1 / (1 + exp(z1 - z0)). The logits come from a
    hand construction: q = (a, 0); c0 = (1, 0) and c1 = (x, y)."""
    a, x, y, s, T = 2.0, 0.5, -0.75, 1.25, 0.5
    q = np.array([a, 0], np.float32)
    C = np.array([[1, 0], [x, y]], np.float32)
    if normalize:
        z0, z1 = s / T, s * (x / math.hypot(x, y)) / T
    else:
        z0, z1 = s * a / T, s * a * x / T
    p = oracle.score_batch(q, C, normalize, s, T)[0]
    np.testing.assert_allclose(p[0], 1.0 / (1.0 + math.exp(z1 - z0)), rtol=1e-14)
    np.testing.assert_allclose(p[1], 1.0 / (1.0 + math.exp(z0 - z1)), rtol=1e-14)


@pytest.mark.parametrize("normalize", [0, 1])
def test_identical_candidates_uniform(normalize):
    rng = _rng(2)
    for K in (2, 5, 64, 255):
        c = _rand(rng, 512)
        C = np.repeat(c[None, :], K, axis=0)
        p = oracle.score_batch(_rand(rng, 512), C, normalize, 14.2857, 1.0)[0]
        np.testing.assert_allclose(p, np.full(K, 1.0 / K), rtol=0, atol=1e-16)


def test_zero_candidate_gets_zero_logit():
    """Cosine: a zero candidate's logit is exactly 0 (t = 0 over clamped norms)."""
    rng = _rng(3)
    C = _rand(rng, 64, 512)
    C[17] = 0
    z = oracle.logits(_rand(rng, 512), C, 1, 14.2857, 1.0)[0]
    assert z[17] == 0.0
    assert np.count_nonzero(z) == 63


@pytest.mark.parametrize("normalize", [0, 1])
def test_zero_query_uniform(normalize):
    rng = _rng(4)
    p = oracle.score_batch(np.zeros(512, np.float32), _rand(rng, 255, 512), normalize, 14.2857, 1.0)[0]
    np.testing.assert_allclose(p, np.full(255, 1 / 255), rtol=0, atol=1e-16)


# ---------------------------------------------------------------- library cross-check

SHAPES = [(1, 5, 512), (1, 64, 512), (3, 255, 512), (2, 255, 2560), (4, 7, 13), (2, 33, 1)]


@pytest.mark.parametrize("B,K,D", SHAPES)
def test_dot_matches_numpy_scipy(B, K, D):
    """Kev: softmax over k of scale * (C @ q) / T, by numpy matmul and scipy."""
    rng = _rng(B * 1000 + K * 10 + D)
    Q, C = _rand(rng, B, D), _rand(rng, B, K, D, std=0.5)
    s, T = 0.0625, 0.8
    p = oracle.score_batch(Q, C, 0, s, T)
    for b in range(B):
        z = s * (C[b].astype(np.float64) @ Q[b].astype(np.float64)) / T
        np.testing.assert_allclose(p[b], sp_softmax(z), rtol=1e-11, atol=1e-15)


@pytest.mark.parametrize("B,K,D", [s for s in SHAPES if s[2] > 1])
def test_cosine_matches_scipy(B, K, D):
    """CLM: softmax of scale * cos / T, with cos = 1 - scipy's cosine distance."""
    rng = _rng(B * 1000 + K * 10 + D + 1)
    Q, C = _rand(rng, B, D), _rand(rng, B, K, D)
    s, T = 14.285714149475098, 1.3
    p = oracle.score_batch(Q, C, 1, s, T)
    for b in range(B):
        cos = 1.0 - cdist(Q[b][None].astype(np.float64), C[b].astype(np.float64), "cosine")[0]
        np.testing.assert_allclose(p[b], sp_softmax(s * cos / T), rtol=1e-10, atol=1e-15)


# ---------------------------------------------------------------- invariances

@pytest.mark.parametrize("normalize", [0, 1])
def test_rows_sum_to_one(normalize):
    rng = _rng(5)
    p = oracle.score_batch(_rand(rng, 6, 512), _rand(rng, 6, 255, 512), normalize, 14.2857, 0.5)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p >= 0)


def test_softmax_shift_invariance():
    rng = _rng(6)
    z = rng.standard_normal((3, 255)) * 5
    for c in (-700.0, -3.25, 0.5, 650.0):
        np.testing.assert_allclose(oracle.softmax(z + c), oracle.softmax(z), rtol=1e-12, atol=1e-300)


def test_dot_shift_by_common_candidate_offset():
    """Adding v to every candidate shifts every dot logit by scale*(v.q)/T,
    which the softmax must ignore."""
    rng = _rng(7)
    q = np.array([1, -2, 0.5, 4], np.float32)
    C = _rand(rng, 9, 4)
    v = np.array([0.25, 0.5, -1, 2], np.float32)
    p0 = oracle.score_batch(q, C, 0, 0.75, 1.0)
    p1 = oracle.score_batch(q, (C + v).astype(np.float32), 0, 0.75, 1.0)
    np.testing.assert_allclose(p1, p0, rtol=1e-6)  # C + v rounds once in float32


@pytest.mark.parametrize("normalize", [0, 1])
def test_scale_temperature_equivalence(normalize):
    rng = _rng(8)
    Q, C = _rand(rng, 2, 64), _rand(rng, 2, 30, 64)
    for a in (0.5, 3.0, 1e-3):
        np.testing.assert_allclose(oracle.score_batch(Q, C, normalize, 2.0 * a, 0.7 * a),
                                   oracle.score_batch(Q, C, normalize, 2.0, 0.7), rtol=1e-12)


def test_temperature_divides():
    """Halving T doubles every logit: p(T/2) is p(T) squared, renormalised."""
    rng = _rng(9)
    q, C = _rand(rng, 32), _rand(rng, 10, 32)
    p1 = oracle.score_batch(q, C, 1, 5.0, 1.0)[0]
    p2 = oracle.score_batch(q, C, 1, 5.0, 0.5)[0]
    np.testing.assert_allclose(p2, p1 ** 2 / np.sum(p1 ** 2), rtol=1e-12)


def test_cosine_invariant_to_positive_rescaling():
    """Rescaling q or any candidate by a positive factor leaves the cosine
    unchanged: catches a norm that is applied twice, or not at all."""
    rng = _rng(10)
    q, C = _rand(rng, 512), _rand(rng, 64, 512)
    p0 = oracle.score_batch(q, C, 1, 14.2857, 1.0)
    f = rng.uniform(0.01, 100, size=(64, 1)).astype(np.float32)
    p1 = oracle.score_batch((q * np.float32(8.0)), (C * f).astype(np.float32), 1, 14.2857, 1.0)
    np.testing.assert_allclose(p1, p0, rtol=1e-6)
    # power-of-two factors are exact in float32 and leave the result unchanged
    p2 = oracle.score_batch(q * np.float32(0.25), C * np.float32(16.0), 1, 14.2857, 1.0)
    np.testing.assert_allclose(p2, p0, rtol=1e-15)


@pytest.mark.parametrize("normalize", [0, 1])
def test_permutation_equivariance(normalize):
    rng = _rng(11)
    q, C = _rand(rng, 128), _rand(rng, 255, 128)
    perm = rng.permutation(255)
    p = oracle.score_batch(q, C, normalize, 3.0, 1.0)[0]
    pp = oracle.score_batch(q, C[perm], normalize, 3.0, 1.0)[0]
    np.testing.assert_allclose(pp, p[perm], rtol=1e-14)


def test_questions_are_independent():
    """A batch is a grid over questions: question b's answer depends only on
    q_b and C_b."""
    rng = _rng(12)
    Q, C = _rand(rng, 4, 64), _rand(rng, 4, 17, 64)
    p = oracle.score_batch(Q, C, 1, 14.2857, 1.0)
    for b in range(4):
        np.testing.assert_array_equal(oracle.score_batch(Q[b], C[b], 1, 14.2857, 1.0)[0], p[b])


def test_query_norm_is_not_multiplied():
    """The page's second GPU defect was a query norm counted once per warp
    (sqrt(8) too large on 8 warps). For cosine, multiplying |q| by sqrt(8)
    would divide every logit by sqrt(8); the library cosine must not."""
    rng = _rng(13)
    q, C = _rand(rng, 512), _rand(rng, 255, 512)
    z = oracle.logits(q, C, 1, 1.0, 1.0)[0]
    cos = 1.0 - cdist(q[None].astype(np.float64), C.astype(np.float64), "cosine")[0]
    np.testing.assert_allclose(z, cos, rtol=1e-10, atol=1e-14)
    assert np.max(np.abs(z - cos / math.sqrt(8))) > 1e-3


# ---------------------------------------------------------------- projections

def test_project_identity_and_permutation():
    """W = identity gives H back exactly; a permutation matrix permutes
    columns; a scaled identity scales them (powers of two: exact)."""
    rng = _rng(20)
    H = _rand(rng, 7, 16)
    np.testing.assert_array_equal(oracle.project(H, np.eye(16, dtype=np.float32)), H.astype(np.float64))
    perm = rng.permutation(16)
    P = np.eye(16, dtype=np.float32)[perm]
    np.testing.assert_array_equal(oracle.project(H, P), H[:, perm].astype(np.float64))
    np.testing.assert_array_equal(oracle.project(H, 4 * np.eye(16, dtype=np.float32)), 4.0 * H.astype(np.float64))


def test_project_matches_numpy_and_is_linear():
    rng = _rng(21)
    H, W, W2 = _rand(rng, 9, 64), _rand(rng, 12, 64), _rand(rng, 12, 64)
    np.testing.assert_allclose(oracle.project(H, W), H.astype(np.float64) @ W.astype(np.float64).T, rtol=1e-12,
                               atol=1e-12)
    # additive in W (the float32 sum W + W2 is exact when it is computed in
    # float64 and compared in float64)
    lhs = oracle.project(H, W) + oracle.project(H, W2)
    rhs = H.astype(np.float64) @ (W.astype(np.float64) + W2.astype(np.float64)).T
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
    assert oracle.project(H, W).shape == (9, 12)


def test_project_score_with_identity_heads_is_plain_score():
    """Identity heads (D = Din) leave the readout unchanged."""
    rng = _rng(22)
    Hq, Hc = _rand(rng, 3, 32), _rand(rng, 3, 20, 32)
    I = np.eye(32, dtype=np.float32)
    for normalize in (0, 1):
        np.testing.assert_array_equal(oracle.project_score_batch(Hq, I, Hc, I, normalize, 2.0, 1.0),
                                      oracle.score_batch(Hq, Hc, normalize, 2.0, 1.0))


def test_project_score_cosine_ignores_head_scale():
    """Cosine scoring is unchanged when a head is multiplied by a positive
    power of two."""
    rng = _rng(23)
    Hq, Hc = _rand(rng, 2, 32), _rand(rng, 2, 9, 32)
    Wq, Wc = _rand(rng, 16, 32), _rand(rng, 16, 32)
    a = oracle.project_score_batch(Hq, Wq, Hc, Wc, 1, 14.2857, 1.0)
    b = oracle.project_score_batch(Hq, 2 * Wq, Hc, 8 * Wc, 1, 14.2857, 1.0)
    np.testing.assert_allclose(a, b, rtol=1e-15)
