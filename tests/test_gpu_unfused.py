"""GPU parity of the unfused baseline (PR #69 "cuda: add a fused
candidate-scoring kernel for CLM and Kev", "What it is worth": a separate
norm pass plus the scoring block reading the norm from a staged array; for
the dot, a second kernel and a global round trip of the similarities).

The baseline computes the same readout as the fused path, so it is held to
the same bar against the fp64 oracle; its staged array is checked against
numpy's norms and dots (float64).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import ATOL, assert_parity, oracle_probs, pairs_in_rotation, tempered_case

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

SHAPES = [(1, 5, 512), (1, 64, 512), (1, 255, 512), (8, 255, 512), (1, 255, 2560), (300, 255, 512), (3, 37, 132),
          (2, 200, 1028), (5, 1, 4)]


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_unfused_parity_and_staged(cuda_lib, normalize):
    """Shape i takes (scale, temperature) pair i % 5: the page's scale at
    temperature 1, then temperatures 0.7, 3 and 0.05 with positive and
    negative scales (pass 2 forms the factor in its own code)."""
    pairs = pairs_in_rotation(normalize)
    for i, (B, K, D) in enumerate(SHAPES):
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 500 + B + K + D)
        sc, T = wl.scale, wl.temperature
        Q, C = wl.Q.to(DEV), wl.C.to(DEV)
        staged = torch.full((B, K), -7.0, device=DEV)
        p = binding.cs_score_candidates_batch_unfused(Q, C, normalize, sc, T, staged=staged)
        pf = binding.cs_score_candidates_batch(Q, C, normalize, sc, T)
        torch.cuda.synchronize()
        ref = oracle_probs(wl.Q, wl.C, normalize, sc, T)
        assert_parity(p, ref, f"unfused B={B} K={K} D={D} scale={sc} T={T}")
        assert torch.max(torch.abs(p - pf)).item() <= ATOL
        C64 = wl.C.double().numpy()
        want = np.linalg.norm(C64, axis=2) if normalize else np.einsum("bkd,bd->bk", C64, wl.Q.double().numpy())
        got = staged.cpu().double().numpy()
        np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-4 * max(1.0, float(np.abs(want).max())))


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_unfused_every_tempered_pair(cuda_lib, normalize):
    """Both passes with every tempered pair, a few questions and many."""
    for B, K, D in ((3, 37, 132), (300, 255, 512)):
        for pair in pairs_in_rotation(normalize)[1:]:
            wl = tempered_case(B, K, D, normalize, pair, 600 + B + K + D, DEV)
            p = binding.cs_score_candidates_batch_unfused(wl.Q, wl.C, normalize, wl.scale, wl.temperature)
            torch.cuda.synchronize()
            assert_parity(p, oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature),
                          f"unfused B={B} K={K} D={D} scale={wl.scale} T={wl.temperature}")


def test_unfused_workloads(cuda_lib):
    for name in ("clm_k5", "clm_k64", "clm_batch8", "kev_k255"):
        for wl in workloads.CONFIGS[name]("cpu"):
            p = binding.cs_score_candidates_batch_unfused(wl.Q.to(DEV), wl.C.to(DEV), wl.normalize, wl.scale,
                                                          wl.temperature)
            torch.cuda.synchronize()
            assert_parity(p, oracle_probs(wl.Q, wl.C, wl.normalize, wl.scale, wl.temperature), "unfused " + wl.name)


def test_unfused_needs_aligned_inputs(cuda_lib):
    wl = workloads.random_case(2, 9, 513, 1, 2.0, 7, DEV)
    with pytest.raises(binding.CSError) as e:
        binding.cs_score_candidates_batch_unfused(wl.Q, wl.C, 1, 2.0, 1.0)
    assert e.value.status == binding.CS_ERR_BAD_PLAN


def test_unfused_guards(cuda_lib):
    B, K, D = 3, 64, 512
    wl = workloads.random_case(B, K, D, 1, 2.0, 8, DEV)
    pad = 64
    sbuf = torch.full((pad + B * K + pad,), 5555.0, device=DEV)
    obuf = torch.full((pad + B * K + pad,), 7777.0, device=DEV)
    staged = sbuf[pad:pad + B * K].view(B, K)
    out = obuf[pad:pad + B * K].view(B, K)
    binding.cs_score_candidates_batch_unfused(wl.Q, wl.C, 1, 2.0, 1.0, staged=staged, out=out)
    torch.cuda.synchronize()
    for buf, v in ((sbuf, 5555.0), (obuf, 7777.0)):
        assert torch.all(buf[:pad] == v) and torch.all(buf[pad + B * K:] == v)
    assert_parity(out, oracle_probs(wl.Q, wl.C, 1, 2.0, 1.0), "unfused guards")
