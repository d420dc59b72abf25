"""GPU parity of ragged batches (per-question K_b through an offsets array).

Each question of a ragged batch is the readout of PR #69 "cuda: add a fused
candidate-scoring kernel for CLM and Kev" on its own K_b candidates, so every
question is compared with the fp64 oracle on exactly its rows. The ragged
layout is an extension: the page's call takes one K per batch.
"""
from __future__ import annotations

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import TEMPERED, assert_parity, oracle_probs, pairs_in_rotation

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _check_all(wl, p, Cref=None, sample=None):
    off = wl.offsets.cpu().tolist()
    C = wl.C if Cref is None else Cref
    idx = range(wl.B) if sample is None else sample
    for b in idx:
        o0, o1 = off[b], off[b + 1]
        ref = oracle_probs(wl.Q[b:b + 1], C[o0:o1][None], wl.normalize, wl.scale, wl.temperature)
        assert_parity(p[o0:o1][None], ref, f"{wl.name} question {b} (K={o1 - o0})")


CASES = [(1, 512, 1, 255), (3, 512, 1, 255), (8, 512, 200, 255), (40, 512, 1, 64), (300, 512, 1, 255),
         (5, 2560, 100, 255), (200, 128, 1, 8), (7, 513, 1, 255), (3, 12, 250, 255)]


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_ragged_parity(cuda_lib, normalize):
    """Case i takes (scale, temperature) pair i % 5 (temperature 1, then 0.7,
    3 and 0.05 with positive and negative scales); dot candidates of a
    tempered pair are rescaled to keep the logits of a few units."""
    pairs = pairs_in_rotation(normalize)
    for i, (B, D, kmin, kmax) in enumerate(CASES):
        scale, T = pairs[i % len(pairs)]
        wl = workloads.ragged(B, D, normalize, scale, 300 + B + D + kmin, "cpu", kmin=kmin, kmax=kmax)
        wl.temperature = T
        if not normalize and T != 1.0:
            wl.C.mul_(min(1.0, 3.0 * T / (abs(scale) * D ** 0.5)))
        p = binding.cs_score_candidates_ragged(wl.Q.to(DEV), wl.C.to(DEV), wl.offsets.to(DEV), normalize, scale, T)
        torch.cuda.synchronize()
        _check_all(wl, p.cpu())


def test_ragged_bf16(cuda_lib):
    for i, (B, D) in enumerate(((3, 512), (300, 512), (9, 1032))):
        scale, T = TEMPERED[1][i]
        wl = workloads.ragged(B, D, 1, scale, 40 + B, "cpu")
        wl.temperature = T
        Cb = wl.C.to(torch.bfloat16)
        p = binding.cs_score_candidates_ragged(wl.Q.to(DEV), Cb.to(DEV), wl.offsets.to(DEV), 1, scale, T)
        torch.cuda.synchronize()
        _check_all(wl, p.cpu(), Cref=Cb.float())


def test_ragged_uniform_matches_batch(cuda_lib):
    """A ragged batch whose K_b are all equal is the plain batch."""
    B, K, D = 50, 255, 512
    wl = workloads.random_case(B, K, D, 1, 14.2857, 61, DEV)
    offsets = torch.arange(B + 1, device=DEV, dtype=torch.int64) * K
    pr = binding.cs_score_candidates_ragged(wl.Q, wl.C.view(B * K, D), offsets, 1, wl.scale, 1.0)
    pb = binding.cs_score_candidates_batch(wl.Q, wl.C, 1, wl.scale, 1.0)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(pr.view(B, K) - pb)).item() <= 1e-6


def test_ragged_bad_offsets_are_skipped_and_flagged(cuda_lib):
    """A question whose offsets give K_b = 300 (> 255) is skipped: its rows of
    out keep their old contents, the other questions are scored, and the
    device status word says so. The kernel checks each question's range
    before touching it, so no access leaves the buffers."""
    # DIRECT, CLUSTER (rows too long for the DIRECT kernel), STREAM and scalar plans
    for B, D in ((6, 512), (3, 4100), (200, 512), (5, 513)):
        wl = workloads.ragged(B, D, 1, 14.2857, 77 + B, "cpu", kmin=1, kmax=40)
        off = wl.offsets.clone()
        bad = B // 2
        k = (off[1:] - off[:-1]).clone()
        k[bad] = 300
        off[1:] = torch.cumsum(k, 0)
        total = int(off[-1])
        C = workloads.normal((total, D), 5, "cpu")
        wl2 = workloads.RaggedWorkload("bad", wl.Q, C, off, 1, wl.scale)
        binding.cs_device_status(clear=True)
        out = torch.full((total,), 4242.0, device=DEV)
        binding.cs_score_candidates_ragged(wl.Q.to(DEV), C.to(DEV), off.to(DEV), 1, wl.scale, 1.0, out=out)
        torch.cuda.synchronize()
        assert binding.cs_device_status(clear=True) == 4
        o = off.tolist()
        assert torch.all(out[o[bad]:o[bad + 1]] == 4242.0)
        good = [b for b in range(B) if b != bad]
        _check_all(wl2, out.cpu(), sample=good)


def test_ragged_throughput_workload(cuda_lib):
    """16384 questions with K_b uniform in [1, 255] (about 2.1 M rows, 4.3 GB):
    every question's probabilities sum to 1; a sample is compared with the
    oracle."""
    wl = workloads.ragged(16384, 512, 1, workloads.CLM_SCALE, 12, DEV)
    p = binding.cs_score_candidates_ragged(wl.Q, wl.C, wl.offsets, 1, wl.scale, 1.0)
    torch.cuda.synchronize()
    assert torch.isfinite(p).all()
    seg = torch.repeat_interleave(torch.arange(wl.B, device=DEV), wl.offsets[1:] - wl.offsets[:-1])
    sums = torch.zeros(wl.B, device=DEV, dtype=torch.float64).index_add_(0, seg, p.double())
    assert torch.max(torch.abs(sums - 1.0)).item() <= 1e-5
    sample = sorted(set(range(0, wl.B, 151)) | {0, wl.B - 1})
    off = wl.offsets.cpu().tolist()
    for b in sample:
        o0, o1 = off[b], off[b + 1]
        ref = oracle_probs(wl.Q[b:b + 1], wl.C[o0:o1][None], 1, wl.scale, 1.0)
        assert_parity(p[o0:o1][None], ref, f"ragged throughput question {b}")
    assert binding.cs_device_status() == 0
