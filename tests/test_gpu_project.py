"""GPU parity of the tensor-core projections (tcgen05) and the fused
projected readout.

The page (PR #69 "cuda: add a fused candidate-scoring kernel for CLM and
Kev", opening table) scores projected vectors -- CLM's state_head(s) against
action_head(c), Kev's k(h_opts) against q(h_decide) -- and leaves the
projections to the caller; here they run on the tensor cores. Features and
weights are bfloat16; the oracle widens them exactly and projects in fp64.

Projection bound: a float32 accumulation of Din products is within
Din * 2^-24 * sum_i |h_i w_i| of the exact sum; the tests use 1e-4 * that
sum per element (well above the bound, far below any layout mistake, which
permutes or garbles whole columns). Probabilities: the usual 1e-4 / 1e-5.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from similarity_softmax_candidate_gb300 import binding
from tests._util import TEMPERED, assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _bf16(shape, seed, std=1.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def test_project_identity_weights_exact(cuda_lib):
    """W = [I; 0] (D=256 >= Din) returns H exactly in its first Din columns:
    any swizzle, descriptor or lane mistake would move or garble values."""
    for rows, Din in ((128, 64), (300, 128), (129, 256)):
        H = _bf16((rows, Din), rows + Din)
        W = torch.zeros((256, Din), dtype=torch.bfloat16)
        W[:Din] = torch.eye(Din, dtype=torch.bfloat16)
        P = binding.cs_project_rows(H.to(DEV), W.to(DEV))
        torch.cuda.synchronize()
        P = P.cpu()
        assert torch.equal(P[:, :Din], H.float()), f"rows={rows} Din={Din}"
        assert torch.all(P[:, Din:] == 0)


@pytest.mark.parametrize("D", [256, 512])
def test_project_rows_random(cuda_lib, D):
    for rows, Din in ((1, 64), (127, 512), (128, 512), (129, 512), (1000, 1024), (4096, 512)):
        H = _bf16((rows, Din), 10 + rows)
        W = _bf16((D, Din), 20 + Din, std=Din ** -0.5)
        P = binding.cs_project_rows(H.to(DEV), W.to(DEV))
        torch.cuda.synchronize()
        ref = oracle.project(H.float().numpy(), W.float().numpy())
        bound = 1e-4 * (np.abs(H.float().numpy()).astype(np.float64) @ np.abs(W.float().numpy()).astype(np.float64).T)
        err = np.abs(P.cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= bound + 1e-30), f"rows={rows} Din={Din} D={D}: max err {err.max():.3e}"


CASES = [(1, 5, 64, 256), (3, 128, 512, 256), (2, 129, 512, 512), (5, 255, 512, 512), (20, 255, 512, 512),
         (7, 1, 128, 256), (40, 64, 1024, 512)]


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_project_score_parity(cuda_lib, normalize):
    for B, K, Din, D in CASES:
        Hq = _bf16((B, Din), 100 + B)
        Hc = _bf16((B, K, Din), 200 + K)
        Wq = _bf16((D, Din), 300 + D, std=Din ** -0.5)
        Wc = _bf16((D, Din), 400 + D, std=Din ** -0.5)
        scale = 14.2857 if normalize else 0.0625
        qproj = torch.empty((B, D), device=DEV)
        p = binding.cs_project_score_batch(Hq.to(DEV), Wq.to(DEV), Hc.to(DEV), Wc.to(DEV), normalize, scale, 1.0,
                                           qproj=qproj)
        torch.cuda.synchronize()
        ref = oracle.project_score_batch(Hq.float().numpy(), Wq.float().numpy(), Hc.float().numpy(),
                                         Wc.float().numpy(), normalize, scale, 1.0)
        assert_parity(p, ref, f"projected B={B} K={K} Din={Din} D={D}")
        qref = oracle.project(Hq.float().numpy(), Wq.float().numpy())
        np.testing.assert_allclose(qproj.cpu().numpy(), qref, rtol=1e-3, atol=1e-3)
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_project_score_tempered(cuda_lib, normalize):
    """The projected readout forms its logit factor in its own epilogue, so
    it is checked with temperatures 0.05, 0.7 and 3 and negative scales. For
    the dot, the candidate head is scaled down so that the logits stay of a
    few units (projected features are about N(0,1), so a dot has spread
    sqrt(D))."""
    for B, K, Din, D in ((5, 255, 512, 512), (3, 128, 512, 256), (2, 7, 64, 256)):
        for scale, T in TEMPERED[normalize]:
            f = 1.0 if normalize else min(1.0, 3.0 * T / (abs(scale) * D ** 0.5))
            Hq = _bf16((B, Din), 110 + B)
            Hc = _bf16((B, K, Din), 210 + K)
            Wq = _bf16((D, Din), 310 + D, std=Din ** -0.5)
            Wc = _bf16((D, Din), 410 + D, std=f * Din ** -0.5)
            p = binding.cs_project_score_batch(Hq.to(DEV), Wq.to(DEV), Hc.to(DEV), Wc.to(DEV), normalize, scale, T)
            torch.cuda.synchronize()
            ref = oracle.project_score_batch(Hq.float().numpy(), Wq.float().numpy(), Hc.float().numpy(),
                                             Wc.float().numpy(), normalize, scale, T)
            assert_parity(p, ref, f"projected B={B} K={K} D={D} scale={scale} T={T}")
    assert binding.cs_device_status() == 0


def test_project_score_matches_scoring_of_projected_rows(cuda_lib):
    """Fused projection + scoring equals projecting with cs_project_rows and
    scoring with cs_score_candidates_batch (two paths through different
    kernels; agreement within float32 rounding)."""
    B, K, Din, D = 16, 255, 512, 512
    Hq, Hc = _bf16((B, Din), 1).to(DEV), _bf16((B, K, Din), 2).to(DEV)
    Wq, Wc = _bf16((D, Din), 3, Din ** -0.5).to(DEV), _bf16((D, Din), 4, Din ** -0.5).to(DEV)
    fused = binding.cs_project_score_batch(Hq, Wq, Hc, Wc, 1, 14.2857, 1.0)
    q = binding.cs_project_rows(Hq, Wq)
    c = binding.cs_project_rows(Hc.view(B * K, Din), Wc).view(B, K, D)
    composed = binding.cs_score_candidates_batch(q, c, 1, 14.2857, 1.0)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(fused - composed)).item() <= 1e-5


def _sample(n, first, last, rand, seed):
    rng = np.random.default_rng(seed)
    idx = set(range(min(first, n))) | set(range(max(0, n - last), n))
    idx |= set(rng.integers(0, n, size=rand).tolist())
    return np.array(sorted(idx))


@pytest.mark.parametrize("D", [256, 512])
def test_project_rows_many_tiles_per_cta(cuda_lib, D):
    """Enough rows that every CTA projects several tiles (each tensor-memory
    accumulator is reused many times) plus a ragged last tile; every row is
    written and sampled rows match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, Din = sms * 128 * 3 + 77, 512
    H = _bf16((rows, Din), 31)
    W = _bf16((D, Din), 32, std=Din ** -0.5)
    P = torch.full((rows, D), float("nan"), device=DEV)
    binding.cs_project_rows(H.to(DEV), W.to(DEV), out=P)
    torch.cuda.synchronize()
    P = P.cpu().numpy()
    assert np.isfinite(P).all(), "some projected rows were not written"
    idx = _sample(rows, 200, 200, 400, 33)
    Hs = H.float().numpy()[idx]
    ref = oracle.project(Hs, W.float().numpy())
    bound = 1e-4 * (np.abs(Hs).astype(np.float64) @ np.abs(W.float().numpy()).astype(np.float64).T)
    err = np.abs(P[idx].astype(np.float64) - ref)
    assert np.all(err <= bound + 1e-30), f"D={D}: max err {err.max():.3e}"
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("D,K", [(256, 100), (256, 255), (512, 255)])
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_project_score_many_questions_per_cta(cuda_lib, D, K, normalize):
    """Several questions per CTA: accumulators and logit buffers are reused;
    sampled questions match the oracle and every row is a distribution."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, Din = 3 * sms + 5, 512
    Hq, Hc = _bf16((B, Din), 41), _bf16((B, K, Din), 42)
    Wq, Wc = _bf16((D, Din), 43, std=Din ** -0.5), _bf16((D, Din), 44, std=Din ** -0.5)
    scale = 14.2857 if normalize else 0.0625
    p = torch.full((B, K), float("nan"), device=DEV)
    binding.cs_project_score_batch(Hq.to(DEV), Wq.to(DEV), Hc.to(DEV), Wc.to(DEV), normalize, scale, 1.0, out=p)
    torch.cuda.synchronize()
    p = p.cpu().numpy()
    assert np.isfinite(p).all()
    np.testing.assert_allclose(p.astype(np.float64).sum(axis=1), 1.0, atol=1e-5)
    idx = _sample(B, 3, 3, 10, 45)
    ref = oracle.project_score_batch(Hq.float().numpy()[idx], Wq.float().numpy(), Hc.float().numpy()[idx],
                                     Wc.float().numpy(), normalize, scale, 1.0)
    assert_parity(torch.from_numpy(p[idx]), ref, f"projected B={B} K={K} D={D} sampled")
    assert binding.cs_device_status() == 0


def test_project_score_benchmark_size(cuda_lib):
    """The projected readout at the size the benchmark times (4096 questions,
    K=255, Din=D=512, inputs drawn on the device), checked on sampled
    questions."""
    B, K, Din, D = 4096, 255, 512, 512
    g = torch.Generator(device=DEV)
    g.manual_seed(21)
    Hq = torch.randn(B, Din, device=DEV, generator=g).to(torch.bfloat16)
    Hc = torch.randn(B, K, Din, device=DEV, generator=g).to(torch.bfloat16)
    Wq = (torch.randn(D, Din, device=DEV, generator=g) * Din ** -0.5).to(torch.bfloat16)
    Wc = (torch.randn(D, Din, device=DEV, generator=g) * Din ** -0.5).to(torch.bfloat16)
    p = binding.cs_project_score_batch(Hq, Wq, Hc, Wc, 1, 14.285714, 1.0)
    torch.cuda.synchronize()
    idx = _sample(B, 2, 2, 8, 46)
    t = torch.from_numpy(idx).to(DEV)
    ref = oracle.project_score_batch(Hq[t].float().cpu().numpy(), Wq.float().cpu().numpy(),
                                     Hc[t].float().cpu().numpy(), Wc.float().cpu().numpy(), 1, 14.285714, 1.0)
    assert_parity(p[t], ref, "projected readout, benchmark size, sampled")
    sums = p.double().sum(dim=1)
    assert torch.max(torch.abs(sums - 1.0)).item() <= 1e-5
    assert binding.cs_device_status() == 0
