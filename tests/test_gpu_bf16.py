"""GPU parity of the bfloat16-candidate readout.

Candidates stored as bfloat16, widened exactly to float32 and accumulated in
float32: the result must be the float32 readout of the bfloat16-rounded
candidates, so the fp64 oracle is fed C.float() (exact) and the same 1e-4 /
1e-5 bar applies. bfloat16 storage is an extension of the method of PR #69
"cuda: add a fused candidate-scoring kernel for CLM and Kev", whose kernel
reads float32.
"""
from __future__ import annotations

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import ATOL, assert_parity, oracle_probs, pairs_in_rotation, tempered_case

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

SHAPES = [(1, 5, 512), (1, 64, 512), (1, 255, 512), (8, 255, 512), (1, 255, 2560), (300, 255, 512), (3, 37, 136),
          (2, 200, 1032), (5, 1, 8), (4, 17, 4104), (2, 33, 516), (3, 9, 13)]


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_bf16_parity(cuda_lib, normalize):
    """Shape i takes (scale, temperature) pair i % 5 (temperature 1, then
    0.7, 3 and 0.05 with positive and negative scales)."""
    pairs = pairs_in_rotation(normalize)
    for i, (B, K, D) in enumerate(SHAPES):
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 700 + B + K + D)
        sc, T = wl.scale, wl.temperature
        Cb = wl.C.to(torch.bfloat16)
        p = binding.cs_score_candidates_batch_bf16(wl.Q.to(DEV), Cb.to(DEV), normalize, sc, T)
        torch.cuda.synchronize()
        assert_parity(p, oracle_probs(wl.Q, Cb.float(), normalize, sc, T), f"bf16 B={B} K={K} D={D} scale={sc} T={T}")


def test_bf16_single_matches_batch(cuda_lib):
    for wl in workloads.clm_k5("cpu") + workloads.kev_k255("cpu"):
        Cb = wl.C.to(torch.bfloat16).to(DEV)
        Q = wl.Q.to(DEV)
        ps = binding.cs_score_candidates_bf16(Q[0], Cb[0], wl.normalize, wl.scale, wl.temperature)
        pb = binding.cs_score_candidates_batch_bf16(Q, Cb, wl.normalize, wl.scale, wl.temperature)
        torch.cuda.synchronize()
        ref = oracle_probs(wl.Q, wl.C.to(torch.bfloat16).float(), wl.normalize, wl.scale, wl.temperature)
        assert_parity(ps[None], ref, wl.name + " bf16 single")
        assert_parity(pb, ref, wl.name + " bf16 batch")
        assert torch.max(torch.abs(ps - pb[0])).item() <= ATOL


def test_bf16_throughput_workload_full_size(cuda_lib):
    """16384 x 255 x 512 candidates in bfloat16 (4.3 GB), four launches of
    4096 questions; every row sums to 1, a sample of questions is compared
    with the oracle."""
    Q = workloads.normal((workloads.THROUGHPUT_B, 512), 44, DEV)
    C = torch.empty((workloads.THROUGHPUT_B, 255, 512), device=DEV, dtype=torch.bfloat16)
    g = torch.Generator(device=DEV)
    g.manual_seed(45)
    for b0 in range(0, workloads.THROUGHPUT_B, 2048):
        C[b0:b0 + 2048] = torch.randn((2048, 255, 512), generator=g, device=DEV).to(torch.bfloat16)
    out = torch.empty((workloads.THROUGHPUT_B, 255), device=DEV)
    chunk = workloads.THROUGHPUT_CHUNK
    for normalize, scale in ((1, workloads.CLM_SCALE), (0, workloads.KEV_SCALE)):
        for b0 in range(0, workloads.THROUGHPUT_B, chunk):
            binding.cs_score_candidates_batch_bf16(Q[b0:b0 + chunk], C[b0:b0 + chunk], normalize, scale, 1.0,
                                                   out=out[b0:b0 + chunk])
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.max(torch.abs(out.double().sum(dim=1) - 1.0)).item() <= 1e-5
        sel = torch.tensor(sorted(set(range(0, workloads.THROUGHPUT_B, 97)) | {0, workloads.THROUGHPUT_B - 1}),
                           device=DEV)
        ref = oracle_probs(Q.index_select(0, sel), C.index_select(0, sel).float(), normalize, scale, 1.0)
        assert_parity(out.index_select(0, sel), ref, f"bf16 throughput normalize={normalize}")
    del C
    torch.cuda.empty_cache()


def test_bf16_rejects_float32_candidates(cuda_lib):
    wl = workloads.random_case(2, 5, 512, 1, 2.0, 3, DEV)
    with pytest.raises(TypeError):
        binding.cs_score_candidates_batch_bf16(wl.Q, wl.C, 1, 2.0, 1.0)
