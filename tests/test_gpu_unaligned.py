"""GPU parity of rows the bulk copies cannot take whole: D not a multiple of
4 float32 (8 bfloat16) elements, or Q and C off a 16-byte boundary.

Such rows stream through the same bulk-copy ring as aligned ones, each copy
widened to the 16-byte granules around them (unaligned plans); the kernel
reads them in 4-byte units (float32 elements, bfloat16 pairs) from where
they landed, and a few questions take the DIRECT kernel's unit form. The page's float4 rules
("weighted RMS with float4 loads", on the page set's RMS-norm page) say
when 16-byte accesses are allowed; here they decide only the copy's span,
not the path. Each case is compared with the fp64 oracle (1e-4 per
probability, rows summing to 1 within 1e-5).
"""
from __future__ import annotations

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import assert_parity, oracle_probs, pairs_in_rotation, tempered_case

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _placed(t, offset_elems):
    """A copy of t starting offset_elems elements past a 256-byte boundary."""
    flat = torch.empty(t.numel() + offset_elems + 64, dtype=t.dtype, device=DEV)
    v = flat[offset_elems:offset_elems + t.numel()].view(t.shape)
    v.copy_(t)
    return v


SHAPES = [(300, 255, 510), (200, 64, 511), (160, 37, 13), (157, 200, 1), (170, 9, 3), (155, 100, 1025),
          (180, 33, 4097), (160, 5, 12289)]
OFFSETS = [(0, 0), (1, 1), (0, 3), (2, 1)]  # (Q, C) element offsets from a 16-byte boundary


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_many_unaligned_questions_take_the_stream_plan(cuda_lib, normalize):
    """Many questions (2B above the SM count) of odd D or misaligned rows:
    the automatic plan is the stream plan, and every question matches the
    oracle; shape i also takes (scale, temperature) pair i % 5."""
    pairs = pairs_in_rotation(normalize)
    for i, (B, K, D) in enumerate(SHAPES):
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 300 + B + K + D)
        for oq, oc in OFFSETS:
            if D % 4 == 0 and oq == 0 and oc == 0:
                continue
            Q, C = _placed(wl.Q.to(DEV), oq), _placed(wl.C.to(DEV), oc)
            plan = binding.cs_query_plan(Q, C, normalize)
            if D <= 8192:
                assert plan["plan"] == "stream", (B, K, D, oq, oc, plan)
            p = binding.cs_score_candidates_batch(Q, C, normalize, wl.scale, wl.temperature)
            torch.cuda.synchronize()
            assert_parity(p, oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature),
                          f"B={B} K={K} D={D} offsets q={oq} c={oc} plan={plan['plan']}")
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_forced_stream_and_cluster_plans_on_unaligned_rows(cuda_lib, normalize):
    """The stream plan with 1 and 2 CTAs (several questions per CTA, the
    ring wrapping many times) and the cluster plan with 2, 4 and 16 CTAs
    per question, on odd D and misaligned rows, few questions."""
    pairs = pairs_in_rotation(normalize)
    forced = [(binding.CS_PLAN_STREAM, 0, 1), (binding.CS_PLAN_STREAM, 0, 2), (binding.CS_PLAN_CLUSTER, 2, 0),
              (binding.CS_PLAN_CLUSTER, 4, 0), (binding.CS_PLAN_CLUSTER, 16, 0), (binding.CS_PLAN_CLUSTER, 0, 0)]
    for i, (B, K, D, oq, oc) in enumerate(((3, 255, 510, 0, 0), (2, 64, 512, 1, 3), (5, 17, 7, 2, 1),
                                           (2, 200, 1031, 3, 2))):
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 400 + B + K + D)
        Q, C = _placed(wl.Q.to(DEV), oq), _placed(wl.C.to(DEV), oc)
        ref = oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature)
        for kind, cluster, ctas in forced:
            if cluster > K or ctas > B:
                continue
            p = binding.cs_score_candidates_batch_plan(Q, C, normalize, wl.scale, wl.temperature, kind, cluster,
                                                       ctas)
            torch.cuda.synchronize()
            assert_parity(p, ref, f"plan {kind}/{cluster}/{ctas} B={B} K={K} D={D} q+{oq} c+{oc}")
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_unaligned_bf16(cuda_lib, normalize):
    """bfloat16 candidates with D not a multiple of 8 or C off a 16-byte
    boundary by 1 to 7 elements (2-byte offsets)."""
    pairs = pairs_in_rotation(normalize)
    for i, (B, K, D, oq, oc) in enumerate(((300, 255, 510, 0, 0), (200, 64, 512, 1, 1), (160, 33, 13, 0, 5),
                                           (170, 255, 1027, 3, 7), (3, 64, 509, 0, 3))):
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 500 + B + K + D)
        Cb = wl.C.to(torch.bfloat16)
        Q, C = _placed(wl.Q.to(DEV), oq), _placed(Cb.to(DEV), oc)
        p = binding.cs_score_candidates_batch_bf16(Q, C, normalize, wl.scale, wl.temperature)
        torch.cuda.synchronize()
        assert_parity(p, oracle_probs(wl.Q, Cb.float(), normalize, wl.scale, wl.temperature),
                      f"bf16 B={B} K={K} D={D} q+{oq} c+{oc}")
    assert binding.cs_device_status() == 0


# D either side of the unit-wise form's sizes (4, 8 or 16 four-byte units a
# lane; float32 units are elements, bfloat16 units element pairs, an odd D's
# last element added apart) and past its last one (q from shared memory).
UNIT_EDGES = {"f32": [1, 2, 127, 128, 129, 255, 256, 257, 511, 512, 513],
              "bf16": [1, 2, 3, 255, 256, 257, 258, 511, 512, 513, 1023, 1024, 1025, 1026]}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_unit_form_sizes(cuda_lib, dtype, normalize):
    """Unaligned rows at every D where the unit-wise form changes shape
    (units a lane, the guaranteed-inside units, the odd bfloat16 element),
    with rows starting on even and odd 2-byte offsets (bfloat16) and every
    4-byte offset (float32); each question against the oracle."""
    pairs = pairs_in_rotation(normalize)
    bf16 = dtype == "bf16"
    for i, D in enumerate(UNIT_EDGES[dtype]):
        B, K = 40, 23 + i
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 600 + D + (7 if bf16 else 0))
        Cr = wl.C.to(torch.bfloat16) if bf16 else wl.C
        ref = oracle_probs(wl.Q, Cr.float(), normalize, wl.scale, wl.temperature)
        for oq, oc in ((1, 1), (0, 3), (3, 2), (2, 5) if bf16 else (2, 0)):
            Q, C = _placed(wl.Q.to(DEV), oq), _placed(Cr.to(DEV), oc)
            fn = binding.cs_score_candidates_batch_bf16 if bf16 else binding.cs_score_candidates_batch
            p = fn(Q, C, normalize, wl.scale, wl.temperature)
            torch.cuda.synchronize()
            assert_parity(p, ref, f"{dtype} B={B} K={K} D={D} q+{oq} c+{oc}")
    assert binding.cs_device_status() == 0


def test_unaligned_ragged(cuda_lib):
    """A ragged batch of odd D, and one whose C is off a 16-byte boundary:
    many questions (the stream plan), a few short ones (DIRECT) and a few
    long ones (a cluster plan)."""
    for B, D, oc in ((400, 513, 0), (300, 512, 1), (12, 255, 3), (8, 1001, 1)):
        wl = workloads.ragged(B, D, 1, 14.2857, 60 + B, "cpu")
        Q, C = wl.Q.to(DEV), _placed(wl.C.to(DEV), oc)
        p = binding.cs_score_candidates_ragged(Q, C, wl.offsets.to(DEV), 1, wl.scale, 1.0)
        torch.cuda.synchronize()
        p = p.cpu()
        off = wl.offsets.tolist()
        for b in range(0, B, max(1, B // 40)):
            o0, o1 = off[b], off[b + 1]
            ref = oracle_probs(wl.Q[b:b + 1], wl.C[o0:o1][None], 1, wl.scale, 1.0)
            assert_parity(p[o0:o1][None], ref, f"ragged D={D} c+{oc} question {b}")
    assert binding.cs_device_status() == 0


def test_unaligned_ragged_bf16(cuda_lib):
    """Ragged bfloat16 batches off 16-byte boundaries: C one element off with
    an even D (every row read from the word before), an odd D (rows
    alternating between whole-word and split pairs), and D past the
    register form (q from shared memory)."""
    for B, D, oc, normalize in ((300, 512, 1, 1), (250, 255, 0, 0), (200, 777, 3, 1), (60, 2562, 1, 0)):
        wl = workloads.ragged(B, D, normalize, 14.2857 if normalize else 0.0625, 80 + B + D, "cpu")
        Cb = wl.C.to(torch.bfloat16)
        Q, C = wl.Q.to(DEV), _placed(Cb.to(DEV), oc)
        p = binding.cs_score_candidates_ragged(Q, C, wl.offsets.to(DEV), normalize, wl.scale, 1.0)
        torch.cuda.synchronize()
        p = p.cpu()
        off = wl.offsets.tolist()
        for b in range(0, B, max(1, B // 30)):
            o0, o1 = off[b], off[b + 1]
            ref = oracle_probs(wl.Q[b:b + 1], Cb[o0:o1].float()[None], normalize, wl.scale, 1.0)
            assert_parity(p[o0:o1][None], ref, f"ragged bf16 D={D} c+{oc} question {b}")
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("case", ["odd_d", "misaligned"])
def test_unaligned_throughput_workloads_full_size(cuda_lib, case):
    """The two unaligned throughput workloads the benchmark times, 4096
    questions of K=255 (D=510 float32, and D=512 with Q and C one element
    past a 16-byte boundary), cosine and dot, in one launch each: every row
    sums to 1 and sampled questions match the oracle."""
    B, K = 4096, 255
    D = 510 if case == "odd_d" else 512
    off = 0 if case == "odd_d" else 1
    g = torch.Generator(device=DEV)
    g.manual_seed(91)
    Cflat = torch.empty(B * K * D + 64, device=DEV)
    C = Cflat[off:off + B * K * D].view(B, K, D)
    for b0 in range(0, B, 512):
        C[b0:b0 + 512].normal_(generator=g)
    Qflat = torch.empty(B * D + 64, device=DEV)
    Q = Qflat[off:off + B * D].view(B, D)
    Q.normal_(generator=g)
    assert binding.cs_query_plan(Q, C, 1)["plan"] == "stream"
    sel = torch.tensor(sorted(set(range(0, B, 97)) | {0, B - 1}), device=DEV)
    for normalize, scale in ((1, workloads.CLM_SCALE), (0, workloads.KEV_SCALE)):
        p = binding.cs_score_candidates_batch(Q, C, normalize, scale, 1.0)
        torch.cuda.synchronize()
        assert torch.isfinite(p).all()
        assert torch.max(torch.abs(p.double().sum(dim=1) - 1.0)).item() <= 1e-5
        ref = oracle_probs(Q.index_select(0, sel), C.index_select(0, sel), normalize, scale, 1.0)
        assert_parity(p.index_select(0, sel), ref, f"{case} normalize={normalize}")
    del C, Cflat
    torch.cuda.empty_cache()
    assert binding.cs_device_status() == 0
