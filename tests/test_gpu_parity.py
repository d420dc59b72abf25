"""GPU parity: the CUDA library, called through its C ABI, against the fp64
oracle on the same seeded inputs.

Groups follow PR #69 "cuda: add a fused candidate-scoring kernel for CLM and
Kev", "Verified on hardware": the fixed cases (single candidate, identical
candidates, zero candidate, overflow), the batch path (1, 8, 4 and 3
questions with K up to 255 and D up to 256, single-question calls through
cs_score_candidates), plus every execution plan on shapes with ragged tails,
the workloads of "What it is worth" at their full sizes, and output guards.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import ATOL, TEMPERED, assert_parity, oracle_probs, pairs_in_rotation, tempered_case

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(wl, entry="auto", out=None):
    Q, C = wl.Q.to(DEV), wl.C.to(DEV)
    if entry == "single" or (entry == "auto" and wl.B == 1):
        o = binding.cs_score_candidates(Q[0], C[0], wl.normalize, wl.scale, wl.temperature,
                                        out=None if out is None else out[0])
        torch.cuda.synchronize()
        return o[None, :]
    o = binding.cs_score_candidates_batch(Q, C, wl.normalize, wl.scale, wl.temperature, out=out)
    torch.cuda.synchronize()
    return o


def _config_cases():
    cases = []
    for name in ("clm_k5", "clm_k64", "clm_batch8", "kev_k255"):
        for wl in workloads.CONFIGS[name]("cpu"):
            cases.append(wl)
    return cases


CONFIG_CASES = _config_cases()


@pytest.mark.parametrize("wl", CONFIG_CASES, ids=[w.name for w in CONFIG_CASES])
def test_workload_parity(cuda_lib, wl):
    p = _run(wl)
    assert_parity(p, oracle_probs(wl.Q, wl.C, wl.normalize, wl.scale, wl.temperature), wl.name)


def test_single_and_batch_entry_points_agree(cuda_lib):
    for wl in CONFIG_CASES:
        if wl.B != 1:
            continue
        ref = oracle_probs(wl.Q, wl.C, wl.normalize, wl.scale, wl.temperature)
        ps = _run(wl, "single")
        pb = _run(wl, "batch")
        assert_parity(ps, ref, wl.name + " single")
        assert_parity(pb, ref, wl.name + " batch")
        assert torch.max(torch.abs(ps - pb)).item() <= ATOL


def test_degenerate_cases(cuda_lib):
    # K = 1 gives exactly 1; identical candidates give 1/K; zero query gives uniform
    single = workloads.random_case(3, 1, 512, 1, workloads.CLM_SCALE, 11)
    p = _run(single)
    assert torch.all(p == 1.0)
    for normalize in (0, 1):
        same = workloads.random_case(2, 64, 512, normalize, workloads.CLM_SCALE, 12)
        same.C[:] = same.C[:, :1, :].clone()
        p = _run(same)
        assert torch.max(torch.abs(p - 1.0 / 64)).item() <= 1e-7
        zq = workloads.random_case(2, 255, 512, normalize, workloads.CLM_SCALE, 13)
        zq.Q.zero_()
        p = _run(zq)
        assert torch.max(torch.abs(p - 1.0 / 255)).item() <= 1e-7
    # all-zero candidates under cosine: every logit is 0
    zc = workloads.random_case(2, 17, 512, 1, workloads.CLM_SCALE, 14)
    zc.C.zero_()
    assert torch.max(torch.abs(_run(zc) - 1.0 / 17)).item() <= 1e-7


def test_golden_hand_cases(cuda_lib):
    import json
    import os
    from scipy.special import softmax
    with open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = torch.tensor(c["q"], dtype=torch.float32, device=DEV)
        C = torch.tensor(c["C"], dtype=torch.float32, device=DEV)
        p = binding.cs_score_candidates(q, C, c["normalize"], c["scale"], c["temperature"])
        torch.cuda.synchronize()
        expected = softmax(np.array(c["expected_logits"], dtype=np.float64))
        assert_parity(p[None, :], expected[None, :], c["name"])


@pytest.mark.parametrize("B", [1, 8, 4, 3])
def test_page_batch_group(cuda_lib, B):
    """The page's batch group: K up to 255 and D up to 256; B = 1 goes
    through the single-question entry point, the rest through the batch one.
    Each shape runs at the page's scale and temperature 1 and at every
    tempered pair (temperatures 0.05, 0.7 and 3, negative scales)."""
    rng = np.random.default_rng(B)
    for normalize in (0, 1):
        for K, D in ((255, 256), (int(rng.integers(1, 256)), int(rng.integers(1, 257))), (7, 3)):
            for pair in pairs_in_rotation(normalize):
                wl = tempered_case(B, K, D, normalize, pair, 100 + K + D)
                p = _run(wl)
                assert_parity(p, oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature),
                              f"B={B} K={K} D={D} scale={wl.scale} T={wl.temperature}")


PLAN_SHAPES = [
    (3, 255, 512), (2, 37, 132), (5, 1, 4), (1, 64, 2560), (2, 200, 1028), (4, 17, 4100),
    (7, 255, 128), (3, 33, 12), (2, 255, 1024), (1, 255, 2560), (9, 100, 16),
]

PLANS = [
    ("stream_auto", binding.CS_PLAN_STREAM, 0, 0),
    ("stream_1cta", binding.CS_PLAN_STREAM, 0, 1),
    ("stream_2cta", binding.CS_PLAN_STREAM, 0, 2),
    ("cluster_auto", binding.CS_PLAN_CLUSTER, 0, 0),
    ("cluster_1", binding.CS_PLAN_CLUSTER, 1, 0),
    ("cluster_2", binding.CS_PLAN_CLUSTER, 2, 0),
    ("cluster_3", binding.CS_PLAN_CLUSTER, 3, 0),
    ("cluster_8", binding.CS_PLAN_CLUSTER, 8, 0),
    ("cluster_16", binding.CS_PLAN_CLUSTER, 16, 0),
    ("generic", binding.CS_PLAN_GENERIC, 0, 0),
    ("generic_2", binding.CS_PLAN_GENERIC, 2, 0),
    ("generic_5", binding.CS_PLAN_GENERIC, 5, 0),
    ("generic_16", binding.CS_PLAN_GENERIC, 16, 0),
    ("direct_auto", binding.CS_PLAN_DIRECT, 0, 0),
    ("direct_1", binding.CS_PLAN_DIRECT, 1, 0),
    ("direct_3", binding.CS_PLAN_DIRECT, 3, 0),
    ("direct_8", binding.CS_PLAN_DIRECT, 8, 0),
    ("direct_16", binding.CS_PLAN_DIRECT, 16, 0),
]
# shapes a DIRECT plan cannot take must be refused, not run: at most 32 rows
# per CTA with q in registers (D <= 512), 16 with q in shared memory
# (D <= 2560), float32 rows of whole 16-byte chunks


def _direct_row_limit(D):
    if D % 4:
        return 0
    return 32 if D <= 512 else 16 if D <= 2560 else 0


def _plan_eligible(kind, cluster, K, D):
    """False where a forced DIRECT plan must be refused rather than run."""
    if kind != binding.CS_PLAN_DIRECT:
        return True
    lim = _direct_row_limit(D)
    g = cluster or next((x for x in (1, 2, 4, 8, 16) if lim and -(-K // x) <= lim), 16)
    return lim > 0 and -(-K // g) <= lim and g <= K


@pytest.mark.parametrize("plan", PLANS, ids=[p[0] for p in PLANS])
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_every_plan(cuda_lib, plan, normalize):
    """Every forced plan on shapes with ragged tails. Shape i takes the
    (scale, temperature) pair i % 5 -- the page's scale at temperature 1,
    then temperatures 0.7, 3 and 0.05 with positive and negative scales --
    so each plan meets every pair."""
    _, kind, cluster, ctas = plan
    pairs = pairs_in_rotation(normalize)
    for i, (B, K, D) in enumerate(PLAN_SHAPES):
        if cluster > K or ctas > B:
            continue
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 1000 + B * K + D)
        Q, C = wl.Q.to(DEV), wl.C.to(DEV)
        if not _plan_eligible(kind, cluster, K, D):
            with pytest.raises(binding.CSError):
                binding.cs_score_candidates_batch_plan(Q, C, normalize, wl.scale, wl.temperature, kind, cluster,
                                                       ctas)
            continue
        p = binding.cs_score_candidates_batch_plan(Q, C, normalize, wl.scale, wl.temperature, kind, cluster, ctas)
        torch.cuda.synchronize()
        assert_parity(p, oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature),
                      f"{plan[0]} B={B} K={K} D={D} scale={wl.scale} T={wl.temperature}")


TEMPERED_PLAN_SHAPES = [(3, 255, 512), (2, 200, 1028), (9, 100, 16)]


@pytest.mark.parametrize("plan", PLANS, ids=[p[0] for p in PLANS])
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_every_plan_every_tempered_pair(cuda_lib, plan, normalize):
    """Every forced plan with every tempered pair on the same shapes: the
    factor scale / temperature is formed in each kernel's own code, so each
    is checked with temperatures 0.05, 0.7 and 3 and with negative scales."""
    _, kind, cluster, ctas = plan
    for B, K, D in TEMPERED_PLAN_SHAPES:
        if cluster > K or ctas > B or not _plan_eligible(kind, cluster, K, D):
            continue
        for pair in TEMPERED[normalize]:
            wl = tempered_case(B, K, D, normalize, pair, 2000 + B * K + D)
            Q, C = wl.Q.to(DEV), wl.C.to(DEV)
            p = binding.cs_score_candidates_batch_plan(Q, C, normalize, wl.scale, wl.temperature, kind, cluster,
                                                       ctas)
            torch.cuda.synchronize()
            assert_parity(p, oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature),
                          f"{plan[0]} B={B} K={K} D={D} scale={wl.scale} T={wl.temperature}")


def _off_by_one(wl):
    """Copies of wl's Q and C one float past a 16-byte boundary."""
    Qb = torch.empty(wl.B * wl.D + 1, device=DEV)
    Cb = torch.empty(wl.B * wl.K * wl.D + 1, device=DEV)
    Q = Qb[1:].view(wl.B, wl.D)
    C = Cb[1:].view(wl.B, wl.K, wl.D)
    Q.copy_(wl.Q)
    C.copy_(wl.C)
    return Q, C


def test_few_unaligned_or_odd_questions(cuda_lib):
    """A few questions whose rows the bulk copies cannot take whole: the
    DIRECT plan reads rows of up to 512 float32 elements in 4-byte units;
    longer ones take the stream kernel's cluster plan (aligned spans). Every
    plan that takes them matches the oracle."""
    for normalize in (0, 1):
        # odd D past the unit form: a cluster plan; DIRECT refuses it
        wl = workloads.random_case(3, 255, 513, normalize, 2.0, 21)
        Q, C = wl.Q.to(DEV), wl.C.to(DEV)
        assert binding.cs_query_plan(Q, C, normalize)["plan"] == "cluster"
        ref = oracle_probs(wl.Q, wl.C, normalize, 2.0, 1.0)
        assert_parity(_run(wl), ref, "odd D")
        with pytest.raises(binding.CSError):
            binding.cs_score_candidates_batch_plan(Q, C, normalize, 2.0, 1.0, binding.CS_PLAN_DIRECT)
        p = binding.cs_score_candidates_batch_plan(Q, C, normalize, 2.0, 1.0, binding.CS_PLAN_GENERIC, 4)
        torch.cuda.synchronize()
        assert_parity(p, ref, "odd D, scalar plan")
        # odd D and pointers 4 bytes past a 16-byte boundary, within the unit form
        for D in (511, 512):
            wl = workloads.random_case(2, 64, D, normalize, 2.0, 22 + D)
            Q, C = _off_by_one(wl)
            ref = oracle_probs(wl.Q, wl.C, normalize, 2.0, 1.0)
            plan = binding.cs_query_plan(Q, C, normalize)
            assert plan["plan"] == "direct", plan
            p = binding.cs_score_candidates_batch(Q, C, normalize, 2.0, 1.0)
            torch.cuda.synchronize()
            assert_parity(p, ref, f"unaligned D={D}, DIRECT plan")
            # the stream and scalar plans take them too
            for kind in (binding.CS_PLAN_STREAM, binding.CS_PLAN_GENERIC):
                p = binding.cs_score_candidates_batch_plan(Q, C, normalize, 2.0, 1.0, kind)
                torch.cuda.synchronize()
                assert_parity(p, ref, f"unaligned D={D}, plan {kind}")


@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_direct_plan_on_unaligned_rows(cuda_lib, normalize):
    """The DIRECT plan's 4-byte-unit form at every cluster size, on rows off
    16-byte boundaries and of odd length: float32 at D either side of its
    unit counts, bfloat16 with C on even and odd 2-byte boundaries (rows
    read from the word before). Each question against the oracle; a
    ragged batch too."""
    pairs = pairs_in_rotation(normalize)
    cases = [(1, 255, 512, 1, 1, False), (3, 64, 511, 0, 0, False), (2, 37, 129, 2, 3, False),
             (1, 200, 3, 0, 1, False), (1, 255, 512, 1, 1, True), (4, 100, 1024, 0, 3, True),
             (2, 70, 258, 1, 2, True), (1, 31, 2, 0, 5, True)]
    for i, (B, K, D, oq, oc, bf16) in enumerate(cases):
        wl = tempered_case(B, K, D, normalize, pairs[i % len(pairs)], 900 + B + K + D)
        Cr = wl.C.to(torch.bfloat16) if bf16 else wl.C
        ref = oracle_probs(wl.Q, Cr.float(), normalize, wl.scale, wl.temperature)
        Qb = torch.empty(B * D + oq + 8, device=DEV)
        Cb = torch.empty(B * K * D + oc + 8, device=DEV, dtype=Cr.dtype)
        Q, C = Qb[oq:oq + B * D].view(B, D), Cb[oc:oc + B * K * D].view(B, K, D)
        Q.copy_(wl.Q)
        C.copy_(Cr)
        what = f"B={B} K={K} D={D} q+{oq} c+{oc} bf16={bf16}"
        if bf16:
            p = binding.cs_score_candidates_batch_bf16(Q, C, normalize, wl.scale, wl.temperature)
            torch.cuda.synchronize()
            assert_parity(p, ref, "auto " + what)
            continue
        assert binding.cs_query_plan(Q, C, normalize)["plan"] == "direct", what
        for G in (0, 1, 2, 4, 8, 16):
            if G > K or (G and (K + G - 1) // G > 32):
                continue
            p = binding.cs_score_candidates_batch_plan(Q, C, normalize, wl.scale, wl.temperature,
                                                       binding.CS_PLAN_DIRECT, G)
            torch.cuda.synchronize()
            assert_parity(p, ref, f"DIRECT G={G} " + what)
    rw = workloads.ragged(6, 300, 1, 14.2857, 77, "cpu", kmax=60)
    Cb = torch.empty(rw.C.numel() + 8, device=DEV)
    C = Cb[1:1 + rw.C.numel()].view(rw.C.shape)
    C.copy_(rw.C)
    p = binding.cs_score_candidates_ragged(rw.Q.to(DEV), C, rw.offsets.to(DEV), 1, rw.scale, 1.0)
    torch.cuda.synchronize()
    p = p.cpu()
    off = rw.offsets.tolist()
    for b in range(rw.B):
        ref = oracle_probs(rw.Q[b:b + 1], rw.C[off[b]:off[b + 1]][None], 1, rw.scale, 1.0)
        assert_parity(p[off[b]:off[b + 1]][None], ref, f"ragged unaligned DIRECT question {b}")
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("misaligned", [False, True], ids=["odd_d", "misaligned"])
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_scalar_plan_over_a_cluster(cuda_lib, misaligned, normalize):
    """One or a few questions whose rows the bulk copies cannot take (odd D,
    or pointers off a 16-byte boundary): the scalar plan spreads each
    question over a cluster and combines the softmax across its CTAs. Its
    result matches the oracle, and the one-CTA scalar plan's within float32
    rounding, for every cluster size the planner or a caller may pick."""
    for B, K, D in ((1, 255, 510 if not misaligned else 512), (3, 64, 511 if not misaligned else 256), (1, 16, 1001)):
        for pair in pairs_in_rotation(normalize):
            wl = tempered_case(B, K, D, normalize, pair, 700 + B + K + D)
            sc, T = wl.scale, wl.temperature
            if misaligned:
                Qb = torch.empty(B * D + 1, device=DEV)
                Cb = torch.empty(B * K * D + 1, device=DEV)
                Q, C = Qb[1:].view(B, D), Cb[1:].view(B, K, D)
                Q.copy_(wl.Q)
                C.copy_(wl.C)
            else:
                Q, C = wl.Q.to(DEV), wl.C.to(DEV)
            ref = oracle_probs(wl.Q, wl.C, normalize, sc, T)
            what = f"B={B} K={K} D={D} scale={sc} T={T}"
            one = binding.cs_score_candidates_batch_plan(Q, C, normalize, sc, T, binding.CS_PLAN_GENERIC, 1)
            p = (binding.cs_score_candidates(Q[0], C[0], normalize, sc, T)[None]
                 if B == 1 else binding.cs_score_candidates_batch(Q, C, normalize, sc, T))
            torch.cuda.synchronize()
            assert_parity(p, ref, "auto " + what)
            assert_parity(one, ref, "one CTA " + what)
            for G in (2, 4, 7, 16):
                if G > K:
                    continue
                q = binding.cs_score_candidates_batch_plan(Q, C, normalize, sc, T, binding.CS_PLAN_GENERIC, G)
                torch.cuda.synchronize()
                assert_parity(q, ref, f"G={G} " + what)
                assert torch.allclose(q, one, rtol=0, atol=5e-6)
        with pytest.raises(binding.CSError):  # more CTAs than rows
            binding.cs_score_candidates_batch_plan(Q, C, normalize, sc, T, binding.CS_PLAN_GENERIC, 17)
    assert binding.cs_device_status() == 0


def test_large_d(cuda_lib):
    """D large enough that q sits in shared memory, and beyond what the
    shared-memory ring holds (scalar path)."""
    for i, D in enumerate((12288, 20000)):
        for normalize in (0, 1):
            for pair in ((3.0, 1.0), TEMPERED[normalize][i], TEMPERED[normalize][i + 2]):
                wl = tempered_case(2, 9, D, normalize, pair, 31)
                assert_parity(_run(wl), oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature),
                              f"D={D} scale={wl.scale} T={wl.temperature}")


def test_automatic_plans(cuda_lib):
    def plan(B, K, D):
        Q = torch.empty(B, D, device=DEV)
        C = torch.empty(B, K, D, device=DEV)
        return binding.cs_query_plan(Q, C, 1)
    one = plan(1, 255, 512)
    assert one["plan"] == "direct" and one["cluster"] >= 8, one  # at most 32 rows per CTA
    assert plan(1, 5, 512)["plan"] == "direct" and plan(1, 5, 512)["cluster"] == 1
    assert plan(8, 255, 512)["plan"] == "direct"
    kev = plan(1, 255, 2560)  # q in shared memory: at most 16 rows per CTA
    assert kev["plan"] == "direct" and kev["cluster"] == 16, kev
    assert plan(1, 255, 1024)["plan"] == "direct"
    assert plan(1, 255, 4096)["plan"] == "cluster"  # rows too long for registers: the ring
    big = plan(4096, 255, 512)
    assert big["plan"] == "stream" and big["ctas"] == torch.cuda.get_device_properties(0).multi_processor_count
    # rows the bulk copies cannot take: up to 512 float32 elements the DIRECT
    # plan's 4-byte-unit form, at most 32 rows per CTA
    odd = plan(2, 255, 511)
    assert odd["plan"] == "direct" and odd["cluster"] >= 8, odd
    short = plan(1, 12, 511)
    assert short["plan"] == "direct" and short["cluster"] == 1, short
    assert plan(1, 255, 3)["plan"] == "direct" and plan(1, 255, 3)["cluster"] == 8  # the row limit
    # longer ones: the stream kernel's cluster plan, rows copied as aligned
    # spans (at most 16 CTAs a question, 16 KB of rows each)
    long_odd = plan(2, 255, 1001)
    assert long_odd["plan"] == "cluster" and long_odd["cluster"] == 16 and long_odd["ctas"] == 32, long_odd
    assert plan(1, 12, 1001)["cluster"] == 2     # 48 KB of rows: two CTAs of 24 KB
    many = plan(100, 255, 511)  # too many questions for clusters: the stream plan copies aligned spans
    assert many["plan"] == "stream" and many["ctas"] == 100, many
    assert plan(4096, 255, 510)["plan"] == "stream"
    assert plan(2, 9, 20000)["plan"] == "generic"  # rows too long for the ring
    # rows too long for the ring's stages: the scalar plan over a cluster
    assert plan(1, 64, 20001)["plan"] == "generic" and plan(1, 64, 20001)["cluster"] == 8


def test_throughput_workload_full_size(cuda_lib):
    """16384 questions, K=255, D=512 (8.6 GB of candidates), scored as four
    launches over consecutive slices of 4096 questions, exactly as timed by
    the benchmark. Every row is checked to sum to 1 and be finite; a
    deterministic sample of questions (every 64th, plus the first and last of
    each slice) is compared with the oracle."""
    wls = workloads.throughput(DEV)
    out = torch.empty((workloads.THROUGHPUT_B, 255), device=DEV)
    chunk = workloads.THROUGHPUT_CHUNK
    for wl in wls:
        for b0 in range(0, wl.B, chunk):
            binding.cs_score_candidates_batch(wl.Q[b0:b0 + chunk], wl.C[b0:b0 + chunk], wl.normalize,
                                              wl.scale, wl.temperature, out=out[b0:b0 + chunk])
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        sums = out.double().sum(dim=1)
        assert torch.max(torch.abs(sums - 1.0)).item() <= 1e-5
        idx = sorted(set(range(0, wl.B, 64)) | {b + o for b in range(0, wl.B, chunk) for o in (0, chunk - 1)})
        sel = torch.tensor(idx, device=DEV)
        ref = oracle_probs(wl.Q.index_select(0, sel), wl.C.index_select(0, sel), wl.normalize, wl.scale,
                           wl.temperature)
        assert_parity(out.index_select(0, sel), ref, wl.name)
    del wls
    torch.cuda.empty_cache()


def test_deterministic(cuda_lib):
    for B, K, D in ((1, 255, 512), (300, 255, 512), (2, 255, 2560)):
        wl = workloads.random_case(B, K, D, 1, 14.2857, 41, DEV)
        a = binding.cs_score_candidates_batch(wl.Q, wl.C, 1, wl.scale, 1.0)
        b = binding.cs_score_candidates_batch(wl.Q, wl.C, 1, wl.scale, 1.0)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


def test_output_guards_untouched(cuda_lib):
    """Sentinels around out survive every plan, and a rejected call leaves out
    exactly as it was."""
    sentinel = 7777.0
    for B, K, D, kind, cl in ((1, 255, 512, 0, 0), (5, 37, 512, 1, 0), (3, 64, 512, 2, 8), (2, 33, 100, 3, 0)):
        wl = workloads.random_case(B, K, D, 1, 2.0, 51, DEV)
        pad = 64
        buf = torch.full((pad + B * K + pad,), sentinel, device=DEV)
        out = buf[pad:pad + B * K].view(B, K)
        binding.cs_score_candidates_batch_plan(wl.Q, wl.C, 1, 2.0, 1.0, kind, cl, 0, out=out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == sentinel) and torch.all(buf[pad + B * K:] == sentinel)
        assert_parity(out, oracle_probs(wl.Q, wl.C, 1, 2.0, 1.0), f"guards plan {kind}")
    before = buf.clone()
    with pytest.raises(binding.CSError):
        binding.cs_score_candidates_batch(wl.Q, wl.C, 1, 0.0, 1.0, out=out)
    with pytest.raises(binding.CSError):
        binding.cs_score_candidates_batch(wl.Q, wl.C, 1, 1.0, -1.0, out=out)
    torch.cuda.synchronize()
    assert torch.equal(buf, before)


def test_rejects_on_device(cuda_lib):
    q = torch.randn(512, device=DEV)
    C = torch.randn(256, 512, device=DEV)
    with pytest.raises(binding.CSError) as e:
        binding.cs_score_candidates(q, C, 1, 1.0, 1.0)
    assert e.value.status == binding.CS_ERR_K_TOO_LARGE


def test_nondefault_stream(cuda_lib):
    wl = workloads.random_case(4, 255, 512, 1, 14.2857, 61, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p = binding.cs_score_candidates_batch(wl.Q, wl.C, 1, wl.scale, 1.0, stream=s)
    s.synchronize()
    assert_parity(p, oracle_probs(wl.Q, wl.C, 1, wl.scale, 1.0), "side stream")


def test_no_wait_gave_up(cuda_lib):
    torch.cuda.synchronize()
    assert binding.cs_device_status() == 0


@pytest.mark.parametrize("B", [1, 200], ids=["direct", "stream"])
def test_back_to_back_calls_see_the_previous_kernels_writes(cuda_lib, B):
    """The kernels may start while the previous kernel in the stream is still
    running (programmatic dependent launch) and wait for it before touching
    memory: a call whose query is the previous call's output, and a call
    right after an in-stream overwrite of C, must see the new values."""
    K, D = 4, 4
    g = torch.Generator(device="cpu")
    g.manual_seed(77 + B)
    Q1 = torch.randn(B, D, generator=g).to(DEV)
    C1 = torch.randn(B, K, D, generator=g).to(DEV)
    C2 = torch.randn(B, K, D, generator=g).to(DEV)
    p1 = torch.empty(B, K, device=DEV)
    p2 = torch.empty(B, K, device=DEV)
    for _ in range(3):  # repeated, so later rounds overlap earlier launches
        binding.cs_score_candidates_batch(Q1, C1, 1, 3.0, 1.0, out=p1)
        binding.cs_score_candidates_batch(p1, C2, 0, 2.0, 1.0, out=p2)  # q = the previous output
    torch.cuda.synchronize()
    ref1 = oracle_probs(Q1.cpu(), C1.cpu(), 1, 3.0, 1.0)
    assert_parity(p1, ref1, "first call")
    ref2 = oracle_probs(p1.cpu(), C2.cpu(), 0, 2.0, 1.0)
    assert_parity(p2, ref2, "second call reads the first call's output")
    Cnew = torch.randn(B, K, D, generator=g).to(DEV)
    C1.copy_(Cnew)  # an in-stream kernel writes C just before the call
    binding.cs_score_candidates_batch(Q1, C1, 1, 3.0, 1.0, out=p1)
    torch.cuda.synchronize()
    assert_parity(p1, oracle_probs(Q1.cpu(), Cnew.cpu(), 1, 3.0, 1.0), "call after an in-stream overwrite")
    plan = binding.cs_query_plan(Q1, C1, 1)["plan"]
    assert plan == ("direct" if B == 1 else "stream"), plan


def test_calls_without_a_stream_use_torchs_current_stream(cuda_lib):
    """stream=None means torch's current stream on the tensors' device, also
    inside `with torch.cuda.stream(...)`."""
    dev = torch.device(DEV)
    side = torch.cuda.Stream(dev)
    assert binding._stream_handle(None, dev) == torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.stream(side):
        assert binding._stream_handle(None, dev) == side.cuda_stream
        wl = workloads.random_case(2, 9, 64, 1, 3.0, 88, DEV)
        p = binding.cs_score_candidates_batch(wl.Q, wl.C, 1, 3.0, 1.0)
    side.synchronize()
    assert_parity(p, oracle_probs(wl.Q, wl.C, 1, 3.0, 1.0), "call on a side stream")


def test_c_marshalling_matches_ctypes_marshalling(cuda_lib):
    """The readout calls with `out` given go through the binding's C
    marshalling module; the same calls without `out` go through ctypes.
    Both reach the same library entry point, so the results are
    bit-identical, errors come back as the same status, and what the C
    module hands back (a wrong dtype, a non-contiguous tensor) raises the
    ctypes path's error."""
    fp = binding._fastpath()
    assert fp, "the C marshalling module was not built or set up on this machine"
    for B, K, D, normalize in ((1, 5, 512, 1), (1, 255, 2560, 0), (8, 255, 512, 1), (300, 33, 510, 0)):
        wl = workloads.random_case(B, K, D, normalize, 3.0, 81 + B, DEV)
        out = torch.empty(B, K, device=DEV)
        if B == 1:
            ref = binding.cs_score_candidates(wl.Q[0], wl.C[0], normalize, 3.0, 0.7)
            got = binding.cs_score_candidates(wl.Q[0], wl.C[0], normalize, 3.0, 0.7, out=out[0])
            Cb = wl.C[0].to(torch.bfloat16)
            refb = binding.cs_score_candidates_bf16(wl.Q[0], Cb, normalize, 3.0, 0.7)
            gotb = binding.cs_score_candidates_bf16(wl.Q[0], Cb, normalize, 3.0, 0.7,
                                                    out=torch.empty(K, device=DEV))
        else:
            ref = binding.cs_score_candidates_batch(wl.Q, wl.C, normalize, 3.0, 0.7)
            got = binding.cs_score_candidates_batch(wl.Q, wl.C, normalize, 3.0, 0.7, out=out)
            Cb = wl.C.to(torch.bfloat16)
            refb = binding.cs_score_candidates_batch_bf16(wl.Q, Cb, normalize, 3.0, 0.7)
            gotb = binding.cs_score_candidates_batch_bf16(wl.Q, Cb, normalize, 3.0, 0.7,
                                                          out=torch.empty(B, K, device=DEV))
        torch.cuda.synchronize()
        assert torch.equal(ref, got) and torch.equal(refb, gotb), (B, K, D)
    # an error status from the library, through the C module
    q, C = torch.randn(512, device=DEV), torch.randn(256, 512, device=DEV)
    with pytest.raises(binding.CSError) as e:
        binding.cs_score_candidates(q, C, 1, 1.0, 1.0, out=torch.empty(256, device=DEV))
    assert e.value.status == binding.CS_ERR_K_TOO_LARGE
    # handed back to ctypes, which raises its own errors
    C5 = torch.randn(5, 512, device=DEV)
    with pytest.raises(TypeError):
        binding.cs_score_candidates_bf16(q, C5, 1, 1.0, 1.0, out=torch.empty(5, device=DEV))
    with pytest.raises(ValueError, match="contiguous"):
        binding.cs_score_candidates(q, torch.randn(512, 5, device=DEV).t(), 1, 1.0, 1.0,
                                    out=torch.empty(5, device=DEV))
    assert fp.score(q, C5, torch.empty(5, device=DEV), 1, 1.0, 1.0, None, True) is None
