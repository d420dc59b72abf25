"""The library's float32 range on the GPU.

PR #69 "cuda: add a fused candidate-scoring kernel for CLM and Kev",
"Verified on hardware", asks for an error rather than a scored answer where
the arguments are bad. Here that rule meets float32: the fp64 oracle scores
any finite input, the kernels accumulate in float32. So:

  * inputs inside the documented range get the oracle's distribution, also
    where a naive float32 logit would overflow: a logit factor near the
    2^126 limit, a query so short that scale / |q| overflows, dots whose
    differences exceed FLT_MAX, a factor that underflows to 0;
  * a question whose dots or squared norms leave float32's range, or that
    holds a NaN or an infinity, is skipped: its rows of out keep what they
    held, the other questions are scored, and CS_DEVERR_RANGE is set;
  * a factor scale / temperature beyond FLT_MAX is refused on the host
    (2^126 and above: tests/test_abi_host.py) -- here, that no launch
    happened.

Every plan and entry point is run, since each forms its logits in its own
code.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import assert_parity, oracle_probs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SENTINEL = 4242.0

# (name, how a batch is scored); every form takes Q [B,D], C [B,K,D] float32
# on the device and writes out [B,K].
PLANS = ["auto", "direct", "cluster4", "stream", "generic", "generic4", "unfused", "bf16", "ragged",
         "auto_off", "stream_off", "bf16_off"]


def _one_off(t):
    """A copy of t one element past a 16-byte boundary (rows the bulk copies
    cannot take whole: the 4-byte-unit forms)."""
    flat = torch.empty(t.numel() + 8, device=DEV, dtype=t.dtype)
    v = flat[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _score(plan, Q, C, normalize, scale, T, out):
    b = binding
    if plan.endswith("_off"):  # the same plan on copies of Q and C one element off
        if plan == "bf16_off":
            Q, Cb = _one_off(Q), _one_off(C.to(torch.bfloat16))
            return b.cs_score_candidates_batch_bf16(Q, Cb, normalize, scale, T, out=out)
        return _score(plan[:-4], _one_off(Q), _one_off(C), normalize, scale, T, out)
    if plan == "auto":
        return b.cs_score_candidates_batch(Q, C, normalize, scale, T, out=out)
    if plan == "direct":
        return b.cs_score_candidates_batch_plan(Q, C, normalize, scale, T, b.CS_PLAN_DIRECT, 0, 0, out=out)
    if plan == "cluster4":
        return b.cs_score_candidates_batch_plan(Q, C, normalize, scale, T, b.CS_PLAN_CLUSTER, 4, 0, out=out)
    if plan == "stream":
        return b.cs_score_candidates_batch_plan(Q, C, normalize, scale, T, b.CS_PLAN_STREAM, 0, 0, out=out)
    if plan == "generic":
        return b.cs_score_candidates_batch_plan(Q, C, normalize, scale, T, b.CS_PLAN_GENERIC, 1, 0, out=out)
    if plan == "generic4":
        return b.cs_score_candidates_batch_plan(Q, C, normalize, scale, T, b.CS_PLAN_GENERIC, 4, 0, out=out)
    if plan == "unfused":
        return b.cs_score_candidates_batch_unfused(Q, C, normalize, scale, T, out=out)
    if plan == "bf16":
        return b.cs_score_candidates_batch_bf16(Q, C.to(torch.bfloat16), normalize, scale, T, out=out)
    if plan == "ragged":
        B, K, D = C.shape
        off = torch.arange(B + 1, device=DEV, dtype=torch.int64) * K
        b.cs_score_candidates_ragged(Q, C.view(B * K, D), off, normalize, scale, T, out=out.view(B * K))
        return out
    raise ValueError(plan)


def _ref(plan, Q, C, normalize, scale, T):
    if plan in ("bf16", "bf16_off"):
        C = C.to(torch.bfloat16).float()
    return oracle_probs(Q.cpu().double(), C.cpu().double(), normalize, scale, T)


def _run(plan, Q, C, normalize, scale, T):
    out = torch.full(C.shape[:2], SENTINEL, device=DEV)
    binding.cs_device_status(clear=True)
    _score(plan, Q, C, normalize, scale, T, out)
    torch.cuda.synchronize()
    return out, binding.cs_device_status(clear=True)


@pytest.mark.parametrize("plan", PLANS)
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_rows_beyond_float32_are_skipped_and_flagged(cuda_lib, plan, normalize):
    """Question 1 of 3 holds rows whose squared norms (cosine: candidates
    times 1e20) or dots (dot: candidates times 1e36, query times 1e4)
    overflow float32; question 2 holds a NaN candidate element. Both are
    skipped, their rows keep the sentinel; question 0 is scored."""
    B, K, D = 3, 40, 512
    wl = workloads.random_case(B, K, D, normalize, 14.2857 if normalize else 0.0625, 61, DEV)
    Q, C = wl.Q.clone(), wl.C.clone()
    if normalize:
        C[1] *= 1e20
    else:
        C[1] *= 1e36
        Q[1] *= 1e4
    C[2, 7, 100] = float("nan")
    out, status = _run(plan, Q, C, normalize, wl.scale, 1.0)
    assert status == binding.CS_DEVERR_RANGE, f"{plan}: status {status}"
    assert torch.all(out[1:] == SENTINEL), f"{plan}: a skipped question was written"
    assert_parity(out[:1], _ref(plan, Q[:1], C[:1], normalize, wl.scale, 1.0), f"{plan} question 0")


@pytest.mark.parametrize("plan", ["auto", "direct", "cluster4", "stream", "generic", "generic4"])
def test_infinite_query_is_skipped(cuda_lib, plan):
    B, K, D = 2, 40, 512
    for normalize in (1, 0):
        wl = workloads.random_case(B, K, D, normalize, 2.0, 62, DEV)
        Q = wl.Q.clone()
        Q[0, 3] = float("inf")
        out, status = _run(plan, Q, wl.C, normalize, 2.0, 1.0)
        assert status == binding.CS_DEVERR_RANGE
        assert torch.all(out[0] == SENTINEL)
        assert_parity(out[1:], _ref(plan, Q[1:], wl.C[1:], normalize, 2.0, 1.0), f"{plan} question 1")


@pytest.mark.parametrize("plan", PLANS)
def test_rescaled_cosine_inputs_match_the_oracle(cuda_lib, plan):
    """The cosine ignores positive rescaling (pinned on the oracle by
    tests/test_oracle_pins.py): candidates times 1e15 and a query times
    1e-20 (its norm then below the 1e-8 clamp, as in the oracle), inside
    the range, give the oracle's distribution; candidates times 1e-15 fall
    under the clamp on both sides alike."""
    B, K, D = 3, 40, 512
    wl = workloads.random_case(B, K, D, 1, 14.2857, 63, DEV)
    for fq, fc in ((1.0, 1e15), (1e-20, 1.0), (1.0, 1e-15), (1e-20, 1e15)):
        Q, C = wl.Q * fq, wl.C * fc
        out, status = _run(plan, Q, C, 1, wl.scale, 1.0)
        assert status == 0
        assert_parity(out, _ref(plan, Q, C, 1, wl.scale, 1.0), f"{plan} q x {fq}, C x {fc}")


def _one_hot_case(normalize, B=2, K=40, D=512, qscale=1.0):
    """Rows 3 and 11 of each question are copies of 2q (the largest cosine
    and, for the dot, by far the largest dot); row 5 is -2q (the smallest)."""
    wl = workloads.random_case(B, K, D, normalize, 1.0, 64, DEV)
    Q = wl.Q * qscale
    C = wl.C.clone()
    C[:, 3] = 2 * Q
    C[:, 11] = 2 * Q
    C[:, 5] = -2 * Q
    return Q, C


@pytest.mark.parametrize("plan", PLANS)
@pytest.mark.parametrize("normalize", [1, 0], ids=["cos", "dot"])
def test_factor_near_its_limit(cuda_lib, plan, normalize):
    """scale / temperature = 8e37 (and -8e37), just under the 2^126 limit:
    accepted, and the softmax of such logits puts all the weight on the
    largest (smallest) similarity, shared between the two equal rows. For
    the cosine the query is short (times 1e-3), so that scale / (T |q|) --
    the factor a plain float32 kernel would form -- overflows."""
    Q, C = _one_hot_case(normalize, qscale=1e-3 if normalize else 1.0)
    for scale in (8e37, -8e37):
        out, status = _run(plan, Q, C, normalize, scale, 1.0)
        assert status == 0
        ref = _ref(plan, Q, C, normalize, scale, 1.0)
        assert_parity(out, ref, f"{plan} scale {scale}")
        hot = [3, 11] if scale > 0 else [5]
        assert np.allclose(ref[:, hot].sum(axis=1), 1.0)


@pytest.mark.parametrize("plan", PLANS)
def test_dot_differences_beyond_float32_max(cuda_lib, plan):
    """Dots of +3e38 and -3e38 (their difference is beyond FLT_MAX) at scale
    1e-38: logits 3, -3 and 0, which a kernel subtracting the raw dots
    would turn into probabilities 1 and 0."""
    B, K, D = 2, 6, 512
    Q = torch.zeros(B, D, device=DEV)
    Q[:, 0] = 1.0
    C = torch.zeros(B, K, D, device=DEV)
    C[:, 0, 0] = 3e38
    C[:, 1, 0] = -3e38
    C[:, 2, 1] = 5.0  # dot 0
    scale = float(np.float32(1e-38))  # the float32 argument the kernel sees
    out, status = _run(plan, Q, C, 0, scale, 1.0)
    assert status == 0
    ref = _ref(plan, Q, C, 0, scale, 1.0)
    assert ref[0, 1] > 1e-3  # the oracle's answer is not a one-hot
    assert_parity(out, ref, plan)
    # at scale 1e-20 the same dots make logits of +-3e18: all the weight on
    # row 0, although the difference of the two dots is beyond FLT_MAX
    out, status = _run(plan, Q, C, 0, 1e-20, 1.0)
    assert status == 0
    ref = _ref(plan, Q, C, 0, 1e-20, 1.0)
    assert np.allclose(ref[:, 0], 1.0)
    assert_parity(out, ref, plan + " scale 1e-20")


@pytest.mark.parametrize("plan", PLANS)
def test_factor_below_float32_is_uniform(cuda_lib, plan):
    """scale 1e-30 at temperature 1e30: a factor of 1e-60 rounds to 0 in
    float32, and the exact softmax is uniform to within 1e-58."""
    for normalize in (1, 0):
        wl = workloads.random_case(2, 40, 512, normalize, 1.0, 65, DEV)
        out, status = _run(plan, wl.Q, wl.C, normalize, 1e-30, 1e30)
        assert status == 0
        assert_parity(out, _ref(plan, wl.Q, wl.C, normalize, 1e-30, 1e30), f"{plan} normalize={normalize}")
        assert torch.max(torch.abs(out - 1.0 / 40)).item() <= 1e-7


def test_refused_factor_launches_nothing(cuda_lib):
    wl = workloads.random_case(2, 40, 512, 1, 1.0, 66, DEV)
    out = torch.full((2, 40), SENTINEL, device=DEV)
    with pytest.raises(binding.CSError) as e:
        binding.cs_score_candidates_batch(wl.Q, wl.C, 1, 14.2857, 1e-37, out=out)
    assert e.value.status == binding.CS_ERR_RANGE
    torch.cuda.synchronize()
    assert torch.all(out == SENTINEL)
    assert binding.cs_device_status() == 0


def _bf16(shape, seed, std=1.0):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def test_projected_rows_beyond_float32_are_skipped(cuda_lib):
    """The projected readout: question 1's candidate features times 1e20
    project to rows whose squared norms overflow; it is skipped and
    flagged, question 0 is scored."""
    import oracle
    B, K, Din, D = 2, 40, 64, 256
    Hq, Hc = _bf16((B, Din), 71), _bf16((B, K, Din), 72)
    Hc[1] = (Hc[1].float() * 1e20).to(torch.bfloat16)
    Wq, Wc = _bf16((D, Din), 73, Din ** -0.5), _bf16((D, Din), 74, Din ** -0.5)
    out = torch.full((B, K), SENTINEL, device=DEV)
    binding.cs_device_status(clear=True)
    binding.cs_project_score_batch(Hq.to(DEV), Wq.to(DEV), Hc.to(DEV), Wc.to(DEV), 1, 14.2857, 1.0, out=out)
    torch.cuda.synchronize()
    assert binding.cs_device_status(clear=True) == binding.CS_DEVERR_RANGE
    assert torch.all(out[1] == SENTINEL)
    ref = oracle.project_score_batch(Hq[:1].float().numpy(), Wq.float().numpy(), Hc[:1].float().numpy(),
                                     Wc.float().numpy(), 1, 14.2857, 1.0)
    assert_parity(out[:1], ref, "projected question 0")
