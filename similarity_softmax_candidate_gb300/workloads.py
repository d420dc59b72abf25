"""Seeded synthetic inputs shaped like the candidate-scoring workloads.

This module only draws random numbers. It holds none of the scoring
arithmetic, so both the CUDA path and the fp64 oracle can be fed from it.

The shapes and distributions follow the workloads of PR #69 "cuda: add a
fused candidate-scoring kernel for CLM and Kev" (the shape table of "What it
is worth" and the fixed cases of "Verified on hardware"): CLM scores by cosine
with scale exp(logit_scale), Kev by a dot with scale 1/sqrt(256). The page
names no dataset; its inputs are model feature vectors of unstated
distribution, so Gaussian features stand in for them:

  clm_k5       cosine, 1 question,  K=5,   D=512,  q, C ~ N(0,1)
  clm_k64      cosine, 1 question,  K=64,  D=512,  q, C ~ N(0,1)
  clm_k64_*    the degenerate calls: a zero candidate, all candidates equal,
               one duplicated pair, and a single candidate (K=1)
  clm_batch8   cosine, 8 questions, K=255, D=512, C[i,k] = q_i + 0.5 N(0,1)
  kev_k255     dot, 1 question, K=255, D=2560, q, C ~ 0.5 N(0,1)
  kev_overflow the same with C scaled by 1e3 (raw logits far beyond exp range)
  throughput   16384 questions, K=255, D=512, q, C ~ N(0,1), scored as four
               consecutive slices of 4096 questions, cosine and dot
  ragged       B questions with K_b uniform in [kmin, kmax] (the serving mix
               of short and long candidate lists), rows back to back

CLM's logit_scale is ln(1/0.07), so its scale exp(logit_scale) is 1/0.07;
Kev's is 1/sqrt(256) = 1/16. The temperature is 1. Scales are rounded to
float32 here, once, so that the oracle and the kernel see the same argument.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

CLM_SCALE = float(np.float32(math.exp(math.log(1.0 / 0.07))))
KEV_SCALE = float(np.float32(1.0 / math.sqrt(256.0)))
TEMPERATURE = 1.0

THROUGHPUT_B = 16384
THROUGHPUT_CHUNK = 4096
MAX_K = 255


@dataclasses.dataclass
class Workload:
    """One call's worth of inputs: Q[B,D], C[B,K,D] (float32, contiguous)."""
    name: str
    Q: torch.Tensor
    C: torch.Tensor
    normalize: int
    scale: float
    temperature: float = TEMPERATURE

    @property
    def B(self) -> int:
        return int(self.C.shape[0])

    @property
    def K(self) -> int:
        return int(self.C.shape[1])

    @property
    def D(self) -> int:
        return int(self.C.shape[2])

    def algorithmic_bytes(self) -> int:
        """Bytes the readout must move: C and q read once, p written once."""
        return 4 * (self.B * self.K * self.D + self.B * self.D + self.B * self.K)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """float32 N(0, std^2) tensor drawn from a generator seeded with seed."""
    t = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def random_case(B, K, D, normalize, scale, seed, device="cpu", std=1.0,
                temperature=TEMPERATURE, name=None) -> Workload:
    """Independent N(0, std^2) query and candidates."""
    Q = normal((B, D), seed, device, std)
    C = normal((B, K, D), seed + 7919, device, std)
    return Workload(name or f"random_b{B}_k{K}_d{D}_{'cos' if normalize else 'dot'}",
                    Q, C, int(normalize), float(scale), float(temperature))


def clm_k5(device="cpu", seed=0):
    return [random_case(1, 5, 512, 1, CLM_SCALE, seed, device, name="clm_k5")]


def clm_k64(device="cpu", seed=1):
    base = random_case(1, 64, 512, 1, CLM_SCALE, seed, device, name="clm_k64")
    zero = random_case(1, 64, 512, 1, CLM_SCALE, seed + 100, device, name="clm_k64_zero_row")
    zero.C[0, 17].zero_()
    same = random_case(1, 64, 512, 1, CLM_SCALE, seed + 200, device, name="clm_k64_all_equal")
    same.C[0, :] = same.C[0, 3].clone()
    pair = random_case(1, 64, 512, 1, CLM_SCALE, seed + 300, device, name="clm_k64_dup_pair")
    pair.C[0, 40] = pair.C[0, 5].clone()
    single = random_case(1, 1, 512, 1, CLM_SCALE, seed + 400, device, name="clm_k1")
    return [base, zero, same, pair, single]


def clm_batch8(device="cpu", seed=2):
    Q = normal((8, 512), seed, device)
    noise = normal((8, MAX_K, 512), seed + 7919, device, 0.5)
    C = (Q[:, None, :] + noise).contiguous()
    return [Workload("clm_batch8", Q, C, 1, CLM_SCALE)]


def kev_k255(device="cpu", seed=3):
    base = random_case(1, MAX_K, 2560, 0, KEV_SCALE, seed, device, std=0.5, name="kev_k255")
    over = Workload("kev_overflow", base.Q.clone(), (base.C * 1e3).contiguous(), 0, KEV_SCALE)
    return [base, over]


def throughput(device="cuda", seed=4, B=THROUGHPUT_B, K=MAX_K, D=512):
    """The bandwidth workload: one [B,K,D] candidate buffer (8.6 GB at the
    full size), scored cosine and dot. Draw it on the GPU: on the host it
    would take minutes."""
    Q = normal((B, D), seed, device)
    C = torch.empty((B, K, D), device=device, dtype=torch.float32)
    # Fill in slabs so the generator's temporary stays small.
    g = _gen(seed + 7919, device)
    step = max(1, (1 << 28) // (K * D))
    for b0 in range(0, B, step):
        b1 = min(B, b0 + step)
        C[b0:b1].normal_(generator=g)
    return [Workload("throughput_cos", Q, C, 1, CLM_SCALE),
            Workload("throughput_dot", Q, C, 0, KEV_SCALE)]


@dataclasses.dataclass
class RaggedWorkload:
    """A ragged batch: question b owns rows offsets[b]..offsets[b+1]-1 of C."""
    name: str
    Q: torch.Tensor        # [B, D] float32
    C: torch.Tensor        # [total_rows, D] float32
    offsets: torch.Tensor  # [B + 1] int64
    normalize: int
    scale: float
    temperature: float = TEMPERATURE

    @property
    def B(self) -> int:
        return int(self.Q.shape[0])

    @property
    def total_rows(self) -> int:
        return int(self.C.shape[0])


def ragged(B, D, normalize, scale, seed, device="cpu", kmin=1, kmax=MAX_K, name=None) -> RaggedWorkload:
    """B questions with K_b drawn uniformly from [kmin, kmax] (the serving
    mix of short and long candidate lists), q and C ~ N(0,1)."""
    g = _gen(seed, "cpu")
    k = torch.randint(kmin, kmax + 1, (B,), generator=g, dtype=torch.int64)
    offsets = torch.zeros(B + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(k, 0)
    total = int(offsets[-1])
    Q = normal((B, D), seed + 1, device)
    C = torch.empty((total, D), device=device, dtype=torch.float32)
    gc = _gen(seed + 2, device)
    step = max(1, (1 << 28) // D)
    for r0 in range(0, total, step):
        C[r0:r0 + step].normal_(generator=gc)
    return RaggedWorkload(name or f"ragged_b{B}_d{D}_{'cos' if normalize else 'dot'}", Q, C, offsets.to(device),
                          int(normalize), float(scale))


CONFIGS = {
    "clm_k5": clm_k5,
    "clm_k64": clm_k64,
    "clm_batch8": clm_batch8,
    "kev_k255": kev_k255,
    "throughput": throughput,
}
