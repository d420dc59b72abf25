"""fp64 CPU oracle for fused candidate scoring -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and
shares no code with it; the only thing both sides share is the seeded input
generator in ``similarity_softmax_candidate_gb300.workloads``, which holds
none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain loops, double accumulation in
index order). This module compiles it with gcc, loads it with ctypes and
wraps it for numpy arrays.

Method source: PR #69 "cuda: add a fused candidate-scoring kernel for CLM
and Kev" (the opening table of the two models' similarities, and the section
"What is fused, precisely"). Parity pins: tests/test_oracle_pins.py and the
hand cases under tests/golden/.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# A test may point this wrapper at another build of an altered copy of the
# source (tests/test_oracle_mutants.py plants mistakes that way, to show the
# pins catch them); everything else uses the files next to this module.
_SRC = os.environ.get("CS_ORACLE_SRC") or os.path.join(_HERE, "oracle.c")
_LIB = os.environ.get("CS_ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")

#: The norm clamp of the cosine similarity. The page gives no value; each
#: norm is clamped on its own at this floor (plainest cosine convention).
EPS = 1e-8

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no fast-math,
    no FMA contraction so the rounding is the same on x86 and Arm)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            f, d, l, i, p = (ctypes.c_void_p, ctypes.c_double, ctypes.c_long,
                             ctypes.c_int, ctypes.c_void_p)
            lib.oracle_logits.argtypes = [f, f, l, l, l, i, d, d, d, p]
            lib.oracle_logits.restype = i
            lib.oracle_softmax.argtypes = [p, l, l, p]
            lib.oracle_softmax.restype = i
            lib.oracle_score_batch.argtypes = [f, f, l, l, l, i, d, d, d, p]
            lib.oracle_score_batch.restype = i
            lib.oracle_project.argtypes = [f, f, l, l, l, p]
            lib.oracle_project.restype = i
            _lib = lib
    return _lib


def _shapes(Q, C):
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    C = np.ascontiguousarray(C, dtype=np.float32)
    if Q.ndim == 1:
        Q = Q[None, :]
    if C.ndim == 2:
        C = C[None, :, :]
    B, D = Q.shape
    if C.shape[0] != B or C.shape[2] != D:
        raise ValueError(f"shape mismatch: Q {Q.shape}, C {C.shape}")
    return Q, C, B, C.shape[1], D


def logits(Q, C, normalize, scale, temperature, eps=EPS):
    """Similarity logits z[B,K] (float64) for Q[B,D] (or q[D]) and
    C[B,K,D] (or C[K,D])."""
    Q, C, B, K, D = _shapes(Q, C)
    z = np.empty((B, K), dtype=np.float64)
    rc = _load().oracle_logits(Q.ctypes.data, C.ctypes.data, B, K, D, int(normalize),
                               float(scale), float(temperature), float(eps), z.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_logits: bad size")
    return z


def softmax(z):
    """Row-wise softmax of z[B,K] (or z[K]) in float64."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    one = z.ndim == 1
    z2 = z[None, :] if one else z
    p = np.empty_like(z2)
    rc = _load().oracle_softmax(z2.ctypes.data, z2.shape[0], z2.shape[1], p.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_softmax: bad size")
    return p[0] if one else p


def score_batch(Q, C, normalize, scale, temperature, eps=EPS):
    """Softmax probabilities p[B,K] (float64) of the whole readout."""
    Q, C, B, K, D = _shapes(Q, C)
    p = np.empty((B, K), dtype=np.float64)
    rc = _load().oracle_score_batch(Q.ctypes.data, C.ctypes.data, B, K, D, int(normalize),
                                    float(scale), float(temperature), float(eps), p.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_score_batch: bad size")
    return p


def project(H, W):
    """P = H W^T in float64 for H[R, Din] and W[D, Din] (float32 values, e.g.
    bfloat16 weights and features widened exactly)."""
    H = np.ascontiguousarray(H, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.float32)
    if H.ndim != 2 or W.ndim != 2 or H.shape[1] != W.shape[1]:
        raise ValueError(f"shape mismatch: H {H.shape}, W {W.shape}")
    P = np.empty((H.shape[0], W.shape[0]), dtype=np.float64)
    rc = _load().oracle_project(H.ctypes.data, W.ctypes.data, H.shape[0], H.shape[1], W.shape[0], P.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_project: bad size")
    return P


def project_score_batch(Hq, Wq, Hc, Wc, normalize, scale, temperature, eps=EPS):
    """The readout with caller-side projections: q_b = Wq hq_b, c_bk = Wc
    hc_bk, then score_batch on the projected vectors (each projected value is
    rounded once to float32, the precision the scorer takes). Hq [B, Din],
    Hc [B, K, Din]; returns p [B, K] float64."""
    Hq = np.asarray(Hq, dtype=np.float32)
    Hc = np.asarray(Hc, dtype=np.float32)
    B, K, Din = Hc.shape
    q = project(Hq, Wq).astype(np.float32)
    c = project(Hc.reshape(B * K, Din), Wc).astype(np.float32).reshape(B, K, -1)
    return score_batch(q, c, normalize, scale, temperature, eps)
