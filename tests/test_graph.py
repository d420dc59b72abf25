"""CUDA Graph capture of the C ABI (PR #69 "cuda: add a fused candidate-scoring
kernel for CLM and Kev", "Through a CUDA Graph" and "Verified on hardware"):
a call queues on the caller's stream and never synchronizes, so capturing it
yields exactly one graph node, and replaying the graph gives bit-identical
output to a direct call.

Capture uses the CUDA runtime directly through ctypes, in the strict global
capture mode, in which any forbidden call (allocation, synchronization)
inside the library would invalidate the capture.
"""
from __future__ import annotations

import ctypes
import glob
import os

import pytest
import torch

from similarity_softmax_candidate_gb300 import binding, workloads
from tests._util import assert_parity, oracle_probs

pytestmark = pytest.mark.gpu

CAPTURE_MODE_GLOBAL = 0
NODE_TYPE_KERNEL = 0


def _cudart():
    names = ["libcudart.so.13"]
    torch_lib = os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "cu13", "lib")
    names += glob.glob(os.path.join(torch_lib, "libcudart.so*"))
    names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
    for n in names:
        try:
            rt = ctypes.CDLL(n)
        except OSError:
            continue
        V, P = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
        rt.cudaStreamBeginCapture.argtypes = [V, ctypes.c_int]
        rt.cudaStreamEndCapture.argtypes = [V, P]
        rt.cudaGraphGetNodes.argtypes = [V, P, ctypes.POINTER(ctypes.c_size_t)]
        rt.cudaGraphNodeGetType.argtypes = [V, ctypes.POINTER(ctypes.c_int)]
        rt.cudaGraphInstantiate.argtypes = [P, V, ctypes.c_ulonglong]
        rt.cudaGraphLaunch.argtypes = [V, V]
        rt.cudaGraphExecDestroy.argtypes = [V]
        rt.cudaGraphDestroy.argtypes = [V]
        return rt
    pytest.fail("libcudart not found")


def _capture(rt, stream, fn):
    assert rt.cudaStreamBeginCapture(stream.cuda_stream, CAPTURE_MODE_GLOBAL) == 0
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        end = rt.cudaStreamEndCapture(stream.cuda_stream, ctypes.byref(graph))
    assert end == 0, f"cudaStreamEndCapture failed ({end}): the call did something capture forbids"
    return graph


# (B, K, D, normalize, scale, temperature, off): the page's shapes, a large
# batch, odd D, two calls with a temperature other than 1 and a negative
# scale, and Q and C `off` elements past a 16-byte boundary (the DIRECT and
# stream plans' 4-byte-unit forms, and the scalar plan for long rows).
CASES = [(1, 5, 512, 1, 14.2857, 1.0, 0), (1, 255, 512, 1, 14.2857, 1.0, 0), (8, 255, 512, 1, 14.2857, 1.0, 0),
         (1, 255, 2560, 0, 0.0625, 1.0, 0), (700, 255, 512, 0, 0.0625, 1.0, 0), (3, 33, 513, 1, 14.2857, 1.0, 0),
         (4, 255, 512, 1, -14.2857, 0.7, 0), (300, 64, 256, 0, -0.0625, 3.0, 0),
         (1, 255, 512, 1, 14.2857, 1.0, 1), (700, 255, 510, 1, 14.2857, 0.7, 1), (2, 64, 2560, 0, 0.0625, 1.0, 3)]


def _off(t, off):
    if not off:
        return t
    flat = torch.empty(t.numel() + off + 8, device=t.device, dtype=t.dtype)
    v = flat[off:off + t.numel()].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("B,K,D,normalize,scale,temperature,off", CASES)
def test_one_node_and_bitwise_replay(cuda_lib, B, K, D, normalize, scale, temperature, off):
    rt = _cudart()
    wl = workloads.random_case(B, K, D, normalize, scale, 71, "cuda:0", temperature=temperature)
    wl.Q, wl.C = _off(wl.Q, off), _off(wl.C, off)
    s = torch.cuda.Stream()
    direct = torch.empty(B, K, device="cuda:0")
    replay = torch.full((B, K), -1.0, device="cuda:0")
    torch.cuda.synchronize()
    # an ordinary call first: one-time per-device set-up happens here
    binding.cs_score_candidates_batch(wl.Q, wl.C, normalize, wl.scale, wl.temperature, out=direct, stream=s)
    torch.cuda.synchronize()
    ref = oracle_probs(wl.Q, wl.C, normalize, wl.scale, wl.temperature)

    def call():
        if B == 1:
            binding.cs_score_candidates(wl.Q[0], wl.C[0], normalize, wl.scale, wl.temperature, out=replay[0],
                                        stream=s)
        else:
            binding.cs_score_candidates_batch(wl.Q, wl.C, normalize, wl.scale, wl.temperature, out=replay, stream=s)

    graph = _capture(rt, s, call)
    try:
        n = ctypes.c_size_t(0)
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
        assert n.value == 1, f"captured {n.value} nodes, expected exactly one"
        node = (ctypes.c_void_p * 1)()
        assert rt.cudaGraphGetNodes(graph, node, ctypes.byref(n)) == 0
        t = ctypes.c_int(-1)
        assert rt.cudaGraphNodeGetType(node[0], ctypes.byref(t)) == 0 and t.value == NODE_TYPE_KERNEL
        torch.cuda.synchronize()
        assert torch.all(replay == -1.0), "capture must not execute the call"
        exe = ctypes.c_void_p()
        assert rt.cudaGraphInstantiate(ctypes.byref(exe), graph, 0) == 0
        try:
            for _ in range(3):
                assert rt.cudaGraphLaunch(exe, s.cuda_stream) == 0
                torch.cuda.synchronize()
                assert torch.equal(replay, direct), "graph replay differs from the direct call"
                assert_parity(replay, ref, f"replay B={B} K={K} D={D} scale={scale} T={temperature}")
                replay.fill_(-1.0)
                torch.cuda.synchronize()
        finally:
            rt.cudaGraphExecDestroy(exe)
    finally:
        rt.cudaGraphDestroy(graph)
