"""The binding's C marshalling module (_fastpath, csrc/fastpath.c).

It must only ever take the plain case -- contiguous CUDA tensors of the
entry point's dtypes and shapes, on the current device -- and hand
everything else back (None), so that the ctypes path raises the precise
error. On a machine without a GPU no tensor is a CUDA tensor, so every
call here must come back unhandled without touching the library.
"""
from __future__ import annotations

import os

import pytest

from similarity_softmax_candidate_gb300 import _build, binding


def _module():
    if _build.build_fastpath() is None:
        pytest.skip("no C compiler or Python headers: the binding uses ctypes alone")
    from similarity_softmax_candidate_gb300 import _fastpath
    return _fastpath


def test_builds_next_to_the_package():
    _module()
    assert os.path.exists(_build.FASTPATH_PATH)


def test_host_tensors_are_handed_back(host_lib):
    torch = pytest.importorskip("torch")
    fp = binding._fastpath()
    assert fp, "the binding did not set the C marshalling up"
    q, C, out = torch.zeros(8), torch.zeros(3, 8), torch.zeros(3)
    assert fp.score(q, C, out, 1, 1.0, 1.0, None, False) is None
    Q, Cb, ob = torch.zeros(2, 8), torch.zeros(2, 3, 8), torch.zeros(2, 3)
    assert fp.score_batch(Q, Cb, ob, 1, 1.0, 1.0, None, False) is None
    assert fp.score_batch(Q, Cb.to(torch.bfloat16), ob, 1, 1.0, 1.0, None, True) is None
    # wrong arity and non-tensors are handed back too
    assert fp.score(q, C, out) is None
    assert fp.score(1, 2, 3, 1, 1.0, 1.0, None, False) is None
    assert fp.score_batch("Q", None, [], 1, 1.0, 1.0, None, False) is None
    # and the binding then raises the ctypes path's error
    with pytest.raises(ValueError, match="CUDA device"):
        binding.cs_score_candidates(q, C, 1, 1.0, 1.0, out=out)
    with pytest.raises(ValueError, match="CUDA device"):
        binding.cs_score_candidates_batch(Q, Cb, 1, 1.0, 1.0, out=ob)


def test_setup_refuses_null_entry_points():
    fp = _module()
    import torch
    with pytest.raises(ValueError):
        fp.setup(0, 0, 0, 0, torch.float32, torch.bfloat16, torch._C._cuda_getDevice,
                 torch._C._cuda_getCurrentRawStream)
