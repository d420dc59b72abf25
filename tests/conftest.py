"""Shared pytest set-up.

Markers:
  gpu  -- needs a CUDA device and the built CUDA library. Such tests skip
          (they do not pass) on a machine without a device, and fail loudly on
          a machine with a device but without the library.
"""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the built CUDA library")


def _has_cuda() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree if missing. Skips without a device."""
    if not _has_cuda():
        pytest.skip("no CUDA device: could not check (skipped, not passed)")
    from similarity_softmax_candidate_gb300 import _build, binding
    _build.build_library()
    return binding.library()


@pytest.fixture(scope="session")
def host_lib():
    """The CUDA library loaded on a machine that may have no GPU: only
    symbol lookups and argument-validation calls (which return before any
    CUDA call) are allowed through this fixture."""
    from similarity_softmax_candidate_gb300 import _build, binding
    _build.build_library()
    return binding.library()
