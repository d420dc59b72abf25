"""The two native measurement programs the benchmark runs, each on a small
case: cs_latency (microseconds per call of the C ABI, from C++) and
cs_copy_ceiling (the read ceiling of the streaming kernel's bulk-copy
access pattern). Both print one line of JSON."""
from __future__ import annotations

import json
import subprocess

import pytest

pytestmark = pytest.mark.gpu


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, f"{cmd[0]} exited {r.returncode}: {r.stderr.strip()[-300:]}"
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_latency_tool_reports_warm_cold_and_isolated_timings(cuda_lib):
    """Every timing is a mean over many calls; a call that must read its
    inputs from HBM takes at least as long as one served from L2 (within
    the noise of a subtraction), and the input pool it rotates over is
    larger than the 129 MB L2."""
    from similarity_softmax_candidate_gb300 import _build
    tool = _build.build_latency_tool()
    for unfused in (0, 1):
        d = _run([tool, "1", "64", "512", "1", "200", str(unfused)])
        for key in ("direct_warm_us", "direct_cold_us", "graph_warm_us", "graph_cold_us", "isolated_cold_us"):
            assert 0.0 < d[key] < 1000.0, (key, d)
        assert d["pool_mib"] >= 512 and d["slices"] >= 64
        assert d["graph_cold_us"] >= 0.9 * d["graph_warm_us"], d
        assert d["calls"] >= 200


def test_copy_ceiling_tool_streams_every_byte_it_reports(cuda_lib):
    from similarity_softmax_candidate_gb300 import _build
    tool = _build.build_copy_ceiling_tool()
    # 12 KB stages, 16 slots, 8 lanes, 2 launches over about 300 MB
    d = _run([tool, str(300 * 1024 * 1024), "12288", "16", "8", "2"])
    unit = d["ctas"] * 12288 * 2
    assert d["total_bytes"] > 0 and d["total_bytes"] % unit == 0
    assert d["stages"] == 16 and d["lanes"] == 8 and d["launches"] == 2
    assert 0.0 < d["gbs_min"] <= d["gbs"] <= d["gbs_max"]


def test_copy_ceiling_tool_refuses_a_ring_its_lanes_cannot_own(cuda_lib):
    from similarity_softmax_candidate_gb300 import _build
    tool = _build.build_copy_ceiling_tool()
    r = subprocess.run([tool, str(64 * 1024 * 1024), "12288", "12", "8", "1"], capture_output=True, text=True,
                       timeout=60)
    assert r.returncode == 1 and "bad arguments" in r.stderr
