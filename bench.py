#!/usr/bin/env python
"""Benchmark of fused candidate scoring on GB300.

Headline workload: 16384 questions, K=255 candidates of D=512 float32
features each (8.6 GB of candidates, larger than the 129 MB L2), CLM cosine
scoring with scale 1/0.07 and temperature 1, scored as four launches over
consecutive slices of 4096 questions. One "step" is those four launches.
The same workload is also timed with Kev dot scoring (scale 1/16).

Printed on one JSON line (rank 0):
  value      questions/s of the whole job, inputs resident in HBM
  e2e        the same metric with inputs streamed from pinned host memory
             and the probabilities copied back, every step
  roofline   the streaming kernel's algorithmic bytes per launch / its mean
             launch time (CUDA events on its stream), against the measured
             HBM copy bandwidth
  cpu_baseline  the fp64 oracle timed on a bounded sample on the host cores
  extra      dot scoring, bfloat16 candidates, a ragged batch, the unfused
             baseline, the projected readout, the copy ceiling of the
             access pattern, and single-question latency for the page's
             five shapes (us/call: warm and HBM-cold, direct and in a
             CUDA graph, and isolated calls)

--impl reference times the fp64 oracle (the only reference there is) on
bounded samples of the same workload, on the host cores.

Under torchrun each rank runs the whole workload on its own GPU (replicas:
questions are independent, there is nothing to exchange); timing is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

B_TOTAL = 16384
CHUNK = 4096
K = 255
D = 512
BYTES_PER_QUESTION = 4 * (K * D + D + K)  # C row block + q read once, p written once

# The page's five shapes (PR #69, "What it is worth"): RTX 4090 fused time in
# us and fused/unfused speed-up, quoted as context.
PAGE_SHAPES = [
    ("clm-cosine-5x512", 1, 5, 512, 1, 9.2, 1.22),
    ("clm-cosine-64x512", 1, 64, 512, 1, 12.1, 1.51),
    ("clm-cosine-255x512", 1, 255, 512, 1, 23.6, 1.79),
    ("clm-cosine-batch8-255x512", 8, 255, 512, 1, 23.8, 1.84),
    ("kev-dot-255x2560", 1, 255, 2560, 0, 55.3, 1.81),
]

METRIC = "questions/s (K=255, D=512, cosine, 16384 questions in 4 launches of 4096)"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x, device=None):
    """Maximum of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, max_ms, world):
    """Units per second of the whole job: every rank processed
    units_per_rank, the slowest in max_ms."""
    return world * units_per_rank / (max_ms / 1e3)


def _peak_hbm():
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return 6800.0, "fallback"


def _sm_max_mhz():
    """Maximum SM clock in MHz (measured file, else the GB300's 2070)."""
    try:
        with open(os.path.join(_ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["sm_max_mhz"])
    except Exception:
        return 2070.0


def _peak_bf16():
    """Dense bf16 tensor peak in TFLOP/s: the measured cuBLAS burst figure
    (the projections are timed alone), else the recipe's fallback."""
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


def _traffic_from_profile(kernel_src_sha):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(_ROOT, "profiles", "stream_kernel_throughput_k255_d512.txt")
    try:
        fields = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != kernel_src_sha:
            return None
        return float(fields["dram_bytes_per_4096_question_launch"])
    except Exception:
        return None


def _strip_comments(src):
    """C/C++ source without its comments (string and character literals
    kept), blank lines and trailing blanks: a comment-only edit leaves the
    code, and so its fingerprint, alone."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = ("".join(out)).splitlines()
    return "\n".join(line.rstrip() for line in lines if line.strip())


def _kernel_sha():
    """Fingerprint of the streaming kernel's code (kernels.cu, internal.h,
    abi.cpp without comments), matched against the committed ncu summary."""
    import hashlib
    h = hashlib.sha256()
    for name in ("kernels.cu", "internal.h", "abi.cpp"):
        with open(os.path.join(_ROOT, "similarity_softmax_candidate_gb300", "csrc", name)) as f:
            h.update(_strip_comments(f.read()).encode())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during timed regions."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.windows = []
        self.file = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def window(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.close()
        rows = []
        import datetime
        for line in open(self.file.name):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except Exception:
                continue
        os.unlink(self.file.name)
        sel = [r for r in rows if any(a - 0.06 <= r[0] <= b + 0.06 for a, b in self.windows)] or rows
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in sel:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": sorted(reasons), "samples": len(sel)}


def _time_oracle(sample_Q, sample_C, normalize, scale):
    import oracle
    t0 = time.perf_counter()
    oracle.score_batch(sample_Q, sample_C, normalize, scale, 1.0)
    return time.perf_counter() - t0


def _host_sample(n, seed=4):
    """n questions of the throughput workload's shape and distribution,
    drawn on the host (float32 N(0,1))."""
    from similarity_softmax_candidate_gb300 import workloads
    wl = workloads.random_case(n, K, D, 1, workloads.CLM_SCALE, seed, "cpu")
    return wl.Q.numpy(), wl.C.numpy()


# ---- the oracle on every host core: one spawned worker process per core,
# each scoring its own host-drawn sample (the oracle itself is single-threaded
# C; questions are independent, so the workers share nothing).
_POOL_SAMPLE = None


def _pool_init(n, seed):
    global _POOL_SAMPLE
    _POOL_SAMPLE = _host_sample(n, seed=seed)


def _pool_passes(passes):
    from similarity_softmax_candidate_gb300 import workloads
    Qs, Cs = _POOL_SAMPLE
    t = 0.0
    for _ in range(passes):
        t += _time_oracle(Qs, Cs, 1, workloads.CLM_SCALE)
    return len(Qs) * passes, t


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """Spawned worker processes (spawn, never fork, after CUDA has been
    used), each holding n host-drawn questions."""

    def __init__(self, n, seed, workers=None):
        import multiprocessing as mp
        self.workers = workers or _host_cores()
        self.n = n
        self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_pool_init, initargs=(n, seed))
        self.run(1)  # every worker initialised and warm

    def run(self, passes):
        """Each worker scores its sample `passes` times; returns (questions,
        wall seconds)."""
        t0 = time.perf_counter()
        res = self.pool.map(_pool_passes, [passes] * self.workers, chunksize=1)
        return sum(r[0] for r in res), time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline_all_cores(target_s=10.0):
    """The oracle as it stands on every host core (one process per core)
    for about target_s of wall time."""
    from similarity_softmax_candidate_gb300 import workloads
    Qp, Cp = _host_sample(8)
    t_q = _time_oracle(Qp, Cp, 1, workloads.CLM_SCALE) / 8
    n = 128
    pool = OraclePool(n, seed=7)
    try:
        passes = int(max(1, target_s / max(t_q * n, 1e-6)))
        done, dt = pool.run(passes)
    finally:
        pool.close()
    return {"value": done / dt, "unit": "questions/s", "cores": pool.workers, "kind": "oracle",
            "host_cpu_count": os.cpu_count(), "affine_cores": _host_cores(),
            "sample": f"{done} question scorings: {pool.workers} processes (one per affine host core), each "
                      f"{passes} passes over its own {n} host-drawn questions of the K=255, D=512 cosine "
                      f"workload; fp64 C oracle, {dt:.1f} s wall"}


def cpu_baseline(target_s=10.0):
    """The oracle as it stands (single-threaded C, fp64) on a bounded sample:
    passes over up to 2048 host-drawn questions until about target_s of CPU
    time has been spent."""
    from similarity_softmax_candidate_gb300 import workloads
    Qp, Cp = _host_sample(8)
    t_probe = _time_oracle(Qp, Cp, 1, workloads.CLM_SCALE) / 8
    n = int(max(8, min(2048, target_s / max(t_probe, 1e-6))))
    Qs, Cs = _host_sample(n, seed=5)
    dt, done = 0.0, 0
    while dt < target_s or done == 0:
        dt += _time_oracle(Qs, Cs, 1, workloads.CLM_SCALE)
        done += n
    return {"value": done / dt, "unit": "questions/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} question scorings ({done // n} passes over {n} questions of the K=255, D=512 "
                      f"cosine workload, host-drawn N(0,1)), fp64 C oracle, single thread, {dt:.1f} s"}


def run_reference(args):
    """The reference arm: the oracle as it stands, one process per affine
    host core; each step every worker scores its own bounded sample once."""
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    from similarity_softmax_candidate_gb300 import workloads
    Qp, Cp = _host_sample(8)
    t_q = _time_oracle(Qp, Cp, 1, workloads.CLM_SCALE) / 8
    budget = 60.0  # seconds of wall time for warm-up + timed steps
    n = int(max(1, min(256, budget / max(t_q, 1e-6) / max(1, args.steps + args.warmup))))
    pool = OraclePool(n, seed=6)
    try:
        for _ in range(args.warmup):
            pool.run(1)
        total, done = 0.0, 0
        for _ in range(args.steps):
            q, dt = pool.run(1)
            total += dt
            done += q
    finally:
        pool.close()
    qps = done / total
    line = {
        "impl": "reference", "metric": METRIC, "value": qps, "unit": "questions/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"throughput: cosine, K={K}, D={D}; each step a bounded sample of "
                               f"{n} questions per host core",
                   "B": n * pool.workers, "K": K, "D": D},
        "cpu_baseline": {"value": qps, "unit": "questions/s", "cores": pool.workers, "kind": "oracle",
                         "host_cpu_count": os.cpu_count(), "affine_cores": _host_cores(),
                         "sample": f"{n} questions per process per step, {pool.workers} processes (one per "
                                   f"affine host core), host-drawn N(0,1), fp64 C oracle"},
        "e2e": {"value": qps, "unit": "questions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    global B_TOTAL, CHUNK
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--latency-calls", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-extra", action="store_true", help="only the headline throughput and its roofline")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle's CPU baseline")
    ap.add_argument("--questions", type=int, default=B_TOTAL,
                    help="questions per step (default 16384; smaller only for profiling captures)")
    ap.add_argument("--chunk", type=int, default=CHUNK, help="questions per launch (default 4096)")
    ap.add_argument("--only-unaligned", action="store_true",
                    help="profiling aid: time only the unaligned-row workloads and print their record")
    ap.add_argument("--only-unaligned-case", choices=[c[0] for c in UNALIGNED_CASES], default=None,
                    help="profiling aid: W + K calls of one unaligned-row case (cosine, 4096 questions)")
    ap.add_argument("--only-unaligned-dtype", choices=["f32", "bf16"], default="f32",
                    help="candidate type of --only-unaligned-case")
    ap.add_argument("--only-unaligned-plan", choices=["auto", "generic"], default="auto",
                    help="plan of --only-unaligned-case (generic: the scalar plan forced, float32)")
    ap.add_argument("--only-unaligned-b1", action="store_true",
                    help="profiling aid: time only one-question calls on unaligned rows and print their record")
    ap.add_argument("--only-projected", type=int, default=0, metavar="B",
                    help="profiling aid: time only the projected readout on B questions and print its record")
    ap.add_argument("--plan-sweep", action="store_true",
                    help="profiling aid: us per call of every plan the library offers, against the automatic "
                         "choice, for B = 1 .. 152 questions of K=255, D=512 (CUDA-graph replays)")
    ap.add_argument("--only-shape", choices=[r[0] for r in PAGE_SHAPES], default=None,
                    help="profiling aid: W warm-up calls, then K back-to-back calls of one of the page's "
                         "small shapes; prints us per call and the plan")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import similarity_softmax_candidate_gb300 as cs
    from similarity_softmax_candidate_gb300 import _build, workloads
    _build.build_library()
    if args.only_shape:
        if rank == 0:
            print(json.dumps(single_shape(cs, workloads, dev, args.only_shape, args.steps, args.warmup)), flush=True)
        return 0
    if args.plan_sweep:
        if rank == 0:
            print(json.dumps(plan_sweep(cs, dev)), flush=True)
        return 0
    if args.only_unaligned_case:
        if rank == 0:
            print(json.dumps(unaligned_rows(cs, dev, args.steps, args.warmup, only=args.only_unaligned_case,
                                            only_dtype=args.only_unaligned_dtype, only_plan=args.only_unaligned_plan)),
                  flush=True)
        return 0
    if args.only_unaligned:
        if rank == 0:
            print(json.dumps(unaligned_rows(cs, dev, args.steps, args.warmup)), flush=True)
        return 0
    if args.only_unaligned_b1:
        if rank == 0:
            print(json.dumps(unaligned_latency(cs, dev)), flush=True)
        return 0
    if args.only_projected:
        if rank == 0:
            print(json.dumps(projected_readout(cs, dev, args.steps, args.warmup, B=args.only_projected)), flush=True)
        return 0

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max(x, dev)

    B_TOTAL, CHUNK = args.questions, args.chunk
    if B_TOTAL % CHUNK:
        ap.error("--questions must be a multiple of --chunk")
    wls = workloads.throughput(dev, B=B_TOTAL)
    wl_cos, wl_dot = wls
    out = torch.empty((B_TOTAL, K), device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = cs.cs_query_plan(wl_cos.Q[:CHUNK], wl_cos.C[:CHUNK], 1)

    def step(wl):
        for b0 in range(0, B_TOTAL, CHUNK):
            cs.cs_score_candidates_batch(wl.Q[b0:b0 + CHUNK], wl.C[b0:b0 + CHUNK], wl.normalize, wl.scale,
                                         wl.temperature, out=out[b0:b0 + CHUNK], stream=stream)

    clocks = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    clocks.start()

    def timed(wl):
        """K steps between two CUDA events on the launching stream. Nothing
        else enters the stream between the launches: an event recorded
        between two launches makes the second wait for the first's full
        completion, which takes away the dependent-launch overlap a caller's
        back-to-back calls get (about 3 % of the step). The step is nothing
        but these launches, so its time over the launches is the mean launch
        time the roofline uses."""
        for _ in range(args.warmup):
            step(wl)
        barrier()
        n_launch = args.steps * (B_TOTAL // CHUNK)
        t_wall = time.time()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            step(wl)
        stop.record(stream)
        barrier()
        clocks.window(t_wall, time.time())
        ms = max_over_ranks(start.elapsed_time(stop))
        return ms, [ms / n_launch] * n_launch, n_launch

    ms_cos, launches_cos, n_launch = timed(wl_cos)
    ms_dot, launches_dot, _ = timed(wl_dot)
    clock_info = clocks.stop()

    bf16, ragged_info, unfused = {}, {}, {}
    if not args.skip_extra:
        bf16, ragged_info, unfused = extras(cs, workloads, wl_cos, wl_dot, out, dev, stream, args, world, barrier,
                                            max_over_ranks, ms_cos, ms_dot)

    ms_per_step = ms_cos / args.steps
    value = whole_job_rate(B_TOTAL, ms_per_step, world)
    peak, peak_kind = _peak_hbm()
    launch_bytes = CHUNK * BYTES_PER_QUESTION
    mean_launch_ms = sum(launches_cos) / len(launches_cos)
    achieved = launch_bytes / (mean_launch_ms / 1e3) / 1e9
    traffic = _traffic_from_profile(_kernel_sha())
    if traffic is not None:
        traffic *= CHUNK / 4096.0
    dot_ms_step = ms_dot / args.steps
    dot_launch_ms = sum(launches_dot) / len(launches_dot)

    line = {
        "metric": METRIC, "value": value, "unit": "questions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"throughput: {B_TOTAL} questions x K=255 x D=512 fp32 N(0,1), CLM cosine "
                               f"(scale 1/0.07, T=1), {B_TOTAL // CHUNK} launches of {CHUNK} questions per step",
                   "B": B_TOTAL, "K": K, "D": D, "launches_per_step": B_TOTAL // CHUNK,
                   "l2": f"inputs ({B_TOTAL * K * D * 4 / 1e9:.1f} GB per rank) larger than L2 (129 MB); no flush",
                   "plan": plan, "parallelism": f"replicas x{world}"},
        "gpu_launches": n_launch,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": f"stream_kernel (STREAM plan), one launch = {CHUNK} questions",
                     "algorithmic_bytes_per_launch": launch_bytes, "mean_launch_ms": mean_launch_ms,
                     "mean_launch_ms_from": "the timed steps' CUDA events over their launches (the step is "
                                            "only this kernel's launches, back to back)",
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"},
        "clocks": clock_info,
        "extra": {
            "hbm_gbs_step": world * B_TOTAL * BYTES_PER_QUESTION / (ms_per_step / 1e3) / 1e9,
            "frac_of_8tbs_nominal": achieved / 8000.0,
            "dot": {"questions_per_s": world * B_TOTAL / (dot_ms_step / 1e3), "ms_per_step": dot_ms_step,
                    "launch_gbs": launch_bytes / (dot_launch_ms / 1e3) / 1e9,
                    "frac": launch_bytes / (dot_launch_ms / 1e3) / 1e9 / peak},
            "unfused_baseline": unfused,
            "bf16_candidates": bf16,
            "ragged_cosine": ragged_info,
        },
    }

    if not args.skip_extra:
        line["extra"]["projected_readout"] = projected_readout(cs, dev, 20, args.warmup)
        line["extra"]["unaligned_rows"] = unaligned_rows(cs, dev, 20, args.warmup)
        line["extra"]["unaligned_b1"] = unaligned_latency(cs, dev)
        line["extra"]["latency_b1"] = latency_table(cs, workloads, dev, args.latency_calls)
        line["e2e"] = e2e(cs, wl_cos, dev, args, world, barrier, max_over_ranks)
    del wls, wl_cos, wl_dot
    torch.cuda.empty_cache()
    if rank == 0 and not args.skip_extra:
        line["extra"]["copy_ceiling"] = copy_ceiling(line["extra"]["hbm_gbs_step"] / world, achieved)

    if rank == 0 and not args.no_cpu:
        try:
            line["cpu_baseline"] = cpu_baseline_all_cores(args.cpu_seconds)
            line["extra"]["cpu_baseline_one_core"] = cpu_baseline(args.cpu_seconds / 2)
        except Exception as e:  # the oracle is optional for the GPU numbers
            line["cpu_baseline"] = {"value": None, "unit": "questions/s", "cores": 1, "kind": "oracle",
                                    "sample": f"failed: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def extras(cs, workloads, wl_cos, wl_dot, out, dev, stream, args, world, barrier, max_over_ranks, ms_cos, ms_dot):
    """bfloat16 candidates, a ragged batch and the unfused baseline on the
    throughput workload's sizes (extra keys of the JSON line)."""
    import torch
    bf16 = {}
    Cb = torch.empty(wl_cos.C.shape, device=dev, dtype=torch.bfloat16)
    for b0 in range(0, B_TOTAL, CHUNK):
        Cb[b0:b0 + CHUNK].copy_(wl_cos.C[b0:b0 + CHUNK])
    bytes_q_bf16 = 2 * K * D + 4 * D + 4 * K
    for wl in (wl_cos, wl_dot):
        def bstep(wl=wl):
            for b0 in range(0, B_TOTAL, CHUNK):
                cs.cs_score_candidates_batch_bf16(wl.Q[b0:b0 + CHUNK], Cb[b0:b0 + CHUNK], wl.normalize, wl.scale,
                                                  wl.temperature, out=out[b0:b0 + CHUNK], stream=stream)
        for _ in range(args.warmup):
            bstep()
        barrier()
        ba, bb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        bsteps = max(3, args.steps // 2)
        ba.record(stream)
        for _ in range(bsteps):
            bstep()
        bb.record(stream)
        barrier()
        bms = max_over_ranks(ba.elapsed_time(bb)) / bsteps
        gbs = world * B_TOTAL * bytes_q_bf16 / (bms / 1e3) / 1e9
        bf16["cos" if wl.normalize else "dot"] = {
            "questions_per_s": world * B_TOTAL / (bms / 1e3), "ms_per_step": bms, "hbm_gbs": gbs,
            "frac": gbs / _peak_hbm()[0], "algorithmic_bytes_per_question": bytes_q_bf16, "steps": bsteps}
    del Cb

    # A ragged batch of the same size: K_b uniform in [1, 255], one launch.
    rw = workloads.ragged(B_TOTAL, D, 1, workloads.CLM_SCALE, 12, dev)
    rout = torch.empty(rw.total_rows, device=dev)
    ragged_bytes = 4 * (rw.total_rows * D + B_TOTAL * D + rw.total_rows)

    def rstep():
        cs.cs_score_candidates_ragged(rw.Q, rw.C, rw.offsets, 1, rw.scale, 1.0, out=rout, stream=stream)
    for _ in range(args.warmup):
        rstep()
    barrier()
    ra, rb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rsteps = max(3, args.steps // 2)
    ra.record(stream)
    for _ in range(rsteps):
        rstep()
    rb.record(stream)
    barrier()
    rms = max_over_ranks(ra.elapsed_time(rb)) / rsteps
    ragged_info = {"questions_per_s": world * B_TOTAL / (rms / 1e3), "ms_per_call": rms,
                   "hbm_gbs": world * ragged_bytes / (rms / 1e3) / 1e9,
                   "frac": world * ragged_bytes / (rms / 1e3) / 1e9 / _peak_hbm()[0],
                   "total_rows": rw.total_rows, "K_range": [1, 255], "steps": rsteps}
    del rw, rout

    # The unfused baseline on the same workload (two launches per slice).
    staged = torch.empty((B_TOTAL, K), device=dev)
    unfused = {}
    for wl in (wl_cos, wl_dot):
        def ustep(wl=wl):
            for b0 in range(0, B_TOTAL, CHUNK):
                cs.cs_score_candidates_batch_unfused(wl.Q[b0:b0 + CHUNK], wl.C[b0:b0 + CHUNK], wl.normalize,
                                                     wl.scale, wl.temperature, staged=staged[b0:b0 + CHUNK],
                                                     out=out[b0:b0 + CHUNK], stream=stream)
        for _ in range(args.warmup):
            ustep()
        barrier()
        ua, ub = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        usteps = max(3, args.steps // 4)
        ua.record(stream)
        for _ in range(usteps):
            ustep()
        ub.record(stream)
        barrier()
        ums = max_over_ranks(ua.elapsed_time(ub)) / usteps
        fused_ms = (ms_cos if wl.normalize else ms_dot) / args.steps
        unfused["cos" if wl.normalize else "dot"] = {
            "questions_per_s": world * B_TOTAL / (ums / 1e3), "ms_per_step": ums,
            "fused_over_unfused": ums / fused_ms, "steps": usteps}
    del staged

    return bf16, ragged_info, unfused


# (name, D, element offset of Q and C from a 16-byte boundary, questions,
# the aligned case it is compared with)
UNALIGNED_CASES = (("aligned_d512", 512, 0, 4096, None), ("odd_d510", 510, 0, 4096, "aligned_d512"),
                   ("misaligned_d512", 512, 1, 4096, "aligned_d512"), ("aligned_d2560", 2560, 0, 1024, None),
                   ("misaligned_d2560", 2560, 1, 1024, "aligned_d2560"))


def unaligned_rows(cs, dev, steps, warmup, only=None, only_dtype="f32", only_plan="auto"):
    """Rows the bulk copies cannot take whole, at throughput size: 4096
    questions of K=255 with D=510 (rows of 2040 bytes), and with D=512 but
    Q and C one element past a 16-byte boundary, each against the aligned
    D=512 readout on the same buffer; and 1024 questions of D=2560 one
    element off, against aligned D=2560. Float32 cases also against the
    scalar plan forced on the same rows; float32 and bfloat16 candidates.
    One launch per call over at least 2.1 GB (larger than L2). only: time
    just that case's cosine readout with only_dtype candidates and the
    automatic plan, or with only_plan "generic" the scalar plan forced
    (float32; profiling aids)."""
    import torch
    n_c = max(B * K * d for _, d, _, B, _ in UNALIGNED_CASES) + 64
    n_q = max(B * d for _, d, _, B, _ in UNALIGNED_CASES) + 64
    flatC = torch.empty(n_c, device=dev)
    flatQ = torch.empty(n_q, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(31)
    flatC.normal_(generator=g)
    flatQ.normal_(generator=g)
    s = torch.cuda.current_stream(dev)
    if only is not None:
        _, d, off, B, _ = next(c for c in UNALIGNED_CASES if c[0] == only)
        out = torch.empty(B, K, device=dev)
        Q = flatQ[off:off + B * d].view(B, d)
        bf = only_dtype == "bf16"
        flat = flatC[:B * K * d + 64].to(torch.bfloat16) if bf else flatC
        C = flat[off:off + B * K * d].view(B, K, d)
        score = cs.cs_score_candidates_batch_bf16 if bf else cs.cs_score_candidates_batch
        if only_plan == "generic":
            if bf:
                raise SystemExit("--only-unaligned-plan generic takes float32 candidates")

            def score(Q, C, normalize, scale, T, out, stream):
                return cs.cs_score_candidates_batch_plan(Q, C, normalize, scale, T, cs.CS_PLAN_GENERIC, 1, 0,
                                                         out=out, stream=stream)
        for _ in range(warmup + steps):
            score(Q, C, 1, 14.285714, 1.0, out=out, stream=s)
        torch.cuda.synchronize()
        return {"case": only, "dtype": only_dtype, "plan_forced": only_plan, "calls": warmup + steps,
                "plan": None if bf else cs.cs_query_plan(Q, C, 1)}

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(steps):
            fn()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    res = {}
    flatCb = flatC.to(torch.bfloat16)
    for name, d, off, B, _ in UNALIGNED_CASES:
        out = torch.empty(B, K, device=dev)
        Q = flatQ[off:off + B * d].view(B, d)
        row = {"questions": B, "D": d}
        for dt, flat, eb in (("f32", flatC, 4), ("bf16", flatCb, 2)):
            C = flat[off:off + B * K * d].view(B, K, d)
            score = cs.cs_score_candidates_batch if dt == "f32" else cs.cs_score_candidates_batch_bf16
            if dt == "f32":
                row["plan"] = cs.cs_query_plan(Q, C, 1)["plan"]
            nbytes = B * (eb * K * d + 4 * d + 4 * K)
            for normalize, scale in ((1, 14.285714), (0, 0.0625)):
                tag = dt + ("_cos" if normalize else "_dot")
                ms = timed(lambda: score(Q, C, normalize, scale, 1.0, out=out, stream=s))
                row[tag + "_gbs"] = nbytes / (ms / 1e3) / 1e9
                row[tag + "_questions_per_s"] = B / (ms / 1e3)
                if dt == "f32" and (off or d % 4):
                    ms_g = timed(lambda: cs.cs_score_candidates_batch_plan(Q, C, normalize, scale, 1.0,
                                                                           cs.CS_PLAN_GENERIC, 1, 0, out=out,
                                                                           stream=s))
                    row[tag + "_scalar_plan_gbs"] = nbytes / (ms_g / 1e3) / 1e9
        res[name] = row
    for name, _, _, _, ref in UNALIGNED_CASES:
        if ref:
            for tag in ("f32_cos", "f32_dot", "bf16_cos", "bf16_dot"):
                res[name][tag + "_over_aligned"] = res[name][tag + "_gbs"] / res[ref][tag + "_gbs"]
    res["workload"] = (f"K=255, N(0,1), float32 and bfloat16 candidates, one launch per call, {steps} calls; "
                       f"each unaligned case against the aligned case of its D and question count")
    del flatC, flatQ, flatCb
    return res


def projected_readout(cs, dev, steps, warmup, B=4096):
    """The readout with caller-side projections on the tensor cores
    (cs_project_score_batch), B questions (4096 by default), K=255,
    Din=D=512, bfloat16 features and heads; against projecting with cuBLAS
    (torch.matmul, bf16 out) and scoring the bfloat16 result with the
    streaming kernel."""
    import torch
    Kq, Din, Dp = K, 512, 512
    g = torch.Generator(device=dev)
    g.manual_seed(21)
    Hq = torch.randn(B, Din, device=dev, generator=g).to(torch.bfloat16)
    Hc = torch.randn(B, Kq, Din, device=dev, generator=g).to(torch.bfloat16)
    Wq = (torch.randn(Dp, Din, device=dev, generator=g) * Din ** -0.5).to(torch.bfloat16)
    Wc = (torch.randn(Dp, Din, device=dev, generator=g) * Din ** -0.5).to(torch.bfloat16)
    qproj = torch.empty(B, Dp, device=dev)
    outp = torch.empty(B, Kq, device=dev)
    s = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(steps):
            fn()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    fused_ms = timed(lambda: cs.cs_project_score_batch(Hq, Wq, Hc, Wc, 1, 14.285714, 1.0, qproj=qproj, out=outp,
                                                       stream=s))

    def composed():
        c = torch.matmul(Hc.view(B * Kq, Din), Wc.t()).view(B, Kq, Dp)
        q = torch.matmul(Hq, Wq.t()).float()
        cs.cs_score_candidates_batch_bf16(q, c, 1, 14.285714, 1.0, out=outp, stream=s)
    composed_ms = timed(composed)
    Hrows = Hc.view(B * Kq, Din)
    Prows = torch.empty((B * Kq, Dp), device=dev)
    rows_ms = timed(lambda: cs.cs_project_rows(Hrows, Wc, out=Prows, stream=s))
    rows_bytes = 2.0 * B * Kq * Din + 2.0 * Dp * Din + 4.0 * B * Kq * Dp
    # Writes alone: P filled (torch's fill_), the kernel's 2.14 GB of
    # stores without its reads or arithmetic.
    fill_ms = timed(lambda: Prows.fill_(1.0))
    hbm, hbm_src = _peak_hbm()
    flop = 2.0 * B * Kq * Din * Dp + 2.0 * B * Din * Dp
    peak, peak_src = _peak_bf16()
    # Shared-memory bound of a one-SM tcgen05 kernel: each 128-row x 256-
    # feature unit (Din deep) writes its A and W tiles into shared memory by
    # TMA and the MMAs read them back once, 2 x (128 + 256) x Din x 2 bytes
    # through a port of 32 banks x 4 bytes per clock.
    smem_bytes_unit = 2 * (128 + 256) * Din * 2
    flop_unit = 2.0 * 128 * 256 * Din
    sm_mhz, sms = _sm_max_mhz(), torch.cuda.get_device_properties(dev).multi_processor_count
    smem_bound = flop_unit / (smem_bytes_unit / 128.0) * sms * sm_mhz * 1e6 / 1e12
    rows_smem_unit = smem_bytes_unit  # the outputs go from registers to global memory
    rows_units = -(-(B * Kq) // 128) * (Dp // 256)
    rows_smem_ms = -(-rows_units // sms) * rows_smem_unit / 128.0 / (sm_mhz * 1e6) * 1e3
    return {"workload": f"{B} questions x K=255, Din=512 -> D=512, bf16 features and heads, cosine",
            "questions_per_s": B / (fused_ms / 1e3), "ms_per_call": fused_ms,
            "tflops": flop / (fused_ms / 1e3) / 1e12, "peak_tflops": peak,
            "frac": flop / (fused_ms / 1e3) / 1e12 / peak,
            "peak_source": peak_src,
            "smem_bound": {"bytes_per_unit": smem_bytes_unit, "bytes_per_clock": 128, "sm_mhz": sm_mhz,
                           "tflops": smem_bound, "frac": flop / (fused_ms / 1e3) / 1e12 / smem_bound},
            "composed_cublas_bf16_ms": composed_ms, "fused_over_composed": composed_ms / fused_ms,
            "project_rows": {"rows": B * Kq, "ms_per_call": rows_ms,
                             "tflops": 2.0 * B * Kq * Din * Dp / (rows_ms / 1e3) / 1e12,
                             "gbs": rows_bytes / (rows_ms / 1e3) / 1e9,
                             "frac_of_copy": rows_bytes / (rows_ms / 1e3) / 1e9 / hbm,
                             "peak_source": f"hbm_gbs ({hbm_src})",
                             "smem_bound": {"bytes_per_unit": rows_smem_unit, "bytes_per_clock": 128,
                                            "sm_mhz": sm_mhz, "ms": rows_smem_ms, "frac": rows_smem_ms / rows_ms},
                             "writes_alone": {
                                 "what": "torch fill_ of P (the kernel's stores, no reads, no arithmetic)",
                                 "ms": fill_ms, "write_gbs": 4.0 * B * Kq * Dp / (fill_ms / 1e3) / 1e9,
                                 "rows_ms_over_fill_ms": rows_ms / fill_ms}}}


def plan_sweep(cs, dev, Bs=(1, 2, 4, 8, 16, 24, 32, 48, 64, 76, 100, 152), n=32):
    """us per call, cosine K=255 D=512, of the automatic plan and of every
    forced plan (STREAM; CLUSTER with 2..16 CTAs per question; DIRECT over 8
    and 16 CTAs where it fits), each as n calls on consecutive slices of a
    4096-question buffer captured in one CUDA graph after a read of a
    256 MiB buffer (which leaves L2 holding none of the slices), minus the
    same graph without the calls: device time per call, every call reading
    from HBM, no host work."""
    import torch
    Bmax = 4096
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    C = torch.randn(Bmax, K, D, device=dev, generator=g)
    Q = torch.randn(Bmax, D, device=dev, generator=g)
    out = torch.empty(Bmax, K, device=dev)
    flush = torch.ones(64 << 20, device=dev)  # 256 MiB, read only
    plans = [("stream", cs.CS_PLAN_STREAM, 0)] + [(f"cluster{G}", cs.CS_PLAN_CLUSTER, G) for G in (2, 4, 8, 16)] + \
        [("direct8", cs.CS_PLAN_DIRECT, 8), ("direct16", cs.CS_PLAN_DIRECT, 16)]

    def timed(B, plan, G):
        nsl = Bmax // B

        def call(i):
            s0 = (i % nsl) * B
            if plan is None:
                cs.cs_score_candidates_batch(Q[s0:s0 + B], C[s0:s0 + B], 1, 14.285714, 1.0, out=out[s0:s0 + B])
            else:
                cs.cs_score_candidates_batch_plan(Q[s0:s0 + B], C[s0:s0 + B], 1, 14.285714, 1.0, plan, G, 0,
                                                  out=out[s0:s0 + B])
        for i in range(4):
            call(i)
        torch.cuda.synchronize()

        def graph_ms(calls):
            graph, st = torch.cuda.CUDAGraph(), torch.cuda.Stream(dev)
            with torch.cuda.stream(st):
                with torch.cuda.graph(graph, stream=st):
                    flush.sum()
                    for i in range(calls):
                        call(i)
            graph.replay()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(10):
                    graph.replay()
                b.record()
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b) / 10)
            return best
        return 1e3 * (graph_ms(n) - graph_ms(0)) / n

    rows = []
    for B in Bs:
        auto = cs.cs_query_plan(Q[:B], C[:B], 1)
        row = {"B": B, "auto": f"{auto['plan']}{auto['cluster'] if auto['cluster'] > 1 else ''}",
               "auto_us": timed(B, None, 0)}
        for name, plan, G in plans:
            try:
                row[name + "_us"] = timed(B, plan, G)
            except cs.CSError:
                row[name + "_us"] = None
        best = min(v for k, v in row.items() if k.endswith("_us") and k != "auto_us" and v is not None)
        row["auto_over_best"] = row["auto_us"] / best
        rows.append(row)
    return {"plan_sweep": rows, "workload": "cosine, K=255, D=512, inputs in HBM (larger than L2 across the graph)"}


def unaligned_latency(cs, dev, n=32):
    """us per call for one question of K=255 whose rows the bulk copies
    cannot take whole (D=510, and D=512 with Q and C one element off a
    16-byte boundary; float32 and bfloat16, cosine): the automatic plan
    against the scalar plan (one question over a 16-CTA cluster) forced on
    the same rows, and the stream kernel's cluster plan (16 CTAs, rows copied
    as aligned spans). Device time per call as in the plan sweep: n calls on
    consecutive slices of a 2.1 GB buffer in one CUDA graph after a read of
    256 MiB, minus the same graph without the calls (every call from HBM)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    n_elem = 4096 * K * 512
    flatC = torch.randn(n_elem + 64, device=dev, generator=g)
    flatCb = flatC.to(torch.bfloat16)
    flatQ = torch.randn(4096 * 512 + 64, device=dev, generator=g)
    out = torch.empty(K, device=dev)
    flush = torch.ones(64 << 20, device=dev)  # 256 MiB, read only

    def timed(score):
        for i in range(4):
            score(i)
        torch.cuda.synchronize()

        def graph_ms(calls):
            graph, st = torch.cuda.CUDAGraph(), torch.cuda.Stream(dev)
            with torch.cuda.stream(st):
                with torch.cuda.graph(graph, stream=st):
                    flush.sum()
                    for i in range(calls):
                        score(i)
            graph.replay()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(10):
                    graph.replay()
                b.record()
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b) / 10)
            return best
        return 1e3 * (graph_ms(n) - graph_ms(0)) / n

    rows = []
    for name, d, off in (("odd_d510", 510, 0), ("misaligned_d512", 512, 1), ("misaligned_d2560", 2560, 1)):
        nsl = n_elem // (K * d) - 1
        views = [(flatQ[off + (i % 4096) * d:off + (i % 4096) * d + d],
                  flatC[off + (i % nsl) * K * d:off + ((i % nsl) + 1) * K * d].view(K, d),
                  flatCb[off + (i % nsl) * K * d:off + ((i % nsl) + 1) * K * d].view(K, d)) for i in range(n)]
        plan = cs.cs_query_plan(views[0][0][None], views[0][1][None], 1)
        row = {"case": name, "K": K, "D": d, "auto_plan": f"{plan['plan']}{plan['cluster']}"}
        row["f32_auto_us"] = timed(lambda i: cs.cs_score_candidates(views[i][0], views[i][1], 1, 14.285714, 1.0,
                                                                    out=out))
        row["f32_scalar16_us"] = timed(lambda i: cs.cs_score_candidates_batch_plan(
            views[i][0][None], views[i][1][None], 1, 14.285714, 1.0, cs.CS_PLAN_GENERIC, 16, 0, out=out[None]))
        row["f32_cluster16_us"] = timed(lambda i: cs.cs_score_candidates_batch_plan(
            views[i][0][None], views[i][1][None], 1, 14.285714, 1.0, cs.CS_PLAN_CLUSTER, 16, 0, out=out[None]))
        row["bf16_auto_us"] = timed(lambda i: cs.cs_score_candidates_bf16(views[i][0], views[i][2], 1, 14.285714,
                                                                          1.0, out=out))
        rows.append(row)
    del flatC, flatCb, flatQ, flush
    return {"rows": rows, "workload": "one question, K=255, cosine, inputs in HBM (larger than L2 across the graph)"}


def single_shape(cs, workloads, dev, name, calls, warmup):
    """One of the page's small shapes alone: warm-up calls, then `calls`
    back-to-back calls timed with CUDA events."""
    import torch
    _, B, k, d, normalize, page_us, _ = next(r for r in PAGE_SHAPES if r[0] == name)
    wl = workloads.random_case(B, k, d, normalize, workloads.CLM_SCALE if normalize else workloads.KEV_SCALE,
                               90 + k, dev)
    out = torch.empty(B, k, device=dev)
    s = torch.cuda.current_stream(dev)

    q0, c0, o0 = wl.Q[0], wl.C[0], out[0]  # views made once, outside the timed calls

    def call():
        if B == 1:
            cs.cs_score_candidates(q0, c0, normalize, wl.scale, 1.0, out=o0, stream=s)
        else:
            cs.cs_score_candidates_batch(wl.Q, wl.C, normalize, wl.scale, 1.0, out=out, stream=s)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(calls):
        call()
    b.record(s)
    torch.cuda.synchronize()
    return {"shape": name, "B": B, "K": k, "D": d, "us_per_call": 1e3 * a.elapsed_time(b) / calls,
            "calls": calls, "plan": cs.cs_query_plan(wl.Q, wl.C, normalize), "page_rtx4090_us": page_us}


def latency_table(cs, workloads, dev, calls):
    """us per call for the page's shapes. From native code (cs_latency, the
    C ABI called from C++): back-to-back calls on the same inputs (warm L2)
    and on rotating slices of a 512 MiB pool (every call reads from HBM),
    directly and inside a 50-call CUDA graph, and an isolated call (each
    preceded by an empty kernel, so it overlaps nothing) reading from HBM;
    the unfused baseline in the same graphs. From Python: back-to-back
    calls through the binding on the same inputs (the binding's own cost is
    the difference from the native direct figure)."""
    import torch
    rows = []
    for name, B, k, d, normalize, page_us, page_ratio in PAGE_SHAPES:
        wl = workloads.random_case(B, k, d, normalize, workloads.CLM_SCALE if normalize else workloads.KEV_SCALE,
                                   90 + k, dev)
        out = torch.empty(B, k, device=dev)
        s = torch.cuda.current_stream(dev)

        q0, c0, o0 = wl.Q[0], wl.C[0], out[0]  # views made once, outside the timed calls

        def call():
            if B == 1:
                cs.cs_score_candidates(q0, c0, normalize, wl.scale, 1.0, out=o0, stream=s)
            else:
                cs.cs_score_candidates_batch(wl.Q, wl.C, normalize, wl.scale, 1.0, out=out, stream=s)

        for _ in range(20):
            call()
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(calls):
                call()
            b.record(s)
            torch.cuda.synchronize()
            reps.append(1e3 * a.elapsed_time(b) / calls)
        python_direct = statistics.median(reps)
        plan = cs.cs_query_plan(wl.Q, wl.C, normalize)
        native = native_latency(B, k, d, normalize, calls)
        row = {"shape": name, "B": B, "K": k, "D": d, "c_abi": native, "python_direct_warm_us": python_direct,
               "plan": plan["plan"], "cluster": plan["cluster"], "ctas": plan["ctas"],
               "rtx4090_fused_us_context": page_us, "rtx4090_ratio_context": page_ratio}
        if "direct_warm_us" in native:
            row["python_over_c_abi_direct_us"] = python_direct - native["direct_warm_us"]
        rows.append(row)
    return rows


def native_latency(B, K, D, normalize, calls):
    """us per call from native code (cs_latency: the C ABI called from C++,
    no Python between calls): warm and HBM-cold back-to-back calls, direct
    and in a 50-call graph, and isolated HBM-cold calls; the unfused
    baseline's graph figures beside them."""
    from similarity_softmax_candidate_gb300 import _build
    try:
        tool = _build.build_latency_tool()
        res = {}
        for unfused in (0, 1):
            r = subprocess.run([tool, str(B), str(K), str(D), str(normalize), str(calls), str(unfused)],
                               capture_output=True, text=True, timeout=300)
            if r.returncode != 0:
                return {"error": r.stderr.strip()[-200:]}
            d = json.loads(r.stdout.strip().splitlines()[-1])
            if unfused:
                for key in ("graph_warm_us", "graph_cold_us"):
                    res["unfused_" + key] = d[key]
            else:
                for key in ("direct_warm_us", "direct_cold_us", "graph_warm_us", "graph_cold_us", "isolated_cold_us",
                            "calls", "pool_mib", "flush_us", "empty_kernel_us"):
                    res[key] = d[key]
        res["fused_over_unfused_graph_warm"] = res["unfused_graph_warm_us"] / res["graph_warm_us"]
        res["fused_over_unfused_graph_cold"] = res["unfused_graph_cold_us"] / res["graph_cold_us"]
        return res
    except Exception as e:  # the Python-side numbers stand without it
        return {"error": str(e)[:200]}


def copy_ceiling(step_gbs, launch_gbs):
    """The read ceiling of the streaming kernel's access pattern on this GPU
    (cs_copy_ceiling: the same 152-CTA geometry, 12 KB stages, a 16-stage
    ring, 8 issuing lanes, no arithmetic) over the workload's 8.6 GB, as one
    launch and as the step's 4 launches; and the kernel's fraction of it."""
    from similarity_softmax_candidate_gb300 import _build
    try:
        tool = _build.build_copy_ceiling_tool()
        res = {"what": "bulk-copy stream, same geometry as the stream plan, no arithmetic (cs_copy_ceiling)"}
        for launches in (1, B_TOTAL // CHUNK):
            r = subprocess.run([tool, str(B_TOTAL * K * D * 4), "12288", "16", "8", str(launches)],
                               capture_output=True, text=True, timeout=120)
            if r.returncode != 0:
                return {"error": (r.stderr.strip() or f"exit {r.returncode}")[-200:]}
            res[f"gbs_{launches}_launch" + ("es" if launches > 1 else "")] = json.loads(r.stdout.strip())["gbs"]
        four = res[f"gbs_{B_TOTAL // CHUNK}_launches"]
        res["step_over_ceiling"] = step_gbs / four
        res["launch_over_ceiling_one_launch"] = launch_gbs / res["gbs_1_launch"]
        return res
    except Exception as e:  # the kernel's own numbers stand without it
        return {"error": str(e)[:200]}


def numa_placement(dev, ptrs):
    """Host NUMA facts for the e2e buffers: the nodes with memory and CPUs,
    the GPU's node (sysfs, from its PCI address) and the node of the first,
    middle and last page of each pinned buffer (get_mempolicy on the
    address). Linux only; fields it cannot read are left out."""
    import ctypes
    import glob
    import platform
    info = {}
    try:
        nodes = {}
        for nd in sorted(glob.glob("/sys/devices/system/node/node[0-9]*")):
            cpus = open(nd + "/cpulist").read().strip()
            mem_kb = int(next(l for l in open(nd + "/meminfo") if "MemTotal" in l).split()[-2])
            nodes[nd.rsplit("node", 1)[1]] = {"cpus": cpus, "mem_gb": round(mem_kb / 2 ** 20, 1)}
        info["nodes"] = nodes
        r = subprocess.run(["nvidia-smi", "-i", str(dev.index or 0), "--query-gpu=pci.bus_id",
                            "--format=csv,noheader"], capture_output=True, text=True, timeout=30)
        bus = r.stdout.strip().splitlines()[0].strip()
        dom, rest = bus.split(":", 1)
        info["gpu_pci"] = bus
        info["gpu_node"] = int(open(f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest.lower()}/numa_node").read())
    except Exception as e:  # not Linux, or no sysfs view
        info["error"] = str(e)[:120]
    try:
        libc = ctypes.CDLL(None, use_errno=True)
        sysno = {"aarch64": 236, "x86_64": 239}[platform.machine()]  # get_mempolicy

        def node_of(addr):
            mode = ctypes.c_int(-1)
            rc = libc.syscall(sysno, ctypes.byref(mode), None, ctypes.c_ulong(0), ctypes.c_void_p(addr),
                              ctypes.c_ulong(3))  # MPOL_F_NODE | MPOL_F_ADDR
            return mode.value if rc == 0 else None
        info["pinned_page_nodes"] = {name: sorted({node_of(p + o) for o in offs})
                                     for name, (p, offs) in ptrs.items()}
    except Exception as e:
        info["pinned_page_nodes_error"] = str(e)[:120]
    return info


def e2e(cs, wl, dev, args, world, barrier, max_over_ranks):
    """questions/s with the inputs in pinned host memory: every step copies
    Q and C host->device (two chunk buffers, copies overlapped with compute
    on a second stream) and the probabilities device->host. Beside it, the
    host link measured the same way in the same run: the step's copies
    alone, no kernel (link_ceiling); per-step rates show the steps the host
    slowed down, and the NUMA placement of the pinned buffers."""
    import torch
    Qh = wl.Q.cpu().pin_memory()
    Ch = torch.empty(wl.C.shape, dtype=torch.float32, pin_memory=True)
    for b0 in range(0, B_TOTAL, CHUNK):
        Ch[b0:b0 + CHUNK].copy_(wl.C[b0:b0 + CHUNK])
    outh = torch.empty((B_TOTAL, K), dtype=torch.float32, pin_memory=True)
    dQ = [torch.empty((CHUNK, D), device=dev) for _ in range(2)]
    dC = [torch.empty((CHUNK, K, D), device=dev) for _ in range(2)]
    dO = [torch.empty((CHUNK, K), device=dev) for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    loaded = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def one_step(score=True):
        n = B_TOTAL // CHUNK
        for i in range(n):
            j = i % 2
            b0 = i * CHUNK
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(freed[j])
                dQ[j].copy_(Qh[b0:b0 + CHUNK], non_blocking=True)
                dC[j].copy_(Ch[b0:b0 + CHUNK], non_blocking=True)
                loaded[j].record(copy)
            comp.wait_event(loaded[j])
            if score:
                cs.cs_score_candidates_batch(dQ[j], dC[j], wl.normalize, wl.scale, wl.temperature, out=dO[j],
                                             stream=comp)
                outh[b0:b0 + CHUNK].copy_(dO[j], non_blocking=True)
            freed[j].record(comp)
        comp.synchronize()

    h2d = (Qh.numel() + Ch.numel()) * 4
    d2h = outh.numel() * 4

    def timed(score):
        for _ in range(2):
            one_step(score)
        barrier()
        per = []
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            t = time.perf_counter()
            one_step(score)
            per.append(time.perf_counter() - t)
        barrier()
        return max_over_ranks(time.perf_counter() - t0), per

    dt, per = timed(True)
    ldt, lper = timed(False)
    numa = numa_placement(dev, {"C": (Ch.data_ptr(), (0, h2d // 2, Ch.numel() * 4 - 4096)),
                                "Q": (Qh.data_ptr(), (0,)), "out": (outh.data_ptr(), (0,))})
    del Ch, Qh, outh, dQ, dC, dO
    link_gbs = h2d * args.e2e_steps / ldt / 1e9
    e2e_gbs = h2d * args.e2e_steps / dt / 1e9
    return {"value": world * B_TOTAL * args.e2e_steps / dt, "unit": "questions/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "h2d_gbs": e2e_gbs,
            "step_h2d_gbs": [round(h2d / t / 1e9, 1) for t in per],
            "median_step_questions_per_s": world * B_TOTAL / statistics.median(per),
            "link_ceiling": {"what": "the same steps' host-to-device copies, no kernel and no read-back",
                             "h2d_gbs": link_gbs, "median_step_h2d_gbs": h2d / statistics.median(lper) / 1e9,
                             "step_h2d_gbs": [round(h2d / t / 1e9, 1) for t in lper]},
            "h2d_frac_of_link": e2e_gbs / link_gbs,
            "median_step_frac_of_link": statistics.median(lper) / statistics.median(per),
            "numa": numa}


if __name__ == "__main__":
    sys.exit(main())
