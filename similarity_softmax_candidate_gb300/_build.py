"""In-tree build of libcandidate_scoring.so for GB300 (sm_103a).

nvcc compiles the kernels and the C ABI into one shared library next to this
file. The build is skipped when the library is newer than every source.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sysconfig
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libcandidate_scoring.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
# Bounds-checked build of the same sources (-DCS_DEBUG_BOUNDS), for tests.
DEBUG_LIB_NAME = "libcandidate_scoring_debug.so"
DEBUG_LIB_PATH = os.path.join(PKG, DEBUG_LIB_NAME)
# Native latency harness (calls the C ABI from C++; see csrc/latency_main.cu).
LATENCY_NAME = "cs_latency"
LATENCY_PATH = os.path.join(PKG, LATENCY_NAME)
LATENCY_SRC = os.path.join(CSRC, "latency_main.cu")
# Read ceiling of the streaming access pattern (bulk copies, no arithmetic;
# see csrc/copy_ceiling_main.cu). Standalone: it does not link the library.
CEILING_NAME = "cs_copy_ceiling"
CEILING_PATH = os.path.join(PKG, CEILING_NAME)
CEILING_SRC = os.path.join(CSRC, "copy_ceiling_main.cu")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


# The binding's per-call marshalling in C (csrc/fastpath.c): a CPython
# extension module next to the package, built with the host C compiler
# against Python's headers. Optional: without it the binding marshals with
# ctypes alone.
FASTPATH_SRC = os.path.join(CSRC, "fastpath.c")
FASTPATH_PATH = os.path.join(PKG, "_fastpath" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def _sources():
    """Library sources: every .cu/.cpp in csrc except programs (*_main.cu)."""
    files = glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp"))
    return sorted(f for f in files if not f.endswith("_main.cu"))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: cannot build the CUDA library")


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile (if needed) and return the library path. Raises on failure.
    debug_bounds: the bounds-checked variant (DEBUG_LIB_PATH)."""
    path, name = (DEBUG_LIB_PATH, DEBUG_LIB_NAME) if debug_bounds else (LIB_PATH, LIB_NAME)
    if not debug_bounds:
        build_fastpath(force)
    if not force and not is_stale(path):
        return path
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", *ARCH_FLAGS, "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE, "-I", CSRC] + (["-DCS_DEBUG_BOUNDS"] if debug_bounds else [])
    with tempfile.TemporaryDirectory(prefix="cs_build_") as tmp:
        objs = []
        procs = []
        for src in _sources():
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [nvcc, *common, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd))
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
            objs.append(obj)
        for cmd, pr in procs:
            out, _ = pr.communicate()
            if pr.returncode != 0:
                raise RuntimeError(f"nvcc failed ({pr.returncode}): {' '.join(cmd)}\n{out.decode(errors='replace')}")
            if verbose and out:
                print(out.decode(errors="replace"))
        tmp_lib = os.path.join(tmp, name)
        link = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp_lib, *objs]
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout.decode(errors='replace')}")
        staged = path + f".tmp{os.getpid()}"
        shutil.copyfile(tmp_lib, staged)
        os.replace(staged, path)
    return path


def build_fastpath(force: bool = False):
    """Compile the binding's C marshalling module if it is missing or older
    than its source. Returns its path, or None when it cannot be built (no
    C compiler or no Python headers): the binding then uses ctypes alone."""
    if not force and os.path.exists(FASTPATH_PATH) and \
            os.path.getmtime(FASTPATH_PATH) >= os.path.getmtime(FASTPATH_SRC):
        return FASTPATH_PATH
    include = sysconfig.get_paths().get("include")
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc or not include or not os.path.exists(os.path.join(include, "Python.h")):
        return None
    staged = FASTPATH_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-O2", "-shared", "-fPIC", "-Wall", "-I", include, FASTPATH_SRC, "-o", staged],
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        if os.path.exists(staged):
            os.unlink(staged)
        return None
    os.replace(staged, FASTPATH_PATH)
    return FASTPATH_PATH


def _tool_jobs(force: bool):
    """(path, staged output, nvcc command) of each native tool that needs
    compiling: the latency harness (linked to the library, found at run time
    through an $ORIGIN rpath) and the copy-ceiling program."""
    jobs = []
    if force or not os.path.exists(LATENCY_PATH) or \
            os.path.getmtime(LATENCY_PATH) < max(os.path.getmtime(LATENCY_SRC), os.path.getmtime(LIB_PATH)):
        staged = LATENCY_PATH + f".tmp{os.getpid()}"
        jobs.append((LATENCY_PATH, staged,
                     [_nvcc(), "-O2", "-std=c++17", *ARCH_FLAGS, "-I", INCLUDE, LATENCY_SRC, "-o", staged, "-L",
                      PKG, "-lcandidate_scoring", "-Xlinker", "-rpath,$ORIGIN"]))
    if force or not os.path.exists(CEILING_PATH) or os.path.getmtime(CEILING_PATH) < os.path.getmtime(CEILING_SRC):
        staged = CEILING_PATH + f".tmp{os.getpid()}"
        jobs.append((CEILING_PATH, staged, [_nvcc(), "-O2", "-std=c++17", *ARCH_FLAGS, CEILING_SRC, "-o", staged]))
    return jobs


def build_tools(force: bool = False) -> None:
    """Compile the native tools next to the library, in parallel."""
    build_library()
    procs = [(path, staged, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT))
             for path, staged, cmd in _tool_jobs(force)]
    failed = []
    for path, staged, cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append(f"nvcc failed: {' '.join(cmd)}\n{out.decode(errors='replace')}")
        else:
            os.replace(staged, path)
    if failed:
        raise RuntimeError("\n".join(failed))


def build_latency_tool(force: bool = False) -> str:
    """The native latency harness (built with the other tools)."""
    build_tools(force)
    return LATENCY_PATH


def build_copy_ceiling_tool(force: bool = False) -> str:
    """The copy-ceiling program (built with the other tools)."""
    build_tools(force)
    return CEILING_PATH


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
    build_tools(force=True)
    print(LATENCY_PATH)
    print(CEILING_PATH)
