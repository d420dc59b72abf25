"""Thin Python binding of libcandidate_scoring.so (ctypes).

Argument marshalling only: every step of the readout runs in the library's
CUDA kernels. Function names match the C ABI in include/candidate_scoring.h.
Tensors must be float32, contiguous and on a CUDA device (a host buffer
passed as a device pointer faults the kernel, the first defect listed in
PR #69 "cuda: add a fused candidate-scoring kernel for CLM and Kev",
"Defects the GPU found, in order"; the binding refuses one up front).

The readout calls (cs_score_candidates[_batch][_bf16]) with an `out` given
marshal through a small C module (_fastpath, csrc/fastpath.c) when it was
built: the same checks and the same library call, for well under the ~4 us
ctypes takes per call. Anything it does not handle plainly falls back to the
ctypes path below, which raises the precise error.

If the library has not been built, every call raises: there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

CS_MAX_K = 255
CS_PLAN_AUTO, CS_PLAN_STREAM, CS_PLAN_CLUSTER, CS_PLAN_GENERIC, CS_PLAN_DIRECT = 0, 1, 2, 3, 4
PLAN_NAMES = {CS_PLAN_STREAM: "stream", CS_PLAN_CLUSTER: "cluster", CS_PLAN_GENERIC: "generic",
              CS_PLAN_DIRECT: "direct"}

STATUS = {
    0: "CS_OK", 1: "CS_ERR_NULL_POINTER", 2: "CS_ERR_K_ZERO", 3: "CS_ERR_K_TOO_LARGE",
    4: "CS_ERR_D_ZERO", 5: "CS_ERR_BAD_SCALE", 6: "CS_ERR_BAD_TEMPERATURE", 7: "CS_ERR_BAD_BATCH",
    8: "CS_ERR_BAD_SIMILARITY", 9: "CS_ERR_LAUNCH", 10: "CS_ERR_ALIAS", 11: "CS_ERR_TOO_LARGE",
    12: "CS_ERR_BAD_PLAN", 13: "CS_ERR_SCRATCH_TOO_SMALL", 14: "CS_ERR_RANGE", 15: "CS_ERR_MISALIGNED",
}
CS_NOALLOC_MAX_ROWS = 1 << 20
CS_PROJ_MAX_ROWS = (1 << 31) - 256
globals().update({name: code for code, name in STATUS.items()})

_lock = threading.Lock()
_lib = None
_debug_lib = None
# The C marshalling module (_fastpath, built from csrc/fastpath.c) once set
# up with the entry points of _fast_owner; False when it is unavailable.
_fast = None
_fast_owner = None
CS_DEVERR_BOUNDS = 8
CS_DEVERR_BAD_OFFSETS = 4
CS_DEVERR_RANGE = 16


class CSError(RuntimeError):
    """A nonzero cs_status from the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)} ({cs_status_string(self.status)})")


def library() -> ctypes.CDLL:
    """The loaded library with argument types declared. Raises RuntimeError
    if it has not been built (call ``_build.build_library()``)."""
    global _lib
    lib = _lib
    if lib is not None:  # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"{_build.LIB_NAME} is not built; run __graft_entry__.build() or "
                               "python -m similarity_softmax_candidate_gb300._build")
        _lib = _declare(ctypes.CDLL(_build.LIB_PATH))
        return _lib


def debug_library() -> ctypes.CDLL:
    """The bounds-checked build of the same library (compiled on first use,
    about half a minute). For tests: ``with using(debug_library()):`` routes
    this module's calls through it."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _declare(ctypes.CDLL(_build.build_library(debug_bounds=True)))
        return _debug_lib


class using:
    """Context manager: this module's calls go to `lib` (another build of
    the same ABI, e.g. debug_library()) until the block ends."""

    def __init__(self, lib):
        self.lib = lib

    def __enter__(self):
        global _lib
        library()
        with _lock:
            self.saved, _lib = _lib, self.lib
        return self.lib

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare argument and result types of every entry point of `lib`."""
    P, I, F, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.POINTER(ctypes.c_uint)
    IP = ctypes.POINTER(ctypes.c_int)
    lib.cs_abi_version.argtypes = []
    lib.cs_abi_version.restype = I
    lib.cs_status_string.argtypes = [I]
    lib.cs_status_string.restype = ctypes.c_char_p
    lib.cs_score_candidates.argtypes = [P, P, I, I, I, F, F, P, P]
    lib.cs_score_candidates.restype = I
    lib.cs_score_candidates_batch.argtypes = [P, P, I, I, I, I, F, F, P, P]
    lib.cs_score_candidates_batch.restype = I
    lib.cs_score_candidates_batch_plan.argtypes = [P, P, I, I, I, I, F, F, P, P, I, I, I]
    lib.cs_score_candidates_batch_plan.restype = I
    lib.cs_score_candidates_batch_unfused.argtypes = [P, P, I, I, I, I, F, F, P, P, P]
    lib.cs_score_candidates_batch_unfused.restype = I
    lib.cs_score_candidates_batch_unfused_noalloc.argtypes = [P, P, I, I, I, I, F, F, P, P]
    lib.cs_score_candidates_batch_unfused_noalloc.restype = I
    lib.cs_score_candidates_bf16.argtypes = [P, P, I, I, I, F, F, P, P]
    lib.cs_score_candidates_bf16.restype = I
    lib.cs_score_candidates_batch_bf16.argtypes = [P, P, I, I, I, I, F, F, P, P]
    lib.cs_score_candidates_batch_bf16.restype = I
    LL = ctypes.c_longlong
    lib.cs_score_candidates_ragged.argtypes = [P, P, P, I, LL, I, I, F, F, P, P]
    lib.cs_score_candidates_ragged.restype = I
    lib.cs_score_candidates_ragged_bf16.argtypes = [P, P, P, I, LL, I, I, F, F, P, P]
    lib.cs_score_candidates_ragged_bf16.restype = I
    lib.cs_query_plan.argtypes = [P, P, I, I, I, I, IP, IP, IP, IP]
    lib.cs_query_plan.restype = I
    LL2 = ctypes.c_longlong
    lib.cs_project_rows.argtypes = [P, P, LL2, I, I, P, P]
    lib.cs_project_rows.restype = I
    lib.cs_project_score_batch.argtypes = [P, P, P, P, I, I, I, I, I, F, F, P, P, P]
    lib.cs_project_score_batch.restype = I
    lib.cs_selftest_bounded_wait.argtypes = [I, P]
    lib.cs_selftest_bounded_wait.restype = I
    lib.cs_device_status.argtypes = [U, I]
    lib.cs_device_status.restype = I
    lib.cs_debug_bounds_build.argtypes = []
    lib.cs_debug_bounds_build.restype = I
    lib.cs_bounds_violation.argtypes = [U, I]
    lib.cs_bounds_violation.restype = I
    lib.cs_selftest_bounds.argtypes = [P]
    lib.cs_selftest_bounds.restype = I
    return lib


def _fastpath():
    """The C marshalling module set up for the library in use, or None
    (not built here, or another build of the library is in use)."""
    global _fast, _fast_owner
    lib = library()
    if _fast_owner is lib:
        return _fast
    if _fast is False:
        return None
    with _lock:
        if _fast is None:
            try:
                from . import _fastpath as fp
                import torch
                addr = [ctypes.cast(f, ctypes.c_void_p).value for f in
                        (lib.cs_score_candidates, lib.cs_score_candidates_batch, lib.cs_score_candidates_bf16,
                         lib.cs_score_candidates_batch_bf16)]
                fp.setup(*addr, torch.float32, torch.bfloat16, torch._C._cuda_getDevice,
                         torch._C._cuda_getCurrentRawStream)
                _fast, _fast_owner = fp, lib
            except Exception:  # no C compiler or Python headers where it was built, or an older torch
                _fast = False
        return _fast if _fast_owner is lib else None


def cs_abi_version() -> int:
    return int(library().cs_abi_version())


def cs_status_string(status: int) -> str:
    return library().cs_status_string(int(status)).decode()


def _check(t, name, ndim, dtype=None):
    import torch
    dtype = torch.float32 if dtype is None else dtype
    try:
        ok = t.is_cuda and t.dtype == dtype and t.dim() == ndim and t.is_contiguous()
    except AttributeError:
        raise TypeError(f"{name} must be a torch.Tensor") from None
    if not ok:
        if not t.is_cuda:
            raise ValueError(f"{name} must be on a CUDA device (host memory cannot be read by the kernel)")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if t.dim() != ndim:
            raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _current_raw_stream(device):
    """cudaStream_t of torch's current stream on `device`. torch's raw-stream
    accessor (the one Triton launches on) skips building a Stream object,
    ~2 us per call; the public API is the fallback."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(device.index if device.index is not None else torch.cuda.current_device())
    return torch.cuda.current_stream(device).cuda_stream


def _stream_handle(stream, device):
    if stream is None:
        return _current_raw_stream(device)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(fn, device, args, stream):
    """Call fn(*args, stream) with `device` current (the library launches on
    the current device); switches device only when it has to."""
    import torch
    if device.index == torch.cuda.current_device():
        return fn(*args, _stream_handle(stream, device))
    with torch.cuda.device(device):
        return fn(*args, _stream_handle(stream, device))


def cs_score_candidates(q, C, normalize: int, scale: float, temperature: float, out=None, stream=None):
    """One question: q[D], C[K,D] -> out[K] (float32, CUDA)."""
    if out is not None:
        fp = _fast if _fast_owner is _lib and _lib is not None else _fastpath()
        if fp:
            s = fp.score(q, C, out, normalize, scale, temperature, stream, False)
            if s is not None:
                if s != 0:
                    raise CSError(s, "cs_score_candidates")
                return out
    import torch
    qp = _check(q, "q", 1)
    cp = _check(C, "C", 2)
    K, D = int(C.shape[0]), int(C.shape[1])
    if q.shape[0] != D or q.device != C.device:
        raise ValueError(f"q {tuple(q.shape)} does not match C {tuple(C.shape)}")
    if out is None:
        out = torch.empty(K, device=C.device, dtype=torch.float32)
    op = _check(out, "out", 1)
    if out.shape[0] != K or out.device != C.device:
        raise ValueError(f"out must be [K={K}] on {C.device}")
    s = _call(library().cs_score_candidates, C.device,
              (qp, cp, K, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates")
    return out


def _batch_ptrs(Q, C, out, c_dtype=None):
    import torch
    qp = _check(Q, "Q", 2)
    cp = _check(C, "C", 3, c_dtype)
    B, K, D = (int(x) for x in C.shape)
    if tuple(Q.shape) != (B, D) or Q.device != C.device:
        raise ValueError(f"Q {tuple(Q.shape)} does not match C {tuple(C.shape)}")
    if out is None:
        out = torch.empty((B, K), device=C.device, dtype=torch.float32)
    op = _check(out, "out", 2)
    if tuple(out.shape) != (B, K) or out.device != C.device:
        raise ValueError(f"out must be [B={B}, K={K}] on {C.device}")
    return qp, cp, op, out, B, K, D


def cs_score_candidates_batch(Q, C, normalize: int, scale: float, temperature: float, out=None, stream=None):
    """B questions: Q[B,D], C[B,K,D] -> out[B,K] (float32, CUDA), one launch."""
    if out is not None:
        fp = _fast if _fast_owner is _lib and _lib is not None else _fastpath()
        if fp:
            s = fp.score_batch(Q, C, out, normalize, scale, temperature, stream, False)
            if s is not None:
                if s != 0:
                    raise CSError(s, "cs_score_candidates_batch")
                return out
    qp, cp, op, out, B, K, D = _batch_ptrs(Q, C, out)
    s = _call(library().cs_score_candidates_batch, C.device,
              (qp, cp, B, K, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_batch")
    return out


def cs_score_candidates_batch_plan(Q, C, normalize: int, scale: float, temperature: float, plan: int,
                                   cluster: int = 0, ctas: int = 0, out=None, stream=None):
    """cs_score_candidates_batch with a caller-chosen plan (tests, tuning)."""
    import torch
    qp, cp, op, out, B, K, D = _batch_ptrs(Q, C, out)
    lib = library()
    s = _call(lambda *a: lib.cs_score_candidates_batch_plan(*a, int(plan), int(cluster), int(ctas)), C.device,
              (qp, cp, B, K, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_batch_plan")
    return out


def cs_score_candidates_batch_unfused(Q, C, normalize: int, scale: float, temperature: float, staged=None,
                                      out=None, stream=None):
    """The unfused baseline (two launches): pass 1 stages one float per row
    in `staged` [B,K] (allocated here by torch when None), pass 2 scores from
    it. Same result as cs_score_candidates_batch within float32 rounding."""
    import torch
    qp, cp, op, out, B, K, D = _batch_ptrs(Q, C, out)
    if staged is None:
        staged = torch.empty((B, K), device=C.device, dtype=torch.float32)
    sp = _check(staged, "staged", 2)
    if tuple(staged.shape) != (B, K) or staged.device != C.device:
        raise ValueError(f"staged must be [B={B}, K={K}] on {C.device}")
    lib = library()
    s = _call(lambda *a: lib.cs_score_candidates_batch_unfused(*a[:8], sp, op, a[8]), C.device,
              (qp, cp, B, K, D, int(normalize), float(scale), float(temperature)), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_batch_unfused")
    return out


def cs_score_candidates_batch_unfused_noalloc(Q, C, normalize: int, scale: float, temperature: float, out,
                                              stream=None):
    """The unfused baseline with the library's built-in staged buffer, for
    callers that cannot allocate device memory: nothing is allocated here or
    in the library, so `out` [B,K] must be given. B*K <= CS_NOALLOC_MAX_ROWS;
    calls share the buffer, so calls overlapping on the GPU race."""
    if out is None:
        raise ValueError("out is required: this entry point allocates nothing")
    qp, cp, op, out, B, K, D = _batch_ptrs(Q, C, out)
    s = _call(library().cs_score_candidates_batch_unfused_noalloc, C.device,
              (qp, cp, B, K, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_batch_unfused_noalloc")
    return out


def cs_score_candidates_bf16(q, C, normalize: int, scale: float, temperature: float, out=None, stream=None):
    """One question with bfloat16 candidates: q[D] float32, C[K,D] bfloat16
    -> out[K] float32 (CUDA)."""
    import torch
    if out is not None and getattr(C, "dtype", None) == torch.bfloat16:
        fp = _fast if _fast_owner is _lib and _lib is not None else _fastpath()
        if fp:
            s = fp.score(q, C, out, normalize, scale, temperature, stream, True)
            if s is not None:
                if s != 0:
                    raise CSError(s, "cs_score_candidates_bf16")
                return out
    qp = _check(q, "q", 1)
    cp = _check(C, "C", 2, torch.bfloat16)
    K, D = int(C.shape[0]), int(C.shape[1])
    if q.shape[0] != D or q.device != C.device:
        raise ValueError(f"q {tuple(q.shape)} does not match C {tuple(C.shape)}")
    if out is None:
        out = torch.empty(K, device=C.device, dtype=torch.float32)
    op = _check(out, "out", 1)
    if out.shape[0] != K or out.device != C.device:
        raise ValueError(f"out must be [K={K}] on {C.device}")
    s = _call(library().cs_score_candidates_bf16, C.device,
              (qp, cp, K, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_bf16")
    return out


def cs_score_candidates_batch_bf16(Q, C, normalize: int, scale: float, temperature: float, out=None, stream=None):
    """B questions with bfloat16 candidates: Q[B,D] float32, C[B,K,D]
    bfloat16 -> out[B,K] float32 (CUDA), one launch."""
    import torch
    if out is not None and getattr(C, "dtype", None) == torch.bfloat16:
        fp = _fast if _fast_owner is _lib and _lib is not None else _fastpath()
        if fp:
            s = fp.score_batch(Q, C, out, normalize, scale, temperature, stream, True)
            if s is not None:
                if s != 0:
                    raise CSError(s, "cs_score_candidates_batch_bf16")
                return out
    qp, cp, op, out, B, K, D = _batch_ptrs(Q, C, out, torch.bfloat16)
    s = _call(library().cs_score_candidates_batch_bf16, C.device,
              (qp, cp, B, K, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_batch_bf16")
    return out


def cs_score_candidates_ragged(Q, C, offsets, normalize: int, scale: float, temperature: float, out=None,
                               stream=None):
    """Ragged batch: Q[B,D] float32, C[total_rows,D] (float32 or bfloat16),
    offsets[B+1] int64 on the device (question b owns rows
    offsets[b]..offsets[b+1]-1) -> out[total_rows] float32, one launch."""
    import torch
    qp = _check(Q, "Q", 2)
    bf16 = getattr(C, "dtype", None) == torch.bfloat16
    cp = _check(C, "C", 2, torch.bfloat16 if bf16 else torch.float32)
    op_ = _check(offsets, "offsets", 1, torch.int64)
    B, D = int(Q.shape[0]), int(Q.shape[1])
    total = int(C.shape[0])
    if int(C.shape[1]) != D or int(offsets.shape[0]) != B + 1 or Q.device != C.device or offsets.device != C.device:
        raise ValueError(f"shapes do not match: Q {tuple(Q.shape)}, C {tuple(C.shape)}, offsets {tuple(offsets.shape)}")
    if out is None:
        out = torch.empty(total, device=C.device, dtype=torch.float32)
    op = _check(out, "out", 1)
    if out.shape[0] != total or out.device != C.device:
        raise ValueError(f"out must be [total_rows={total}] on {C.device}")
    lib = library()
    fn = lib.cs_score_candidates_ragged_bf16 if bf16 else lib.cs_score_candidates_ragged
    s = _call(fn, C.device, (qp, cp, op_, B, total, D, int(normalize), float(scale), float(temperature), op), stream)
    if s != 0:
        raise CSError(s, "cs_score_candidates_ragged")
    return out


def cs_project_rows(H, W, out=None, stream=None):
    """P = H W^T on the tensor cores: H [rows, Din] and W [D, Din] bfloat16
    (CUDA) -> P [rows, D] float32. D in {256, 512}, Din a multiple of 64."""
    import torch
    hp = _check(H, "H", 2, torch.bfloat16)
    wp = _check(W, "W", 2, torch.bfloat16)
    rows, Din = (int(x) for x in H.shape)
    D = int(W.shape[0])
    if int(W.shape[1]) != Din or W.device != H.device:
        raise ValueError(f"W {tuple(W.shape)} does not match H {tuple(H.shape)}")
    if out is None:
        out = torch.empty((rows, D), device=H.device, dtype=torch.float32)
    op = _check(out, "out", 2)
    if tuple(out.shape) != (rows, D):
        raise ValueError(f"out must be [{rows}, {D}]")
    s = _call(library().cs_project_rows, H.device, (hp, wp, rows, Din, D, op), stream)
    if s != 0:
        raise CSError(s, "cs_project_rows")
    return out


def cs_project_score_batch(Hq, Wq, Hc, Wc, normalize: int, scale: float, temperature: float, qproj=None, out=None,
                           stream=None):
    """Projected readout: q_b = Wq hq_b, c_bk = Wc hc_bk (bfloat16 features
    and weights, float32 accumulation on the tensor cores), scored as
    cs_score_candidates_batch; the projected candidates stay on chip.
    Hq [B, Din], Hc [B, K, Din], Wq and Wc [D, Din] -> out [B, K]; qproj
    [B, D] float32 receives the projected queries."""
    import torch
    bf = torch.bfloat16
    hq, wq, hc, wc = (_check(Hq, "Hq", 2, bf), _check(Wq, "Wq", 2, bf), _check(Hc, "Hc", 3, bf),
                      _check(Wc, "Wc", 2, bf))
    B, K, Din = (int(x) for x in Hc.shape)
    D = int(Wc.shape[0])
    if tuple(Hq.shape) != (B, Din) or tuple(Wq.shape) != (D, Din) or tuple(Wc.shape) != (D, Din):
        raise ValueError("shapes do not match: Hq [B, Din], Hc [B, K, Din], Wq and Wc [D, Din]")
    if qproj is None:
        qproj = torch.empty((B, D), device=Hc.device, dtype=torch.float32)
    if out is None:
        out = torch.empty((B, K), device=Hc.device, dtype=torch.float32)
    qp = _check(qproj, "qproj", 2)
    op = _check(out, "out", 2)
    lib = library()
    s = _call(lambda *a: lib.cs_project_score_batch(*a[:11], qp, op, a[11]), Hc.device,
              (hq, wq, hc, wc, B, K, Din, D, int(normalize), float(scale), float(temperature)), stream)
    if s != 0:
        raise CSError(s, "cs_project_score_batch")
    return out


def cs_query_plan(Q, C, normalize: int) -> dict:
    """The automatic plan for these tensors: kind, cluster, ctas, smem_bytes."""
    import torch
    qp = _check(Q, "Q", 2)
    cp = _check(C, "C", 3)
    B, K, D = (int(x) for x in C.shape)
    vals = [ctypes.c_int(0) for _ in range(4)]
    with torch.cuda.device(C.device):
        s = library().cs_query_plan(qp, cp, B, K, D, int(normalize), *[ctypes.byref(v) for v in vals])
    if s != 0:
        raise CSError(s, "cs_query_plan")
    kind, cluster, ctas, smem = (v.value for v in vals)
    return {"plan": PLAN_NAMES.get(kind, kind), "kind": kind, "cluster": cluster, "ctas": ctas,
            "smem_bytes": smem}


def cs_device_status(clear: bool = False) -> int:
    """The device status word of the current device (synchronizes)."""
    v = ctypes.c_uint(0)
    s = library().cs_device_status(ctypes.byref(v), int(bool(clear)))
    if s != 0:
        raise CSError(s, "cs_device_status")
    return int(v.value)


def cs_debug_bounds_build() -> bool:
    """True when the library in use is the bounds-checked build."""
    return bool(library().cs_debug_bounds_build())


def cs_bounds_violation(clear: bool = False) -> int:
    """Site number of the first failed bounds check (0: none; bounds-checked
    builds only record any). Synchronizes."""
    v = ctypes.c_uint(0)
    s = library().cs_bounds_violation(ctypes.byref(v), int(bool(clear)))
    if s != 0:
        raise CSError(s, "cs_bounds_violation")
    return int(v.value)


def cs_selftest_bounds(stream=None) -> None:
    """Bounds-checked builds: record site 99 from a check of a range one
    past a buffer's end (nothing is accessed)."""
    import torch
    s = _call(library().cs_selftest_bounds, torch.device("cuda", torch.cuda.current_device()), (), stream)
    if s != 0:
        raise CSError(s, "cs_selftest_bounds")
