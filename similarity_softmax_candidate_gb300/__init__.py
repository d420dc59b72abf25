"""Fused candidate scoring on GB300 (sm_103a).

Per question, a query q[D] and up to 255 candidates C[K,D] become softmax
probabilities over the candidates, scored by scale * cosine (CLM) or
scale * dot (Kev) over a temperature, with the similarities kept on chip
(PR #69 "cuda: add a fused candidate-scoring kernel for CLM and Kev").

The work runs in the C-ABI library libcandidate_scoring.so (hand-written
CUDA; header include/candidate_scoring.h). This package holds its in-tree
build (``_build``), the thin ctypes binding (``binding``) and seeded input
generators (``workloads``).
"""
from .binding import (  # noqa: F401
    CS_MAX_K,
    CS_PLAN_AUTO,
    CS_PLAN_CLUSTER,
    CS_PLAN_DIRECT,
    CS_PLAN_GENERIC,
    CS_PLAN_STREAM,
    CSError,
    cs_abi_version,
    cs_bounds_violation,
    cs_debug_bounds_build,
    cs_device_status,
    cs_project_rows,
    cs_project_score_batch,
    cs_query_plan,
    cs_score_candidates,
    cs_score_candidates_bf16,
    cs_score_candidates_batch,
    cs_score_candidates_batch_bf16,
    cs_score_candidates_batch_plan,
    cs_score_candidates_batch_unfused,
    cs_score_candidates_batch_unfused_noalloc,
    cs_score_candidates_ragged,
    cs_selftest_bounds,
    cs_status_string,
    debug_library,
    library,
    using,
)
