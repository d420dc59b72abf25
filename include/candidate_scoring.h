/*
 * candidate_scoring.h -- C ABI of the GB300 (sm_103a) fused candidate-scoring
 * library, libcandidate_scoring.so.
 *
 * The operation (PR #69 "cuda: add a fused candidate-scoring kernel for CLM
 * and Kev"; its opening table gives the two similarities and "What is fused,
 * precisely" the fusion): for each question b, given a query q_b[D] and K
 * candidates C_b[K,D],
 *
 *   sim_k = cos(q_b, c_k)   normalize = 1  (CLM; each norm clamped at 1e-8)
 *   sim_k = c_k . q_b       normalize = 0  (Kev)
 *   z_k   = scale * sim_k / temperature
 *   p_k   = exp(z_k - max_j z_j) / sum_j exp(z_j - max_j z_j)
 *
 * and only p is written: the similarities never reach global memory, and each
 * candidate row is read from memory once (its dot with q and its squared norm
 * come from the same load).
 *
 * Conventions shared by every entry point below:
 *   - All array pointers are CUDA DEVICE pointers to float32 data the caller
 *     owns (cudaMalloc, or a torch CUDA tensor). Host pointers are not
 *     detected; passing one is undefined (the kernel faults). Each pointer
 *     must be aligned to its element (4 bytes; 2 for bfloat16 candidates);
 *     CS_ERR_MISALIGNED otherwise. Any offset from a 16-byte boundary is
 *     fine: rows that do not start on one, or whose length is not a multiple
 *     of 16 bytes, are copied as the aligned span around them (the bytes of
 *     the same 16-byte granules, never used).
 *   - Layout is dense row-major: Q is [B][D], C is [B][K][D], out is [B][K].
 *     out must not overlap Q or C. Inputs are only read.
 *   - The work is queued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream). Calls are asynchronous: they never synchronize,
 *     allocate, free or memset, and one call enqueues exactly one kernel, so
 *     it captures into a CUDA graph as one node (PR #69, "Through a CUDA
 *     Graph" and "Verified on hardware").
 *   - The first call on a device does one-time set-up (kernel attributes and
 *     an occupancy query, and the device addresses of the library's own
 *     status words) and caches it for the life of the process; make one
 *     ordinary call per device before starting a stream capture. The cache
 *     does not survive cudaDeviceReset: do not use the library on a device
 *     after resetting it in the same process.
 *   - Invalid arguments return a nonzero status BEFORE any CUDA call: nothing
 *     is launched and out is untouched (PR #69, "Verified on hardware", the
 *     rejected-arguments group). A failed launch returns CS_ERR_LAUNCH.
 *     Faults inside the kernel surface, as usual in CUDA, at the caller's
 *     next synchronizing call.
 *   - Results are deterministic: the same call on the same device gives
 *     bit-identical output, directly or replayed from a graph.
 *   - Range. Every finite input within the range below gets a probability
 *     distribution, never NaN. The logit factor scale / temperature is
 *     formed in double precision; a factor with |scale / temperature| >
 *     2^126 (about 8.5e37; e.g. scale 14.3 at temperature 1e-37) is refused
 *     with CS_ERR_RANGE before any CUDA call -- the exact softmax of such
 *     logits is an argmax that float32 similarities cannot settle. The
 *     logits enter the softmax only as differences from their maximum,
 *     formed so that a huge factor drives them to -inf (probability exactly
 *     0) and never to NaN, and a factor below float32's range scores every
 *     candidate alike, as the exact softmax does to within far less than
 *     1e-4. Dots, squared norms and |q|^2
 *     accumulate in float32, so they must stay within FLT_MAX: for the dot
 *     |c| |q| <= FLT_MAX is enough, for the cosine |c| and |q| below about
 *     1.8e19 (every element below 1.8e19 / sqrt(D) is enough); tiny rows
 *     need nothing, since their norms are clamped at 1e-8 before float32
 *     loses them. A question outside that range, or with a NaN or
 *     infinite element, is skipped: its rows of out are left unwritten and
 *     CS_DEVERR_RANGE is set in the device status word (cs_device_status).
 *     The page's rule is the same: an error rather than a scored answer
 *     (PR #69, "Verified on hardware", rejected arguments).
 */
#ifndef CANDIDATE_SCORING_H
#define CANDIDATE_SCORING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *cs_stream_t;

/* Largest number of candidates per question. The softmax runs over an
 * on-chip array of this many logits; a larger K is refused rather than
 * truncated (PR #69, "Verified on hardware": scoring only the first 255
 * would give a confident wrong answer). */
#define CS_MAX_K 255

typedef enum {
    CS_OK = 0,
    CS_ERR_NULL_POINTER = 1,   /* Q, C or out is NULL */
    CS_ERR_K_ZERO = 2,         /* K <= 0: no candidates */
    CS_ERR_K_TOO_LARGE = 3,    /* K > CS_MAX_K */
    CS_ERR_D_ZERO = 4,         /* D <= 0 */
    CS_ERR_BAD_SCALE = 5,      /* scale == 0, NaN or infinite */
    CS_ERR_BAD_TEMPERATURE = 6,/* temperature <= 0, NaN or infinite */
    CS_ERR_BAD_BATCH = 7,      /* B <= 0 */
    CS_ERR_BAD_SIMILARITY = 8, /* normalize is neither 0 nor 1 */
    CS_ERR_LAUNCH = 9,         /* a CUDA call failed; nothing useful was queued */
    CS_ERR_ALIAS = 10,         /* out overlaps Q or C */
    CS_ERR_TOO_LARGE = 11,     /* B*K*D elements do not fit the 64-bit index space */
    CS_ERR_BAD_PLAN = 12,      /* cs_score_candidates_batch_plan: plan not feasible */
    CS_ERR_SCRATCH_TOO_SMALL = 13,/* B*K above CS_NOALLOC_MAX_ROWS (no-allocation entry) */
    CS_ERR_RANGE = 14,         /* |scale / temperature| exceeds 2^126 (about 8.5e37) */
    CS_ERR_MISALIGNED = 15     /* a pointer is not aligned to its element size */
} cs_status;

/* ABI version of this header and library: 1. The page's manifest records
 * the kernel's ABI as version 1 (PR #69, "The manifest, and CI":
 * abi_version 1); a caller can check it before binding the entry points.
 * Takes no arguments, touches no device, cannot fail. */
int cs_abi_version(void);

/* Static English text for a status code (never NULL; "unknown status" for
 * a code this library does not return). An addition of this library: the
 * page names the rejected arguments but no way to print them. Touches no
 * device, cannot fail. */
const char *cs_status_string(int status);

/*
 * One question: q[D], C[K][D] -> out[K]. The page's single-question call
 * (PR #69, "Verified on hardware": its batch group scores one question
 * through this call and more through cs_score_candidates_batch, so the two
 * entry points must agree); here it is cs_score_candidates_batch with B = 1.
 *   normalize   1 = cosine (CLM), 0 = dot (Kev)
 *   scale       multiplies the similarity; for CLM pass exp(logit_scale),
 *               for Kev 1/sqrt(256). Any finite nonzero value.
 *   temperature divides the scaled similarity; finite and > 0.
 */
int cs_score_candidates(const float *q, const float *C, int K, int D,
                        int normalize, float scale, float temperature,
                        float *out, cs_stream_t stream);

/*
 * B questions in one launch (a grid over questions, not a loop of launches;
 * PR #69, "What is fused, precisely"): Q[B][D], C[B][K][D] -> out[B][K].
 * K is the same for every question. Arguments as cs_score_candidates.
 */
int cs_score_candidates_batch(const float *Q, const float *C, int B, int K,
                              int D, int normalize, float scale,
                              float temperature, float *out,
                              cs_stream_t stream);

/*
 * The same readouts with the candidates stored as bfloat16 (C holds the
 * 16-bit patterns, [B][K][D] row-major), half the bytes of the float32
 * layout on a path whose time is the reading of C. Each element is widened
 * exactly to float32 and accumulated in float32, so the result is the
 * float32 readout of the bfloat16-rounded candidates. q and out stay
 * float32. Rows with D % 8 != 0 or off a 16-byte boundary stream as
 * aligned spans like float32 ones (a few such questions take the scalar
 * plan). Arguments, errors and conventions as
 * cs_score_candidates / cs_score_candidates_batch. (bfloat16 storage is our
 * extension; the page's kernel reads float32.)
 */
int cs_score_candidates_bf16(const float *q, const uint16_t *C, int K, int D,
                             int normalize, float scale, float temperature,
                             float *out, cs_stream_t stream);
int cs_score_candidates_batch_bf16(const float *Q, const uint16_t *C, int B,
                                   int K, int D, int normalize, float scale,
                                   float temperature, float *out,
                                   cs_stream_t stream);

/*
 * Ragged batches: question b has its own K_b candidates (1 <= K_b <= 255).
 * C holds all candidate rows back to back, [total_rows][D] (float32, or
 * bfloat16 bit patterns for the _bf16 form); question b owns rows
 * offsets[b] .. offsets[b+1]-1, and out [total_rows] receives its
 * probabilities at the same rows. offsets is a DEVICE array of B+1 int64
 * with offsets[0] = 0 and offsets[B] = total_rows; Q is [B][D] as before.
 * One launch, as cs_score_candidates_batch (work is split by rows, not by
 * questions, so mixed K_b stays balanced).
 * The host cannot read offsets without synchronizing, so it checks only
 * what it is given (B >= 1, B <= total_rows <= 255*B, pointers, scalars,
 * overlaps of out with Q, C and offsets -- the usual status codes). Each
 * question's own offsets are checked by the kernel: a question with K_b
 * outside [1, 255] or rows outside [0, total_rows) is skipped (its rows of
 * out are not written) and CS_DEVERR_BAD_OFFSETS is set in the device status
 * word (cs_device_status). The ragged layout is our extension; the page's
 * call takes one K for the whole batch.
 */
int cs_score_candidates_ragged(const float *Q, const float *C,
                               const long long *offsets, int B,
                               long long total_rows, int D, int normalize,
                               float scale, float temperature, float *out,
                               cs_stream_t stream);
int cs_score_candidates_ragged_bf16(const float *Q, const uint16_t *C,
                                    const long long *offsets, int B,
                                    long long total_rows, int D, int normalize,
                                    float scale, float temperature, float *out,
                                    cs_stream_t stream);

/*
 * Caller-side projections on the tensor cores (the page leaves them to the
 * caller: CLM scores state_head(s) against action_head(c), Kev k(h_opts)
 * against q(h_decide)). Features and weights are bfloat16 bit patterns,
 * row-major; accumulation is float32.
 *
 * cs_project_rows: P[r][n] = sum_i H[r][i] * W[n][i] for H [rows][Din],
 *   W [D][Din], P [rows][D] float32.
 * cs_project_score_batch: q_b = Wq hq_b (written to qproj [B][D] float32,
 *   a caller-owned buffer), then for each question the projected candidates
 *   c_bk = Wc hc_bk (Hc [B][K][Din]) are scored against q_b exactly as
 *   cs_score_candidates_batch scores C -- without the projected candidates
 *   ever being written to memory: they exist only in tensor memory.
 *   Two kernels are enqueued on `stream`.
 * Shapes: D = 256 or 512, Din a multiple of 64, 1 <= K <= 255; all pointers
 * 16-byte aligned (CS_ERR_BAD_PLAN otherwise); at most CS_PROJ_MAX_ROWS rows
 * (rows, or B*K; tensor-copy coordinates are 32-bit; CS_ERR_BAD_BATCH
 * otherwise). Other errors and conventions as cs_score_candidates_batch.
 * This is our extension of the page's kernel.
 */
#define CS_PROJ_MAX_ROWS 2147483392LL /* 2^31 - 256 */
int cs_project_rows(const uint16_t *H, const uint16_t *W, long long rows,
                    int Din, int D, float *P, cs_stream_t stream);
int cs_project_score_batch(const uint16_t *Hq, const uint16_t *Wq,
                           const uint16_t *Hc, const uint16_t *Wc, int B,
                           int K, int Din, int D, int normalize, float scale,
                           float temperature, float *qproj, float *out,
                           cs_stream_t stream);

/* Execution plans (kernel choices) the library picks between. */
#define CS_PLAN_AUTO 0
#define CS_PLAN_STREAM 1   /* persistent CTAs, each streams a run of questions
                              (bulk copies; unaligned rows as aligned spans) */
#define CS_PLAN_CLUSTER 2  /* one thread-block cluster per question, rows split */
#define CS_PLAN_GENERIC 3  /* scalar loads; any D, any alignment (one CTA per
                              question, or a cluster of CTAs per question
                              when a uniform-K batch has few questions):
                              rows too long for the shared-memory ring */
#define CS_PLAN_DIRECT 4   /* one CTA (or cluster) per short question: at most 32
                              rows per CTA (16 for long rows), q and rows
                              loaded straight into registers, no
                              shared-memory ring */

/*
 * The plan cs_score_candidates_batch would use for these arguments.
 * Arguments are validated exactly as there (status on failure). On CS_OK,
 * every non-NULL output pointer receives: plan (CS_PLAN_*), cluster (CTAs
 * per cluster, 1 = none), ctas (CTAs launched), smem_bytes (dynamic shared
 * memory per CTA). Needs a CUDA device (it queries the current one).
 */
int cs_query_plan(const float *Q, const float *C, int B, int K, int D,
                  int normalize, int *plan, int *cluster, int *ctas,
                  int *smem_bytes);

/*
 * cs_score_candidates_batch with the plan chosen by the caller, for tests
 * and tuning. plan is CS_PLAN_*; cluster (CS_PLAN_CLUSTER and
 * CS_PLAN_DIRECT: 1..16, at most K) and ctas (CS_PLAN_STREAM: 1..B) may be 0
 * for the automatic choice. CS_PLAN_DIRECT also needs ceil(K / cluster) <=
 * 32 for D <= 512 and ceil(K / cluster) <= 16 for 512 < D <= 2560; rows
 * that do not start on 16-byte boundaries or whose length is not a
 * multiple of 16 bytes only up to D = 512 (read in 4-byte units). For
 * CS_PLAN_GENERIC, cluster 0 or 1 means one CTA per question and 2..16 (at
 * most K) spreads each question's rows over a cluster of that many CTAs.
 * Returns CS_ERR_BAD_PLAN when the plan cannot run these arguments (e.g.
 * CS_PLAN_DIRECT on rows longer than its forms take, or a ring that does
 * not fit shared memory for CS_PLAN_STREAM/CLUSTER; these two take
 * unaligned rows as aligned spans). The result equals the automatic plan's
 * within float32 rounding.
 */
int cs_score_candidates_batch_plan(const float *Q, const float *C, int B,
                                   int K, int D, int normalize, float scale,
                                   float temperature, float *out,
                                   cs_stream_t stream, int plan, int cluster,
                                   int ctas);

/*
 * The unfused baseline, for comparison with the fused readout (PR #69,
 * "What it is worth": a separate norm pass plus the scoring block with the
 * row norm loaded from a staged array, reading C twice; for the dot, whose
 * similarity has no norm to fuse, the same split costs a second kernel and a
 * global round trip of the similarities, "What is fused, precisely").
 *   pass 1: staged[b][k] = |c_bk| (cosine) or c_bk . q_b (dot)
 *   pass 2: cosine: the scoring kernel again, dots recomputed from C, norms
 *           read from staged; dot: softmax of scale * staged / temperature.
 * Same arguments and result as cs_score_candidates_batch (within float32
 * rounding), plus `staged`: a caller-owned device buffer of B*K floats that
 * must not overlap Q, C or out; its contents on return are pass 1's values.
 * Two kernels are enqueued on `stream` (two graph nodes when captured).
 * Needs D % 4 == 0 and 16-byte aligned Q and C (CS_ERR_BAD_PLAN otherwise:
 * the baseline's passes have no unaligned build).
 */
int cs_score_candidates_batch_unfused(const float *Q, const float *C, int B,
                                      int K, int D, int normalize, float scale,
                                      float temperature, float *staged,
                                      float *out, cs_stream_t stream);

/*
 * cs_score_candidates_batch_unfused without the `staged` argument: the
 * staged array is a buffer built into the library, so the call allocates
 * nothing and needs no scratch from the caller. The page has no counterpart
 * of this entry point; it serves callers that cannot call cudaMalloc -- code
 * running under a host framework that owns all device memory through its
 * own pool and forbids raw allocations, or latency-critical code that cannot
 * afford cudaMalloc's implicit device-wide synchronization.
 *   - B*K must not exceed CS_NOALLOC_MAX_ROWS (CS_ERR_SCRATCH_TOO_SMALL
 *     otherwise, before any CUDA call).
 *   - The buffer takes 4 MiB of device memory on every GPU that loads the
 *     library, until the process exits.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress) and caches it for the life of the process.
 *   - Every call shares the one buffer and leaves its own pass-1 values in
 *     it. Nothing in it needs to start at zero (pass 1 writes every row that
 *     pass 2 reads), but calls that overlap on the GPU -- e.g. on two streams
 *     at once -- race on it: serialize them.
 * Other arguments, requirements and results as cs_score_candidates_batch_unfused.
 */
#define CS_NOALLOC_MAX_ROWS 1048576
int cs_score_candidates_batch_unfused_noalloc(const float *Q, const float *C,
                                              int B, int K, int D,
                                              int normalize, float scale,
                                              float temperature, float *out,
                                              cs_stream_t stream);

/* Device status word bits (see cs_device_status). */
#define CS_DEVERR_WAIT_TIMEOUT 1u  /* an on-chip wait gave up after ~1 s */
#define CS_DEVERR_BAD_CONFIG 2u    /* a kernel refused an inconsistent launch plan */
#define CS_DEVERR_BAD_OFFSETS 4u   /* a ragged question had invalid offsets and was skipped */
#define CS_DEVERR_BOUNDS 8u        /* bounds-checked build: an access outside its buffer was skipped */
#define CS_DEVERR_RANGE 16u        /* a question's dots or norms left float32's range (or an input was
                                      NaN or infinite): it was skipped, its rows of out unwritten */

/*
 * Reads (and, if clear != 0, resets) the status word the kernels of this
 * library set on the current device when one of their bounded waits gives
 * up, skips a question it cannot score (CS_DEVERR_*). A kernel that gives
 * up stops early; the results it could not finish are left NaN or
 * unwritten. Synchronizes the device; not for the hot path.
 */
int cs_device_status(unsigned *flags, int clear);

/*
 * Self-test of the kernels' bounded waits: enqueues one tiny kernel whose
 * single thread waits, with the same wait routine the scoring kernels use,
 * on an on-chip barrier nothing will complete. After limit_us microseconds
 * (1 .. 1000000; CS_ERR_BAD_PLAN otherwise) it gives up, sets
 * CS_DEVERR_WAIT_TIMEOUT in the device status word and exits, leaving the
 * context usable. For tests and health checks: it shows that a wait that
 * never completes ends in a status, not a hang.
 */
int cs_selftest_bounded_wait(int limit_us, cs_stream_t stream);

/*
 * Bounds-checked builds. The library can also be compiled with
 * -DCS_DEBUG_BOUNDS (libcandidate_scoring_debug.so, built on demand by the
 * tests; same entry points). There, before every global-memory access a
 * kernel makes -- rows of C and q copied into shared memory, probabilities,
 * staged values, ragged offsets, projected queries -- the range is checked
 * against the extent of its buffer (from the call's arguments); a failing
 * check skips the access, sets CS_DEVERR_BOUNDS in the device status word
 * and records its site number (first failure only). It stands in for a
 * memory checker and has no counterpart on the page. Release builds compile
 * the checks away.
 *
 * cs_debug_bounds_build: 1 in a bounds-checked build, 0 otherwise.
 * cs_bounds_violation: reads (and, if clear != 0, resets) the recorded site
 *   number, 0 when no check has failed; synchronizes the device.
 * cs_selftest_bounds: enqueues one tiny kernel that checks a range one past
 *   the end of a buffer (arithmetic only, nothing is read or written), so
 *   that site 99 is recorded; CS_ERR_BAD_PLAN in a release build.
 */
int cs_debug_bounds_build(void);
int cs_bounds_violation(unsigned *site, int clear);
int cs_selftest_bounds(cs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CANDIDATE_SCORING_H */
