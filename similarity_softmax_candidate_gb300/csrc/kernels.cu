// Fused candidate-scoring kernels for GB300 (sm_103a).
//
// Operation (PR #69 "cuda: add a fused candidate-scoring kernel for CLM and
// Kev", opening table and "What is fused, precisely"): per question b,
//   z_k = scale * sim(q_b, c_k) / temperature,  p = softmax_k(z)
// with sim the cosine (each norm clamped at 1e-8) or the plain dot. Each
// candidate row is read once: its dot with q and its squared norm accumulate
// from the same registers. Per-row results live only in shared memory.
//
// GB300 design (the page's kernel was one 1024-thread block per question on
// sm_89; of that only "softmax over shared memory" is kept):
//   * stream_kernel -- a warp-specialised CTA: eight lanes of a producer
//     warp issue 1-D bulk copies (cp.async.bulk, TMA engine) of whole
//     candidate rows into a ring of shared-memory stages tracked by
//     mbarriers, a second producer warp the query rows. Stage g (up to 8
//     rows) is issued by lane g % 8 and belongs to consumer warp g % 8 --
//     eight independent pipelines per CTA -- which computes the dots and
//     squared norms of all its rows from float4 shared loads against q held
//     in registers, then reduces them together with one transposed butterfly
//     of warp shuffles. The per-row cosine and the softmax run later, one
//     lane per row, in the warp that finishes the question.
//       - STREAM plan: persistent, one CTA per SM, each CTA streams a
//         contiguous run of questions, prefetching the next question while a
//         single warp finishes the previous question's softmax.
//       - CLUSTER plan: one thread-block cluster (up to 16 CTAs) per
//         question, the K rows split over the CTAs; each CTA reduces its rows
//         to (local max, local sum of exp) and pushes the pair into every
//         peer's shared memory with st.async, completing on the peer's
//         mbarrier, so one question uses up to 16 SMs.
//     Dots and norms accumulate as packed float32 pairs (fma.rn.f32x2);
//     plans of at most 2 rows per stage run a short-stage build. Rows that
//     do not start on 16-byte boundaries (or whose length is not a multiple
//     of 16 bytes) are copied as the aligned span around them and read from
//     shared memory in 4-byte units (stage_dots_units).
//   * direct_kernel -- DIRECT plan, one or a few short questions: one CTA or
//     cluster per question, at most 32 rows per CTA (16 for long rows), q
//     and the rows loaded straight into registers (q in shared memory for
//     long rows; unaligned rows as 4-byte units), one trip to memory, the
//     same cluster exchange.
//   * generic_kernel -- scalar loads, any D and any alignment: one CTA per
//     question, or, for a few questions of a uniform batch, one cluster per
//     question with the same exchange as the DIRECT plan.
// The stream and direct kernels are launched with programmatic dependent
// launch: they may start while the previous kernel runs and wait for it
// (griddepcontrol.wait) before their first global access. Before that wait
// a stream-kernel CTA only asks L2 for its first ring's worth of rows (a
// prefetch changes no value anyone reads).
//   * the unfused baseline (PR #69, "What it is worth": a separate norm pass
//     and a scoring block that loads the norm from a staged array) reuses
//     stream_kernel: pass 1 writes one value per row (the norm, or for the dot
//     the similarity) to a staged array in global memory; pass 2 is the
//     scoring block reading the staged norms (cosine) or staged_softmax_kernel
//     (dot).
// Logits enter the softmax in a range-safe form (softmax_form.cuh): no
// finite input gives NaN, and a question whose sums leave float32's range
// is skipped with a device status bit instead of being scored.
// Every on-chip wait is bounded (about 1 s); a CTA that gives up sets a
// device status bit, leaves what it could not finish NaN or unwritten,
// waits (bounded) for its own copies in flight, and exits.
#include "internal.h"
#include "softmax_form.cuh"

#include <math.h>

#include <mutex>
#include <type_traits>

namespace cs {

__device__ unsigned int g_status;
__device__ unsigned int g_bounds_site;  // bounds-checked builds: first failing site (0 = none)

namespace {

#ifdef CS_DEBUG_BOUNDS
// [ptr, ptr + bytes) inside [base, base + extent)? Otherwise record the site
// (first one only) and the status bit, and tell the caller to skip.
__device__ __noinline__ bool check_range(const void* ptr, unsigned long long bytes, const void* base,
                                         unsigned long long extent, unsigned site) {
    const unsigned long long a = reinterpret_cast<unsigned long long>(ptr);
    const unsigned long long b = reinterpret_cast<unsigned long long>(base);
    if (a >= b && bytes <= extent && a - b <= extent - bytes) return true;
    atomicCAS(&g_bounds_site, 0u, site);
    atomicOr(&g_status, kDevErrBounds);
    return false;
}
#define CS_IN_BOUNDS(ptr, bytes, base, extent, site) \
    check_range((ptr), static_cast<unsigned long long>(bytes), (base), static_cast<unsigned long long>(extent), (site))
#else
#define CS_IN_BOUNDS(ptr, bytes, base, extent, site) true
#endif

// Rows of C (and of out, and of staged) of a launch.
[[maybe_unused]] __host__ __device__ inline long long rows_total(const Problem& p) {
    return p.offsets ? p.total_rows : p.B * static_cast<long long>(p.K);
}

using form::qnan;
using form::softmax_term;
using form::value_scale;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s
constexpr int kSlotsPerLane = kLogitSlots / 32;

// What a StreamMode accumulates per row and what it finishes with.
__host__ __device__ constexpr bool acc_norm(int m) { return m == kFusedCos || m == kRowNorm; }  // c . c
__host__ __device__ constexpr bool acc_dot(int m) { return m != kRowNorm; }                     // c . q
__host__ __device__ constexpr int values_per_row(int m) { return acc_norm(m) && acc_dot(m) ? 2 : 1; }
__host__ __device__ constexpr bool does_softmax(int m) { return m == kFusedCos || m == kFusedDot || m == kStagedCos; }
__host__ __device__ constexpr bool cos_logits(int m) { return m == kFusedCos || m == kStagedCos; }

// Elements of C. The streaming kernel moves rows as 16-byte chunks: 4
// float32 or 8 bfloat16 (stored as their 16-bit patterns). A chunk widens to
// QF4 float4s, matched against the same number of float4s of q.
template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kPerChunk = 4;
    static constexpr int kQF4 = 1;
    __device__ __forceinline__ static void widen(const uint4& c, float4 (&f)[1]) {
        f[0] = make_float4(__uint_as_float(c.x), __uint_as_float(c.y), __uint_as_float(c.z), __uint_as_float(c.w));
    }
    __device__ __forceinline__ static float value(const float* row, int d) { return __ldg(row + d); }
    __device__ __forceinline__ static float widen1(float x) { return x; }
};
template <>
struct Elem<uint16_t> {  // bfloat16: the high half of a float32
    static constexpr int kPerChunk = 8;
    static constexpr int kQF4 = 2;
    __device__ __forceinline__ static void widen(const uint4& c, float4 (&f)[2]) {
        f[0] = make_float4(__uint_as_float(c.x << 16), __uint_as_float(c.x & 0xffff0000u), __uint_as_float(c.y << 16),
                           __uint_as_float(c.y & 0xffff0000u));
        f[1] = make_float4(__uint_as_float(c.z << 16), __uint_as_float(c.z & 0xffff0000u), __uint_as_float(c.w << 16),
                           __uint_as_float(c.w & 0xffff0000u));
    }
    __device__ __forceinline__ static float value(const uint16_t* row, int d) {
        return __uint_as_float(static_cast<uint32_t>(__ldg(row + d)) << 16);
    }
    __device__ __forceinline__ static float widen1(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }
};

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes`
// transactions on `bar`. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Hint: fetch `bytes` (a multiple of 16, src 16-byte aligned) of global
// memory into L2. It changes no value anyone reads (L2 is where global
// memory is coherent), so it may be issued before the previous kernel's
// writes are visible.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Programmatic dependent launch. The kernels are launched so that they may
// start while the previous kernel in the stream is still running; before
// its first global-memory access each thread waits until that kernel has
// completed and its writes are visible (so inputs it produced are read
// intact), and each CTA at once lets the next launch be scheduled.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Arrive without ordering this thread's memory operations: the cluster
// barrier phases here publish nothing but the mbarrier initialisation
// (already ordered by fence.mbarrier_init.release.cluster) or only keep CTAs
// alive until every push into them has landed (which their own mbarrier
// wait has seen).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    return remote;
}

// Store a float2 into a peer CTA's shared memory; the 8 bytes complete as
// transactions on the peer's mbarrier.
__device__ __forceinline__ void st_async_peer(uint32_t remote_dst, float2 v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                     remote_dst),
                 "f"(v.x), "f"(v.y), "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ void consumer_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

// ------------------------------------------------------------------ helpers

// Packed float32 pairs (low = first element): d = a * b + c element-wise,
// one instruction for two fused multiply-adds.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
// The two halves of a packed pair.
__device__ __forceinline__ float2 unpack2(unsigned long long x) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
    return make_float2(lo, hi);
}
// The two halves of a packed pair, added: the value its partial sums make.
__device__ __forceinline__ float sum2(unsigned long long x) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
    return lo + hi;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Bounded wait on an mbarrier phase. Returns false if this CTA has given up
// (now or earlier); the first thread to hit the limit raises the CTA's flag
// and the device status bit.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* give_up,
                                           unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*give_up) return false;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*give_up) return false;
        if ((it & 31u) == 0 && globaltimer() - t0 > limit_ns) {
            *give_up = 1;
            atomicOr(&g_status, 1u);
            return false;
        }
    }
}

// Wait until a deadline regardless of the give-up flag (used to let copies
// in flight land before the CTA exits after giving up).
__device__ __forceinline__ void wait_phase_until(uint32_t bar, uint32_t parity, unsigned long long deadline) {
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() > deadline) return;
    }
}

// ------------------------------------------------------------------ range-safe softmax
//
// Rows become values v_k (softmax_form.cuh): the probabilities are
// 2^(kexp (v_k - max v)) normalised, which no finite input turns into NaN,
// and a row float32 could not hold has the value NaN. NaN carries into the
// question's sum of exponentials (the max ignores it), and a question whose
// sum is NaN is skipped unscored.

// v of one row from its dot t and, for the fused cosine, its squared norm
// nsq (the staged cosine passes the staged norm instead).
template <int MODE>
__device__ __forceinline__ float row_value(float t, float nsq, float w) {
    if (MODE == kFusedCos) return form::cos_value(t, nsq, w);
    if (MODE == kStagedCos) return form::staged_cos_value(t, nsq, w);
    return form::dot_value(t, w);
}

// Values of rows lane, lane+32, ... (< n) from their dots t and, for the
// fused cosine, squared norms n_sq, or, for the staged cosine, norms read
// from the staged array; -inf beyond n.
template <int MODE, int S = kSlotsPerLane>
__device__ __forceinline__ void load_values(const float* t, const float* n_sq, const float* staged_norm, int n,
                                            float w, int lane, float (&v)[S]) {
#pragma unroll
    for (int j = 0; j < S; ++j) {
        const int k = lane + 32 * j;
        v[j] = -INFINITY;
        if (k < n)
            v[j] = row_value<MODE>(t[k], MODE == kFusedCos ? n_sq[k] : MODE == kStagedCos ? staged_norm[k] : 0.f, w);
    }
}

// One warp's rows (lane + 32 j < n) reduced to the max of their values
// (flagged rows ignored) and, in v, their exponentials relative to it;
// returns the warp's sum of those, NaN when a row is flagged.
template <int S>
__device__ __forceinline__ float exp_rows(float (&v)[S], int n, float kexp, int lane, float* m_out) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < S; ++j) m = fmaxf(m, v[j]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < S; ++j) {
        v[j] = lane + 32 * j < n ? softmax_term(kexp, v[j] - m) : 0.f;
        s += v[j];
    }
    *m_out = m;
    return warp_sum(s);
}

// Softmax over one warp (rows lane + 32 j < n) of the values v, written to
// dst[0..n). Returns false, writing nothing, when a row is flagged; the
// caller then records the range bit (unless its CTA gave up waiting, which
// is what flagged the rows).
template <int S = kSlotsPerLane>
__device__ __forceinline__ bool softmax_store(float (&v)[S], int n, float kexp, float* __restrict__ dst, int lane) {
    float m;
    const float s = exp_rows(v, n, kexp, lane, &m);
    if (isnan(s)) return false;
    const float inv = 1.0f / s;
#pragma unroll
    for (int j = 0; j < S; ++j) {
        const int k = lane + 32 * j;
        if (k < n) dst[k] = v[j] * inv;
    }
    return true;
}

// A question's rows were flagged: record it, unless this CTA gave up
// waiting (the status word already says so, and that is what flagged them).
__device__ __forceinline__ void record_range(volatile int* give_up) {
    if (!*give_up) atomicOr(&g_status, kDevErrRange);
}

// Cluster exchange: each CTA reduces its rows to (m, s) = (max v, sum of
// 2^(kexp (v - m))), s NaN when it holds a flagged row, and every CTA of
// the cluster then skips the question. combine_pairs reads the G pairs in
// xch (lanes < G one each) and returns the normaliser
// 1 / sum_g s_g 2^(kexp (m_g - M)) with M = max m_g (M_out); flagged: some
// CTA sent NaN. A CTA without rows sends (-inf, 0) and adds nothing.
__device__ __forceinline__ float combine_pairs(const float2* xch, int G, float kexp, int lane, float* M_out,
                                               bool* flagged) {
    float mj = -INFINITY, sj = 0.f;
    if (lane < G) {
        const float2 x = xch[lane];
        mj = x.x;
        sj = x.y;
    }
    *flagged = __any_sync(0xffffffffu, isnan(sj));
    const float M = warp_max(mj);
    *M_out = M;
    return 1.0f / warp_sum(sj > 0.f ? sj * softmax_term(kexp, mj - M) : 0.f);
}

// Sums each of the V values v[0..V) over the 32 lanes of a warp with V - 1
// + (5 - log2 V) shuffles: at each butterfly level a lane keeps half of its
// values and receives the matching half from its partner, so the values are
// spread over the lanes instead of every lane reducing all of them. Returns
// the full sum of value *idx; every lane whose low (5 - log2 V) bits are zero
// holds a distinct value.
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&v)[V], int lane, int* idx) {
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
    int id = 0;
#pragma unroll
    for (int h = V / 2, o = 16; h >= 1; h >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? v[i] : v[i + h];
            const float keep = upper ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (upper) id += h;
    }
    float x = v[0];
#pragma unroll
    for (int o = 16 / V; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    *idx = id;
    return x;
}

// ------------------------------------------------------------------ questions and rows

constexpr int kMaxK = 255;

// The rows of question b this CTA handles (CTA `rank` of G on the question):
// row0 is the index in C (and in out) of the first, n how many. A ragged
// question whose offsets are out of range -- K_b outside [1, 255], or rows
// outside [0, total_rows) -- gets n = 0 and bad = true: it is skipped, and
// nothing outside the buffers is ever read or written.
struct QRows {
    long long row0;
    int n;
    bool bad;
};

__device__ __forceinline__ QRows question_rows(const Problem& p, long long b, int rank, int G) {
    long long o0 = b * p.K, kb = p.K;
    bool bad = false;
    if (p.offsets) {
        if (!CS_IN_BOUNDS(p.offsets + b, 16, p.offsets, (p.B + 1) * 8, kSiteOffsets)) return QRows{0, 0, true};
        o0 = p.offsets[b];
        const long long o1 = p.offsets[b + 1];
        kb = o1 - o0;
        if (!(o0 >= 0 && kb >= 1 && kb <= kMaxK && o1 <= p.total_rows)) {
            o0 = 0;
            kb = 0;
            bad = true;
        }
    }
    const int k = static_cast<int>(kb);
    const int lo = rank * k / G, hi = (rank + 1) * k / G;
    return QRows{o0 + lo, hi - lo, bad};
}

// First index b in [0, n] with off[b] >= target, position n counting as
// satisfied without being read; off must be non-decreasing for the answer to
// mean anything, but every read stays in [0, n) whatever it holds. One warp
// probes 32 positions per round, so n = 16384 takes three dependent rounds.
__device__ long long lower_bound_warp(const long long* off, long long n, long long target, int lane) {
    long long lo = 0, hi = n;  // the answer lies in [lo, hi]; hi always satisfies
    for (;;) {
        const long long span = hi - lo;
        const long long step = span <= 31 ? 1 : (span + 30) / 31;  // lo + 31 step >= hi
        long long pos = lo + step * lane;
        if (pos > hi) pos = hi;
        const bool ge = pos == n || !CS_IN_BOUNDS(off + pos, 8, off, (n + 1) * 8, kSiteOffsetsSearch) ||
                        off[pos] >= target;
        const unsigned m = __ballot_sync(0xffffffffu, ge);
        const int f = __ffs(m) - 1;  // m != 0: the lanes at hi satisfy
        long long pf = lo + step * f;
        if (pf > hi) pf = hi;
        if (f == 0 || step == 1) return pf;
        lo = lo + step * (f - 1) + 1;
        hi = pf;
    }
}

// ------------------------------------------------------------------ stream kernel

struct StreamArgs {
    Problem p;
    int rows_per_stage;  // R <= the instantiation's MR
    int stages;          // NS, a multiple of kConsumerWarps
    int cluster;         // G: CTAs per question (1 = STREAM plan)
    int q_per_cta;       // STREAM plan: CTA c takes q_per_cta (+1 if c < q_rem) questions
    int q_rem;
};

// Per-row sums of the nr <= MR rows of one stage (rows of DC
// 16-byte chunks each). Lane handles chunks lane, lane+32, ...; q comes from
// registers (NQC > 0: qv holds the q float4s of those chunks) or from shared
// memory (NQC == 0, large D). With two values per row (fused cosine)
// v[2r] = c_r . q and v[2r + 1] = c_r . c_r; with one, v[r] = c_r . q, or
// c_r . c_r for the norm pass. release() is called once, as soon as the
// stage's shared memory is no longer needed: for the modes that accumulate
// norms (twice the arithmetic of a dot), when the stage fits in registers
// (q in registers and at most kEarlyReleaseChunks 16-byte chunks per lane),
// every row is loaded first, so the slot goes back to the producer before
// the arithmetic; otherwise after the last row.
constexpr int kEarlyReleaseChunks = 16;  // 64 registers of staged rows at most

template <int NQC, int MODE, typename T, int MR, typename Release>
__device__ __forceinline__ void stage_dots(const uint4* __restrict__ st, int nr, int DC,
                                           const float4 (&qv)[(NQC > 0 ? NQC : 1) * Elem<T>::kQF4],
                                           const float4* __restrict__ q4, int lane,
                                           float (&v)[values_per_row(MODE) * MR], Release&& release) {
    constexpr int VPR = values_per_row(MODE);
    constexpr int QF4 = Elem<T>::kQF4;
    // Each value accumulates as two partial sums (even and odd elements of
    // the row) with packed float32 FMAs, added together at the end.
    unsigned long long acc[VPR * MR];
#pragma unroll
    for (int i = 0; i < VPR * MR; ++i) acc[i] = 0ull;
    auto accumulate = [&](const float4& c, const float4& q, int r) {
        const unsigned long long c01 = pack2(c.x, c.y), c23 = pack2(c.z, c.w);
        if (acc_dot(MODE)) {
            unsigned long long& t = acc[VPR * r];
            t = fma2(c01, pack2(q.x, q.y), t);
            t = fma2(c23, pack2(q.z, q.w), t);
        }
        if (acc_norm(MODE)) {
            unsigned long long& n = acc[VPR * r + VPR - 1];
            n = fma2(c01, c01, n);
            n = fma2(c23, c23, n);
        }
    };
    if constexpr (NQC > 0 && MR * NQC <= kEarlyReleaseChunks && acc_norm(MODE)) {
        uint4 cr[MR][NQC];
#pragma unroll
        for (int r = 0; r < MR; ++r)
#pragma unroll
            for (int j = 0; j < NQC; ++j) {
                const int i = lane + 32 * j;
                cr[r][j] = r < nr && i < DC ? st[r * DC + i] : make_uint4(0u, 0u, 0u, 0u);
            }
        release();
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            if (r < nr) {
#pragma unroll
                for (int j = 0; j < NQC; ++j) {
                    const int i = lane + 32 * j;
                    if (i < DC) {
                        float4 c[QF4];
                        Elem<T>::widen(cr[r][j], c);
#pragma unroll
                        for (int h = 0; h < QF4; ++h) accumulate(c[h], qv[j * QF4 + h], r);
                    }
                }
            }
        }
    } else if constexpr (NQC > 0 && std::is_same<T, float>::value) {
        // float32: chunks outer, the stage's rows inner (1.4 % more
        // throughput than rows outer for the cosine and the dot)
#pragma unroll
        for (int j = 0; j < NQC; ++j) {
            const int i = lane + 32 * j;
            if (i < DC) {
#pragma unroll
                for (int r = 0; r < MR; ++r) {
                    if (r < nr) {
                        float4 c[QF4];
                        Elem<T>::widen(st[r * DC + i], c);
#pragma unroll
                        for (int h = 0; h < QF4; ++h) accumulate(c[h], qv[j * QF4 + h], r);
                    }
                }
            }
        }
        release();
    } else if constexpr (NQC > 0) {
        // bfloat16: rows outer (chunks outer was 0.9 % slower for the dot)
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            if (r < nr) {
                const uint4* __restrict__ row = st + r * DC;
#pragma unroll
                for (int j = 0; j < NQC; ++j) {
                    const int i = lane + 32 * j;
                    if (i < DC) {
                        float4 c[QF4];
                        Elem<T>::widen(row[i], c);
#pragma unroll
                        for (int h = 0; h < QF4; ++h) accumulate(c[h], qv[j * QF4 + h], r);
                    }
                }
            }
        }
        release();
    } else {
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            if (r < nr) {
                const uint4* __restrict__ row = st + r * DC;
                for (int i = lane; i < DC; i += 32) {
                    float4 q[QF4];
#pragma unroll
                    for (int h = 0; h < QF4; ++h) q[h] = q4[i * QF4 + h];
                    float4 c[QF4];
                    Elem<T>::widen(row[i], c);
#pragma unroll
                    for (int h = 0; h < QF4; ++h) accumulate(c[h], q[h], r);
                }
            }
        }
        release();
    }
#pragma unroll
    for (int i = 0; i < VPR * MR; ++i) v[i] = sum2(acc[i]);
}

// Packed q of the unaligned plans with q in registers (unaligned_units(NQC)
// = NU > 0): NU / 2 pairs a lane for float32 (elements lane + 64 u and
// lane + 64 u + 32), NU for bfloat16 (elements 2k and 2k + 1, k = lane + 32 u;
// or 2k - 1 and 2k for rows read from the word before them, see
// stage_dots_units).
template <typename T, int NU>
struct UnitQ {
    static constexpr int kPairs = NU == 0 ? 1 : (std::is_same<T, float>::value ? NU / 2 : NU);
};

// bfloat16 rows of an even D whose first element is the high half of a
// 4-byte word (C on an odd 2-byte boundary): every row of the launch then
// starts so, and is read from that word on -- unit k holds elements 2k - 1
// and 2k -- against q shifted by one element; element -1 (another row's, or
// bytes of the span) is masked and element D - 1 added apart.
__device__ __forceinline__ bool bf16_rows_from_word_before(const void* C, int D) {
    return !(D & 1) && ((reinterpret_cast<unsigned long long>(C) >> 1) & 1u);
}

// The same sums for a stage whose rows sit at any element-aligned offset in
// their slot, read in 4-byte units with q in registers (qpk, UnitQ): lane
// takes units lane, lane + 32, ... of each row -- float32 elements, or
// bfloat16 pairs -- so consecutive lanes read consecutive words of shared
// memory. Except for the float32 cosine (row by row), the words of RG rows
// at a time are loaded before any arithmetic (all the stage's rows for
// NU <= 8) and the slot is released after the last loads (group sizes and
// orders as measured fastest on 4096 x 255 x 510 and on 4096 x 255 x 512 off
// by one element). Units past the row's end read as zero (for NU > 4 a
// lane's first NU / 2 units are always inside it: the plan picks NU so).
// bfloat16: rows of an even D all start at the parity of C; on an odd
// 2-byte boundary they are read from the word before
// (bf16_rows_from_word_before). Rows of an odd D alternate: a row on an odd
// boundary takes each pair from two words (the high half of one, the low
// half of the next). Either way an element past the last whole unit --
// element D - 1 -- is added by lane 0 (qlast its q). st: the slot, shift:
// the stage's first row's byte offset in it.
template <int NU, int MODE, typename T, int MR, typename Release>
__device__ __forceinline__ void stage_dots_units(const unsigned char* __restrict__ st, uint32_t shift, int nr, int D,
                                                 bool from_word_before,
                                                 const unsigned long long (&qpk)[UnitQ<T, NU>::kPairs], float qlast,
                                                 int lane, float (&v)[values_per_row(MODE) * MR], Release&& release) {
    constexpr int VPR = values_per_row(MODE);
    constexpr int GV = NU > 4 ? NU / 2 : 0;               // units always inside the row
    constexpr int RG = MR * NU <= 64 ? MR : 64 / NU;      // rows loaded at a time
    static_assert(MR % RG == 0, "row groups must tile the stage");
    unsigned long long acc[VPR * MR];
#pragma unroll
    for (int i = 0; i < VPR * MR; ++i) acc[i] = 0ull;
    auto accumulate = [&](unsigned long long c, unsigned long long qq, int r) {
        if (acc_dot(MODE)) acc[VPR * r] = fma2(c, qq, acc[VPR * r]);
        if (acc_norm(MODE)) acc[VPR * r + VPR - 1] = fma2(c, c, acc[VPR * r + VPR - 1]);
    };
    if constexpr (std::is_same<T, float>::value && !acc_norm(MODE)) {
        // float32 dot: a group's rows loaded first (1-2 % faster than row by row)
        const float* __restrict__ base = reinterpret_cast<const float*>(st + shift);
#pragma unroll
        for (int g = 0; g < MR; g += RG) {
            float c[RG][NU];
#pragma unroll
            for (int i = 0; i < RG; ++i) {
                const float* __restrict__ row = base + (g + i) * D;
#pragma unroll
                for (int u = 0; u < NU; ++u) {
                    const int k = lane + 32 * u;
                    c[i][u] = g + i < nr && (u < GV || k < D) ? row[k] : 0.f;
                }
            }
            if (g + RG >= MR) release();
#pragma unroll
            for (int i = 0; i < RG; ++i)
                if (g + i < nr) {
#pragma unroll
                    for (int u = 0; u < NU / 2; ++u) accumulate(pack2(c[i][2 * u], c[i][2 * u + 1]), qpk[u], g + i);
                }
        }
    } else if constexpr (std::is_same<T, float>::value) {
        // float32 cosine: row by row (loading a group's rows first measured
        // 2 % slower)
        const float* __restrict__ base = reinterpret_cast<const float*>(st + shift);
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            if (r < nr) {
                const float* __restrict__ row = base + r * D;
#pragma unroll
                for (int u = 0; u < NU / 2; ++u) {
                    const int k0 = lane + 64 * u, k1 = k0 + 32;
                    const float c0 = 2 * u < GV || k0 < D ? row[k0] : 0.f;
                    const float c1 = 2 * u + 1 < GV || k1 < D ? row[k1] : 0.f;
                    accumulate(pack2(c0, c1), qpk[u], r);
                }
            }
        }
        release();
    } else {
        const uint32_t* __restrict__ words = reinterpret_cast<const uint32_t*>(st);
        const uint16_t* __restrict__ halves = reinterpret_cast<const uint16_t*>(st);
        const int np = D >> 1;
        const uint32_t hb0 = shift >> 1;  // 2-byte index of the stage's element 0
        if (!(D & 1)) {
#pragma unroll
            for (int g = 0; g < MR; g += RG) {
                uint32_t w[RG][NU];
                uint16_t tail[RG];
#pragma unroll
                for (int i = 0; i < RG; ++i) {
                    const uint32_t hb = hb0 + static_cast<uint32_t>((g + i) * D);
                    const uint32_t* __restrict__ row = words + (hb >> 1);
#pragma unroll
                    for (int u = 0; u < NU; ++u) {
                        const int k = lane + 32 * u;
                        w[i][u] = g + i < nr && (u < GV || k < np) ? row[k] : 0u;
                    }
                    if (from_word_before && lane == 0) w[i][0] &= 0xffff0000u;  // element -1
                    tail[i] = from_word_before && lane == 0 && g + i < nr ? halves[hb + D - 1] : uint16_t(0);
                }
                if (g + RG >= MR) release();
                auto widened = [&](uint32_t x) {
                    return pack2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
                };
                if constexpr (acc_norm(MODE)) {
                    // cosine: units outer, every row of the group inner (rows a
                    // short stage lacks hold zeros), so that consecutive packed
                    // FMAs feed different rows' sums: 0.87 -> 0.97 of the aligned
                    // rate, against 2 % less for the dot
#pragma unroll
                    for (int u = 0; u < NU; ++u)
#pragma unroll
                        for (int i = 0; i < RG; ++i) accumulate(widened(w[i][u]), qpk[u], g + i);
                } else {
#pragma unroll
                    for (int i = 0; i < RG; ++i)
                        if (g + i < nr) {
#pragma unroll
                            for (int u = 0; u < NU; ++u) accumulate(widened(w[i][u]), qpk[u], g + i);
                        }
                }
                if (from_word_before) {
#pragma unroll
                    for (int i = 0; i < RG; ++i)
                        accumulate(pack2(Elem<uint16_t>::widen1(tail[i]), 0.f), pack2(qlast, 0.f), g + i);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                if (r < nr) {
                    const uint32_t hb = hb0 + static_cast<uint32_t>(r * D);
                    const uint32_t* __restrict__ row = words + (hb >> 1);
                    if (hb & 1u) {
#pragma unroll
                        for (int u = 0; u < NU; ++u) {
                            const int k = lane + 32 * u;
                            const bool in = u < GV || k < np;
                            const uint32_t a = in ? row[k] : 0u, b = in ? row[k + 1] : 0u;
                            accumulate(pack2(__uint_as_float(a & 0xffff0000u), __uint_as_float(b << 16)), qpk[u], r);
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < NU; ++u) {
                            const int k = lane + 32 * u;
                            const uint32_t x = u < GV || k < np ? row[k] : 0u;
                            accumulate(pack2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u)), qpk[u], r);
                        }
                    }
                    const uint16_t e = lane == 0 ? halves[hb + D - 1] : uint16_t(0);
                    accumulate(pack2(Elem<uint16_t>::widen1(e), 0.f), pack2(qlast, 0.f), r);
                }
            }
            release();
        }
    }
#pragma unroll
    for (int i = 0; i < VPR * MR; ++i) v[i] = sum2(acc[i]);
}

// stage_dots_units for rows too long for q in registers (the plan's
// kNqcUnaligned, any D): the same 4-byte units and the same bfloat16 forms,
// q read from shared memory (qf: q at its offset in the q slot). Such rows
// are long and their stages short (16 KB of rows: 1 to 7 rows), so the rows
// are taken one at a time -- nothing is spent on rows a short stage lacks --
// in blocks of kUnitBlock units a lane, all of a block's loads before its
// arithmetic; q is read again for each row.
constexpr int kUnitBlock = 8;

template <int MODE, typename T, int MR, typename Release>
__device__ __forceinline__ void stage_dots_units_shared_q(const unsigned char* __restrict__ st, uint32_t shift,
                                                          int nr, int D, bool from_word_before,
                                                          const float* __restrict__ qf, float qlast, int lane,
                                                          float (&v)[values_per_row(MODE) * MR], Release&& release) {
    constexpr int VPR = values_per_row(MODE);
    constexpr int NB = kUnitBlock;
#pragma unroll
    for (int i = 0; i < VPR * MR; ++i) v[i] = 0.f;
    const uint32_t* __restrict__ words = reinterpret_cast<const uint32_t*>(st);
    const uint16_t* __restrict__ halves = reinterpret_cast<const uint16_t*>(st);
    const int np = D >> 1;
    const int sh = from_word_before ? 1 : 0;  // bfloat16 q pairs (2k - sh, 2k + 1 - sh)
    for (int r = 0; r < nr; ++r) {
        unsigned long long dot = 0ull, nrm = 0ull;
        auto accumulate = [&](unsigned long long c, unsigned long long qq) {
            if (acc_dot(MODE)) dot = fma2(c, qq, dot);
            if (acc_norm(MODE)) nrm = fma2(c, c, nrm);
        };
        const uint32_t hb = (shift >> 1) + static_cast<uint32_t>(r * D);  // bfloat16: 2-byte index of element 0
        if constexpr (std::is_same<T, float>::value) {
            const float* __restrict__ row = reinterpret_cast<const float*>(st + shift) + r * D;
            for (int k0 = lane; k0 - lane < D; k0 += 32 * NB) {
                float c[NB], q[NB];
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const bool in = k0 + 32 * j < D;
                    c[j] = in ? row[k0 + 32 * j] : 0.f;
                    q[j] = in ? qf[k0 + 32 * j] : 0.f;
                }
#pragma unroll
                for (int j = 0; j < NB; j += 2) accumulate(pack2(c[j], c[j + 1]), pack2(q[j], q[j + 1]));
            }
        } else {
            const uint32_t* __restrict__ row = words + (hb >> 1);
            // an odd 2-byte start takes each pair from two words, unless every
            // row is read from the word before (even D, from_word_before)
            // q's pairs as one 8-byte read when they sit on 8-byte boundaries
            // (two 4-byte reads of every other word take twice the wavefronts)
            auto pairs = [&](auto split_tag, auto q8_tag) {
                constexpr bool SPLIT = decltype(split_tag)::value;
                constexpr bool Q8 = decltype(q8_tag)::value;
                for (int k0 = lane; k0 - lane < np; k0 += 32 * NB) {
                    uint32_t x[NB], y[NB];
                    float qa[NB], qb[NB];
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        const int k = k0 + 32 * j, e = 2 * k - sh;
                        const bool in = k < np;
                        x[j] = in ? row[k] : 0u;
                        if (SPLIT) y[j] = in ? row[k + 1] : 0u;
                        if (Q8) {
                            const float2 qq = in ? *reinterpret_cast<const float2*>(qf + e) : make_float2(0.f, 0.f);
                            qa[j] = e >= 0 ? qq.x : 0.f;
                            qb[j] = qq.y;
                        } else {
                            qa[j] = in && e >= 0 ? qf[e] : 0.f;
                            qb[j] = in ? qf[e + 1] : 0.f;
                        }
                    }
                    if (from_word_before && k0 == 0) x[0] &= 0xffff0000u;  // element -1
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        const float lo = __uint_as_float(SPLIT ? x[j] & 0xffff0000u : x[j] << 16);
                        const float hi = __uint_as_float(SPLIT ? y[j] << 16 : x[j] & 0xffff0000u);
                        accumulate(pack2(lo, hi), pack2(qa[j], qb[j]));
                    }
                }
            };
            const bool q8 = ((reinterpret_cast<unsigned long long>(qf) - 4u * sh) & 7u) == 0;
            const bool split = (hb & 1u) && !from_word_before;
            if (split)
                q8 ? pairs(std::true_type{}, std::true_type{}) : pairs(std::true_type{}, std::false_type{});
            else
                q8 ? pairs(std::false_type{}, std::true_type{}) : pairs(std::false_type{}, std::false_type{});
            if ((D & 1) || from_word_before) {
                const uint16_t e = lane == 0 ? halves[hb + D - 1] : uint16_t(0);
                accumulate(pack2(Elem<uint16_t>::widen1(e), 0.f), pack2(qlast, 0.f));
            }
        }
        // row r's partial sums into their static places for the reduction
#pragma unroll
        for (int i = 0; i < MR; ++i)
            if (i == r) {
                if (acc_dot(MODE)) v[VPR * i] = sum2(dot);
                if (acc_norm(MODE)) v[VPR * i + VPR - 1] = sum2(nrm);
            }
    }
    release();
}

// Global address of `bytes` bytes at src, widened to whole 16-byte granules
// for a bulk copy: returns the aligned start and sets *shift (the offset of
// src in it) and *span (the copy's length, a multiple of 16).
__device__ __forceinline__ const void* aligned_span(const void* src, uint32_t bytes, uint32_t* shift,
                                                    uint32_t* span) {
    const unsigned long long a = reinterpret_cast<unsigned long long>(src);
    *shift = static_cast<uint32_t>(a & 15u);
    *span = (*shift + bytes + 15u) & ~15u;
    return reinterpret_cast<const void*>(a & ~15ull);
}

// MR: most rows per stage this instantiation handles (kMaxRowsPerStage, or
// kSmallStageRows for the fused modes when the plan's stages are that short:
// the per-stage code a batch-1 launch fetches is then a quarter as long).
template <int NQC, int MODE, typename T, int MR>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(const StreamArgs args) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int VPR = values_per_row(MODE);
    constexpr int V = VPR * MR;
    constexpr bool COS = cos_logits(MODE);
    constexpr int QF4 = Elem<T>::kQF4;
    const Problem& p = args.p;
    const int D = p.D;
    const int DC = D / Elem<T>::kPerChunk;  // 16-byte chunks per row of C
    const T* Cg = static_cast<const T*>(p.C);
    const int R = args.rows_per_stage, NS = args.stages, G = args.cluster;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The ring must hold whole rounds of consumer warps (slot s is always
    // owned by warp s % kConsumerWarps) and a stage at most MR
    // rows; the host plans it so. Every CTA sees the same arguments, so a bad
    // plan makes every CTA of every cluster leave here, before any barrier.
    if (NS < kConsumerWarps || NS % kConsumerWarps != 0 || R < 1 || R > MR || G < 1 ||
        G > kMaxCluster) {
        if (threadIdx.x == 0) atomicOr(&g_status, 2u);
        return;
    }

    // UA: rows and queries need not start on 16-byte boundaries; each copy
    // takes their aligned span and readers index from the offset in it
    // (NU > 0: rows read in 4-byte units, q in registers).
    constexpr bool UA = NQC < 0;
    constexpr int NU = unaligned_units(NQC);
    const bool from_word_before = !std::is_same<T, float>::value && bf16_rows_from_word_before(p.C, D);
    const SmemLayout L = smem_layout(NS, R, D, static_cast<int>(sizeof(T)), UA);
    unsigned char* ring = smem + L.ring;
    const uint32_t slot_bytes = static_cast<uint32_t>(L.slot_bytes);
    unsigned char* qbuf = smem + L.qbuf;
    const uint32_t qslot_bytes = static_cast<uint32_t>(L.qslot_bytes);
    float* tn = reinterpret_cast<float*>(smem + L.tn);
    float2* xch = reinterpret_cast<float2*>(smem + L.xch);
    volatile int* give_up = reinterpret_cast<volatile int*>(smem + L.flag);
    long long* range = reinterpret_cast<long long*>(smem + L.range);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8u * NS;
    const uint32_t qfull0 = empty0 + 8u * NS;
    const uint32_t qempty0 = qfull0 + 16u;
    uint64_t* xbar = bars + 2 * NS + 4;

    // Barrier set-up by warp 0: full[s] completes once per use of slot s
    // (the producer's arrival plus the copy's bytes), empty[s] once its owner
    // warp is done with it; qfull/qempty per q slot; xbar when every CTA of
    // the cluster has pushed its (max, sum) here.
    if (warp == 0) {
        const int nbars = 2 * NS + 5;
        for (int i = lane; i < nbars; i += 32) {
            const uint32_t count = (i >= 2 * NS + 2 && i < 2 * NS + 4) ? kConsumerWarps : 1u;
            mbar_init(full0 + 8u * i, count);
        }
        if (lane == 0) *give_up = 0;
        fence_mbar_init();
        __syncwarp();
        if (lane == 0 && G > 1 && does_softmax(MODE)) mbar_arrive_expect_tx(smem_u32(xbar), 8u * G);
    }
    // While the previous kernel in the stream may still be running: the
    // stage-producer lanes ask L2 for the first ring's worth of this CTA's
    // rows, so that its first copies after the wait are served from L2.
    // (Ragged plans skip it: their rows depend on offsets, which may not be
    // read before the wait.)
    if (warp == kConsumerWarps && lane < kConsumerWarps && !p.offsets) {
        long long row0, nrows;
        if (G > 1) {
            const QRows qr = question_rows(p, blockIdx.y, static_cast<int>(cluster_ctarank()), G);
            row0 = qr.row0;
            nrows = qr.n;
        } else {
            const int c = blockIdx.x;
            row0 = (static_cast<long long>(c) * args.q_per_cta + min(c, args.q_rem)) * p.K;
            nrows = static_cast<long long>(args.q_per_cta + (c < args.q_rem ? 1 : 0)) * p.K;
        }
        const long long rb = static_cast<long long>(D) * sizeof(T);
        const long long total = min(nrows, static_cast<long long>(NS) * R) * rb;
        const long long piece = ((total + kConsumerWarps * 16 - 1) / (kConsumerWarps * 16)) * 16;
        const long long off = lane * piece;
        if (off < total) {
            const uint32_t bytes = static_cast<uint32_t>(min(piece, total - off));
            const unsigned char* src = reinterpret_cast<const unsigned char*>(Cg) + row0 * rb + off;
            uint32_t shift, span;  // aligned plans: shift 0, span = bytes
            const void* from = aligned_span(src, bytes, &shift, &span);
            if (CS_IN_BOUNDS(src, bytes, p.C, rows_total(p) * rb, kSitePrefetchC)) bulk_prefetch_l2(from, span);
        }
    }
    wait_prior_grid();  // no global access before this point (prefetch hints aside)
    allow_next_grid();
    if (warp == 0) {
        if (G == 1 && p.offsets) {
            // Ragged STREAM plan: CTA c takes the questions whose first row
            // falls in [c T / grid, (c+1) T / grid), T = total rows. CTA 0
            // starts at 0, the last CTA ends at B, and a CTA never ends before
            // it starts, so every question has a CTA even if offsets are bad.
            const long long c = blockIdx.x, grid = gridDim.x, rows = p.total_rows;
            long long qb0 = c == 0 ? 0 : lower_bound_warp(p.offsets, p.B, c * rows / grid, lane);
            long long qe0 = c + 1 == grid ? p.B : lower_bound_warp(p.offsets, p.B, (c + 1) * rows / grid, lane);
            if (qe0 < qb0) qe0 = qb0;
            if (lane == 0) {
                range[0] = qb0;
                range[1] = qe0;
            }
        }
    }
    __syncthreads();
    // Cluster: announce "my barriers exist"; waited on before the first push.
    if (G > 1 && does_softmax(MODE)) cluster_arrive_relaxed();

    // Questions [qb, qe) of this CTA, and its rank among the CTAs of a question.
    long long qb, qe;
    int rank = 0;
    if (G > 1) {
        rank = static_cast<int>(cluster_ctarank());
        qb = blockIdx.y;
        qe = qb + 1;
    } else if (p.offsets) {
        qb = range[0];
        qe = range[1];
    } else {
        const int c = blockIdx.x;
        qb = static_cast<long long>(c) * args.q_per_cta + min(c, args.q_rem);
        qe = qb + args.q_per_cta + (c < args.q_rem ? 1 : 0);
    }
    const uint32_t row_bytes = static_cast<uint32_t>(D) * sizeof(T);  // a row of C
    const uint32_t q_bytes = static_cast<uint32_t>(D) * 4u;
    float w = 1.f;  // value scale of the current question (value_scale)
    const float kexp = p.kexp;
    QRows last{0, 0, false};  // rows of the last question (the cluster plan's only one)

    if (warp == kConsumerWarps) {
        // ---------------- stage producers: lane l issues stages g = l, l + 8, ...
        // into slots l, l + 8, ... (the slots consumer warp l drains), so each
        // lane reuses its own slots in order; eight lanes issue in parallel.
        if (lane < kConsumerWarps) {
            const long long nqs = qe - qb;
            uint32_t slot = lane, phase = 0;
            unsigned long long issued = 0;
            long long n = 0;  // question of this lane's next stage, relative to qb
            int s = lane;     // its stage index within that question
            QRows qr = nqs > 0 ? question_rows(p, qb, rank, G) : QRows{0, 0, false};
            int nst = (qr.n + R - 1) / R;
            while (n < nqs && s >= nst) {
                s -= nst;
                if (++n < nqs) {
                    qr = question_rows(p, qb + n, rank, G);
                    nst = (qr.n + R - 1) / R;
                }
            }
            for (; n < nqs; ++issued) {
                const uint32_t bar_e = empty0 + 8u * slot, bar_f = full0 + 8u * slot;
                if (lane + kConsumerWarps * issued >= static_cast<unsigned long long>(NS) &&
                    !wait_phase(bar_e, phase ^ 1u, give_up))
                    break;
                const int k0 = s * R;
                const uint32_t bytes = static_cast<uint32_t>(min(R, qr.n - k0)) * row_bytes;
                const T* src = Cg + static_cast<size_t>(qr.row0 + k0) * D;
                unsigned char* dst = ring + static_cast<size_t>(slot) * slot_bytes;
                // UA: the rows' aligned span (the same granules as the rows'
                // own bytes, so no page they do not touch); aligned plans copy
                // exactly the rows
                uint32_t shift = 0, span = bytes;
                const void* from = UA ? aligned_span(src, bytes, &shift, &span) : src;
                const bool inb = CS_IN_BOUNDS(src, bytes, p.C, rows_total(p) * row_bytes, kSiteCopyC) &&
                                 CS_IN_BOUNDS(dst, span, ring, static_cast<size_t>(NS) * slot_bytes, kSiteRing);
                mbar_arrive_expect_tx(bar_f, inb ? span : 0u);
                if (inb) bulk_g2s(smem_u32(dst), from, span, bar_f);
                slot += kConsumerWarps;
                if (slot >= static_cast<uint32_t>(NS)) {
                    slot -= NS;
                    phase ^= 1u;
                }
                s += kConsumerWarps;
                while (n < nqs && s >= nst) {
                    s -= nst;
                    if (++n < nqs) {
                        qr = question_rows(p, qb + n, rank, G);
                        nst = (qr.n + R - 1) / R;
                    }
                }
            }
            if (*give_up) {
                // Let this lane's copies in flight land before the CTA exits.
                const unsigned long long deadline = globaltimer() + kWaitLimitNs;
                const unsigned long long per_lane = static_cast<unsigned long long>(NS / kConsumerWarps);
                for (unsigned long long m = issued > per_lane ? issued - per_lane : 0; m < issued; ++m) {
                    const unsigned long long g = lane + kConsumerWarps * m;
                    wait_phase_until(full0 + 8u * static_cast<uint32_t>(g % NS),
                                     static_cast<uint32_t>((g / NS) & 1u), deadline);
                }
            }
        }
        __syncwarp();
    } else if (warp == kConsumerWarps + 1) {
        // ---------------- query producer: one lane issues every question's q
        if (lane == 0) {
            long long nq = 0;
            for (long long b = qb; b < qe; ++b, ++nq) {
                const uint32_t qs = static_cast<uint32_t>(nq & 1), qpar = static_cast<uint32_t>((nq >> 1) & 1);
                if (nq >= 2 && !wait_phase(qempty0 + 8u * qs, qpar ^ 1u, give_up)) break;
                const float* src = p.Q + static_cast<size_t>(b) * D;
                unsigned char* dst = qbuf + qs * qslot_bytes;
                uint32_t shift = 0, span = q_bytes;
                const void* from = UA ? aligned_span(src, q_bytes, &shift, &span) : src;
                const bool inb = CS_IN_BOUNDS(src, q_bytes, p.Q, p.B * q_bytes, kSiteCopyQ) &&
                                 CS_IN_BOUNDS(dst, span, qbuf, 2 * qslot_bytes, kSiteQbuf);
                mbar_arrive_expect_tx(qfull0 + 8u * qs, inb ? span : 0u);
                if (inb) bulk_g2s(smem_u32(dst), from, span, qfull0 + 8u * qs);
            }
            if (*give_up) {
                const unsigned long long deadline = globaltimer() + kWaitLimitNs;
                for (long long u = nq > 2 ? nq - 2 : 0; u < nq; ++u)
                    wait_phase_until(qfull0 + 8u * static_cast<uint32_t>(u & 1),
                                     static_cast<uint32_t>((u >> 1) & 1), deadline);
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers: stage g belongs to warp g % kConsumerWarps;
        // this warp's slots are warp, warp + 8, ... (NS is a multiple of 8)
        uint32_t gst0 = 0;                // global index of the question's first stage
        uint32_t slot = warp, phase = 0;  // this warp's next slot and its phase
        long long nq = 0;
        QRows qr = qb < qe ? question_rows(p, qb, rank, G) : QRows{0, 0, false};
        for (long long b = qb; b < qe; ++b, ++nq) {
            // the next question's rows: loaded now, used next round
            const QRows qr_next = b + 1 < qe ? question_rows(p, b + 1, rank, G) : QRows{0, 0, false};
            const int nrows = qr.n;
            const int nst = (nrows + R - 1) / R;
            if (qr.bad && warp == 0 && lane == 0) atomicOr(&g_status, 4u);
            const uint32_t qs = static_cast<uint32_t>(nq & 1), qpar = static_cast<uint32_t>((nq >> 1) & 1);
            bool good = wait_phase(qfull0 + 8u * qs, qpar, give_up);
            unsigned char* qslot = qbuf + qs * qslot_bytes;
            const float4* q4 = reinterpret_cast<const float4*>(qslot);
            // UA: q at its offset in the aligned span the producer copied
            const float* qf = reinterpret_cast<const float*>(
                qslot + (reinterpret_cast<unsigned long long>(p.Q + static_cast<size_t>(b) * D) & 15u));
            float4 qv[(NQC > 0 ? NQC : 1) * QF4];
            unsigned long long qpk[UnitQ<T, NU>::kPairs];
            float qlast = 0.f;
            float qsq = 0.f;  // |q|^2 (cosine)
            if constexpr (NU > 0) {
                // unit u of q as packed pairs (UnitQ), zero past the row
                float sq = 0.f;
#pragma unroll
                for (int u = 0; u < UnitQ<T, NU>::kPairs; ++u) {
                    int k0, k1;
                    bool in0, in1;
                    if constexpr (std::is_same<T, float>::value) {
                        k0 = lane + 64 * u;
                        k1 = k0 + 32;
                        in0 = k0 < D;
                        in1 = k1 < D;
                    } else {
                        // pairs (2k, 2k + 1), or (2k - 1, 2k) for rows read from the word before
                        k0 = 2 * (lane + 32 * u) - (from_word_before ? 1 : 0);
                        k1 = k0 + 1;
                        in1 = lane + 32 * u < (D >> 1);
                        in0 = in1 && k0 >= 0;
                    }
                    const float a = in0 ? qf[k0] : 0.f, c = in1 ? qf[k1] : 0.f;
                    qpk[u] = pack2(a, c);
                    if (COS) sq += a * a + c * c;
                }
                if (!std::is_same<T, float>::value && ((D & 1) || from_word_before)) {
                    qlast = qf[D - 1];
                    if (COS && lane == 0) sq += qlast * qlast;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8u * qs);
                if (COS) qsq = warp_sum(sq);
            } else if constexpr (UA) {
                if (!std::is_same<T, float>::value && ((D & 1) || from_word_before)) qlast = qf[D - 1];
                if (COS) {
                    float sq = 0.f;
                    for (int i = lane; i < D; i += 32) sq = fmaf(qf[i], qf[i], sq);
                    qsq = warp_sum(sq);
                }
            } else if constexpr (NQC > 0) {
                float sq = 0.f;
#pragma unroll
                for (int j = 0; j < NQC; ++j) {
                    const int i = lane + 32 * j;
#pragma unroll
                    for (int h = 0; h < QF4; ++h) {
                        float4& x = qv[j * QF4 + h];
                        x = i < DC ? q4[i * QF4 + h] : make_float4(0.f, 0.f, 0.f, 0.f);
                        if (COS) sq += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8u * qs);
                // Every warp holds all of q, so this warp-wide sum is the whole
                // norm; it is never added across warps.
                if (COS) qsq = warp_sum(sq);
            } else if (COS) {
                float sq = 0.f;
                for (int i = lane; i < D / 4; i += 32) {
                    const float4 x = q4[i];
                    sq += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                }
                qsq = warp_sum(sq);
            }
            w = value_scale(p.w0, qsq, COS);

            float* tb = tn + (nq & 1) * 2 * kLogitSlots;  // dots
            float* nb = tb + kLogitSlots;                 // squared norms
            // first stage of this question owned by this warp
            int s = static_cast<int>((static_cast<uint32_t>(warp) + kConsumerWarps - gst0 % kConsumerWarps) %
                                     kConsumerWarps);
            for (; s < nst; s += kConsumerWarps) {
                const uint32_t bar_f = full0 + 8u * slot, bar_e = empty0 + 8u * slot;
                const bool ok = wait_phase(bar_f, phase, give_up) && good;
                const int k0 = s * R;  // relative to klo
                const int nr = min(R, nrows - k0);
                float v[V];
                unsigned char* st = ring + static_cast<size_t>(slot) * slot_bytes;
                auto release = [&] {
                    __syncwarp();  // every lane's reads of the slot are done
                    if (lane == 0) mbar_arrive(bar_e);
                };
                if constexpr (UA) {
                    // the rows at their offset in the aligned span
                    const T* src = Cg + static_cast<size_t>(qr.row0 + k0) * D;
                    const uint32_t shift = static_cast<uint32_t>(reinterpret_cast<unsigned long long>(src) & 15u);
                    // the unit reads end at most one word past the stage's rows
                    if (!CS_IN_BOUNDS(st, shift + nr * row_bytes + 4u, st, slot_bytes, kSiteUnitSlot)) {
                        release();
#pragma unroll
                        for (int i = 0; i < V; ++i) v[i] = 0.f;
                    } else if constexpr (NU > 0) {
                        stage_dots_units<NU, MODE, T, MR>(st, shift, nr, D, from_word_before, qpk, qlast, lane, v,
                                                          release);
                    } else {
                        stage_dots_units_shared_q<MODE, T, MR>(st, shift, nr, D, from_word_before, qf, qlast, lane, v,
                                                               release);
                    }
                } else {
                    stage_dots<NQC, MODE, T, MR>(reinterpret_cast<const uint4*>(st), nr, DC, qv, q4, lane, v,
                                                 release);
                }
                int idx;
                const float sum = transpose_reduce<V>(v, lane, &idx);
                if ((lane & (32 / V - 1)) == 0) {
                    const int r = idx / VPR;
                    const float val = ok ? sum : __int_as_float(0x7fc00000);
                    if (r < nr) {
                        if constexpr (does_softmax(MODE))
                            (VPR == 2 && (idx & 1) ? nb : tb)[k0 + r] = val;
                        else if (CS_IN_BOUNDS(p.staged + qr.row0 + k0 + r, 4, p.staged, rows_total(p) * 4,
                                              kSiteStagedWrite))
                            p.staged[qr.row0 + k0 + r] = MODE == kRowNorm ? sqrtf(val) : val;
                    }
                }
                slot += kConsumerWarps;
                if (slot >= static_cast<uint32_t>(NS)) {
                    slot -= NS;
                    phase ^= 1u;
                }
            }
            if constexpr (NQC == 0 || NQC == kNqcUnaligned) {  // q was read from shared memory by every stage
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8u * qs);
            }
            consumer_bar_sync();  // every row of question b has its dot (and norm)
            if (does_softmax(MODE) && G == 1 && warp == static_cast<int>(nq % kConsumerWarps)) {
                const bool inb =
                    CS_IN_BOUNDS(p.out + qr.row0, nrows * 4, p.out, rows_total(p) * 4, kSiteOut) &&
                    (MODE != kStagedCos ||
                     CS_IN_BOUNDS(p.staged + qr.row0, nrows * 4, p.staged, rows_total(p) * 4, kSiteStagedRead));
                const float* sn = MODE == kStagedCos ? p.staged + qr.row0 : nullptr;
                bool done = true;
                if (inb && nrows <= 32) {  // one row per lane: the short code path
                    float v[1];
                    load_values<MODE, 1>(tb, nb, sn, nrows, w, lane, v);
                    done = softmax_store<1>(v, nrows, kexp, p.out + qr.row0, lane);
                } else if (inb) {
                    float v[kSlotsPerLane];
                    load_values<MODE>(tb, nb, sn, nrows, w, lane, v);
                    done = softmax_store(v, nrows, kexp, p.out + qr.row0, lane);
                }
                if (!done && lane == 0) record_range(give_up);
            }
            gst0 += nst;
            last = qr;
            qr = qr_next;
        }
    }

    if (G > 1 && does_softmax(MODE)) {
        // Cluster plan (one question per cluster): warp 0 reduces this CTA's
        // rows to (m, s) = (max v, sum exp(2|a| (v - m))), pushes the pair into
        // slot `rank` of every peer's xch (completing on the peer's xbar),
        // waits for all G pairs to arrive here, and writes
        // p = exp(2|a| (v - M)) / S with M = max m_g and
        // S = sum s_g exp(2|a| (m_g - M)). A CTA with a flagged row sends NaN
        // for m, and then no CTA writes the question.
        cluster_wait();  // every CTA of the cluster has initialised its barriers
        // Warp 0; S slots of 32 rows per lane (S = 1 whenever this CTA holds
        // at most 32 rows: the short code path).
        auto finish = [&](auto slots) {
            constexpr int S = decltype(slots)::value;
            const uint32_t rank = cluster_ctarank();
            float v[S];
            const int nrows = last.n;
            const bool rd = MODE != kStagedCos || CS_IN_BOUNDS(p.staged + last.row0, nrows * 4, p.staged,
                                                                rows_total(p) * 4, kSiteStagedRead);
            const int nread = rd ? nrows : 0;
            load_values<MODE, S>(tn, tn + kLogitSlots, MODE == kStagedCos ? p.staged + last.row0 : nullptr, nread, w,
                                 lane, v);
            float m;
            const float s = exp_rows<S>(v, nread, kexp, lane, &m);
            if (lane < G && CS_IN_BOUNDS(xch + rank, 8, xch, kMaxCluster * 8, kSitePeer))
                st_async_peer(peer_addr(xch + rank, static_cast<uint32_t>(lane)), make_float2(m, s),
                              peer_addr(xbar, static_cast<uint32_t>(lane)));
            const bool ok = wait_phase(smem_u32(xbar), 0, give_up);
            float M;
            bool flagged;
            const float inv = combine_pairs(xch, G, kexp, lane, &M, &flagged);
            const float rescale = softmax_term(kexp, m - M) * inv;  // 2^(kexp (m - M)) / S
            float* dst = p.out + last.row0;
            if (ok && flagged) {
                if (lane == 0) record_range(give_up);
            } else if (CS_IN_BOUNDS(dst, nrows * 4, p.out, rows_total(p) * 4, kSiteOutCluster)) {
#pragma unroll
                for (int j = 0; j < S; ++j) {
                    const int k = lane + 32 * j;
                    if (k < nrows) dst[k] = ok ? v[j] * rescale : qnan();
                }
            }
        };
        if (warp == 0) {
            if (last.n <= 32)
                finish(std::integral_constant<int, 1>{});
            else
                finish(std::integral_constant<int, kSlotsPerLane>{});
        }
        __syncwarp();
        // Leave only when every CTA has received every pair: no push into a
        // CTA that has exited, none left in flight.
        cluster_arrive_relaxed();
        cluster_wait();
    }
}

// ------------------------------------------------------------------ direct kernel

// Short path for one or a few questions whose rows come to at most 32 per CTA
// (DIRECT plan): no ring and no producer warps. CTA `rank` of a cluster of G
// takes its share of question blockIdx.y; warp w owns rows w, w+8, ... of
// that share and loads them straight into registers with 16-byte loads, all
// issued before any arithmetic, so the whole question costs one trip to
// L2/HBM. q sits in registers (narrow form: RPW = 4 rows per warp, D up to
// 32 * NQC chunks) or, for long rows, once per CTA in shared memory (wide
// form: RPW = 2, QSH). Dots and squared norms are reduced as in the stream
// kernel (packed FMAs, transposed butterfly), one warp takes the softmax of
// the CTA's rows, and a cluster combines (max, sum) through distributed
// shared memory exactly like the CLUSTER plan.
constexpr int kDirectThreads = 256;
constexpr int kDirectRows = kDirectMaxRows;     // rows per CTA, narrow form (4 per warp)
constexpr int kDirectWideNqc = kDirectWideChunks;  // wide form: chunks per lane (D <= 2560 float32, 5120 bfloat16)
constexpr int kDirectMaxQ4 = kDirectWideMaxD / 4;  // wide form: q in shared memory, float4s
static_assert(kDirectWideMaxRows == 2 * (kDirectThreads / 32), "wide form: 2 rows per warp");

template <int NQC, int MODE, typename T, int RPW, bool QSH>
__global__ void __launch_bounds__(kDirectThreads, 1) direct_kernel(const Problem p, int G) {
    constexpr int VPR = values_per_row(MODE);
    constexpr int V = VPR * RPW;
    constexpr int ROWS = RPW * (kDirectThreads / 32);
    constexpr bool COS = cos_logits(MODE);
    constexpr int QF4 = Elem<T>::kQF4;
    __shared__ float tn[2 * kDirectRows];  // dots, then squared norms
    __shared__ float2 xch[kMaxCluster];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ int give_up_flag;
    __shared__ float4 qsh[QSH ? kDirectMaxQ4 : 1];
    volatile int* give_up = &give_up_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.D, DC = D / Elem<T>::kPerChunk;
    const long long b = blockIdx.y;
    const int rank = G > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&xbar), 1);
        give_up_flag = 0;
        fence_mbar_init();
        if (G > 1) mbar_arrive_expect_tx(smem_u32(&xbar), 8u * G);
    }
    wait_prior_grid();  // no global access before this point
    allow_next_grid();

    // NU > 0: rows that do not start on 16-byte boundaries (or whose length
    // is not a multiple of 16 bytes), read in 4-byte units as the stream
    // kernel's unaligned plans read them from shared memory (stage_dots_units):
    // lane takes units lane, lane + 32, ... -- float32 elements or bfloat16
    // pairs, bfloat16 rows of an even D on an odd 2-byte boundary from the
    // word before (bf16_rows_from_word_before); no odd-D bfloat16 form.
    constexpr int NU = unaligned_units(NQC);
    constexpr bool F32 = std::is_same<T, float>::value;
    constexpr int GV = NU > 4 ? NU / 2 : 0;  // units always inside the row (the plan picks NU so)
    const bool from_word_before = !F32 && bf16_rows_from_word_before(p.C, D);

    const QRows qr = question_rows(p, b, rank, G);
    const int n = qr.n;
    const bool skip = qr.bad || n > ROWS || (QSH && D > 4 * kDirectMaxQ4) ||
                      (NU > 0 && !F32 && (D & 1));  // the host plans none of these
    if (threadIdx.x == 0 && qr.bad) atomicOr(&g_status, 4u);
    if (threadIdx.x == 0 && !qr.bad && skip) atomicOr(&g_status, 2u);

    // this warp's rows, then q: every load issued before any arithmetic
    uint4 cv[RPW][NQC > 0 ? NQC : 1];
    uint32_t cw[RPW][NU > 0 ? NU : 1];
    uint16_t ctail[RPW];
    if constexpr (NU > 0) {
#pragma unroll
        for (int m = 0; m < RPW; ++m) {
            const int r = warp + 8 * m;
            const T* row = static_cast<const T*>(p.C) + static_cast<size_t>(qr.row0 + (r < n ? r : 0)) * D;
            const bool ok = !skip && r < n &&
                            CS_IN_BOUNDS(row, static_cast<long long>(D) * sizeof(T), p.C,
                                         rows_total(p) * D * static_cast<long long>(sizeof(T)), kSiteGenericC);
            // float32: the row's own words; bfloat16: from the word holding
            // element -1 when the row starts on an odd 2-byte boundary
            const uint32_t* wr = reinterpret_cast<const uint32_t*>(reinterpret_cast<const unsigned char*>(row) -
                                                                   (from_word_before ? 2 : 0));
            const int units = F32 ? D : D >> 1;
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int k = lane + 32 * u;
                cw[m][u] = ok && (u < GV || k < units) ? __ldg(wr + k) : 0u;
            }
            if (from_word_before && lane == 0) cw[m][0] &= 0xffff0000u;  // element -1
            ctail[m] = 0;
            if constexpr (!F32)
                if (from_word_before && lane == 0 && ok) ctail[m] = __ldg(reinterpret_cast<const uint16_t*>(row) + D - 1);
        }
    }
#pragma unroll
    for (int m = 0; m < (NU > 0 ? 0 : RPW); ++m) {
        const int r = warp + 8 * m;
        const uint4* row = reinterpret_cast<const uint4*>(static_cast<const T*>(p.C) +
                                                          static_cast<size_t>(qr.row0 + (r < n ? r : 0)) * D);
        const bool ok = !skip && r < n &&
                        CS_IN_BOUNDS(row, static_cast<long long>(D) * sizeof(T), p.C,
                                     rows_total(p) * D * static_cast<long long>(sizeof(T)), kSiteGenericC);
#pragma unroll
        for (int j = 0; j < NQC; ++j) {
            const int i = lane + 32 * j;
            cv[m][j] = ok && i < DC ? __ldg(row + i) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    const float4* q4 = reinterpret_cast<const float4*>(p.Q + b * D);
    const bool q_ok = !skip && CS_IN_BOUNDS(q4, D * 4ll, p.Q, p.B * D * 4ll, kSiteGenericQ);
    float4 qv[QSH || NU > 0 ? 1 : NQC * QF4];
    unsigned long long qpk[UnitQ<T, NU>::kPairs];  // NU > 0: q of the lane's units (UnitQ)
    float qlast = 0.f;                             // bfloat16 read from the word before: q[D - 1]
    if constexpr (NU > 0) {
        const float* qg = p.Q + b * D;
#pragma unroll
        for (int u = 0; u < UnitQ<T, NU>::kPairs; ++u) {
            int k0, k1;
            bool in0, in1;
            if constexpr (F32) {
                k0 = lane + 64 * u;
                k1 = k0 + 32;
                in0 = q_ok && k0 < D;
                in1 = q_ok && k1 < D;
            } else {
                k0 = 2 * (lane + 32 * u) - (from_word_before ? 1 : 0);
                k1 = k0 + 1;
                in1 = q_ok && lane + 32 * u < (D >> 1);
                in0 = in1 && k0 >= 0;
            }
            qpk[u] = pack2(in0 ? __ldg(qg + k0) : 0.f, in1 ? __ldg(qg + k1) : 0.f);
        }
        if (!F32 && from_word_before && q_ok) qlast = __ldg(qg + D - 1);
    } else if constexpr (QSH) {
        for (int i = threadIdx.x; i < D / 4; i += kDirectThreads)
            qsh[i] = q_ok ? __ldg(q4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
#pragma unroll
        for (int j = 0; j < NQC; ++j) {
            const int i = lane + 32 * j;
#pragma unroll
            for (int h = 0; h < QF4; ++h)
                qv[j * QF4 + h] = q_ok && i < DC ? __ldg(q4 + i * QF4 + h) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();  // the mbarrier is initialised; q is in shared memory (wide form)
    if (G > 1) cluster_arrive_relaxed();  // "my barrier exists"; waited on before the first push

    // q's chunk (j, h) of this lane
    auto qchunk = [&](int j, int h) -> float4 {
        if constexpr (NU > 0) {  // not used: the unit form keeps q in qpk
            return make_float4(0.f, 0.f, 0.f, 0.f);
        } else if constexpr (QSH) {
            const int i = lane + 32 * j;
            return i < DC ? qsh[i * QF4 + h] : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            return qv[j * QF4 + h];
        }
    };
    float qsq = 0.f;
    if (COS) {
        float sq = 0.f;
        if constexpr (NU > 0) {
#pragma unroll
            for (int u = 0; u < UnitQ<T, NU>::kPairs; ++u) {
                const float2 x = unpack2(qpk[u]);
                sq += x.x * x.x + x.y * x.y;
            }
            if (lane == 0) sq += qlast * qlast;
        } else {
#pragma unroll
            for (int j = 0; j < NQC; ++j)
#pragma unroll
                for (int h = 0; h < QF4; ++h) {
                    const float4 x = qchunk(j, h);
                    sq += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                }
        }
        qsq = warp_sum(sq);  // each warp covers all of q: never summed across warps
    }
    const float w = value_scale(p.w0, qsq, COS);
    const float kexp = p.kexp;

    // dot (and squared norm) of each row: two packed partial sums each
    unsigned long long acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0ull;
    if constexpr (NU > 0) {
        auto accumulate = [&](unsigned long long c, unsigned long long qq, int m) {
            if (acc_dot(MODE)) acc[VPR * m] = fma2(c, qq, acc[VPR * m]);
            if (acc_norm(MODE)) acc[VPR * m + VPR - 1] = fma2(c, c, acc[VPR * m + VPR - 1]);
        };
#pragma unroll
        for (int m = 0; m < RPW; ++m) {
            if constexpr (F32) {
#pragma unroll
                for (int u = 0; u < NU / 2; ++u)
                    accumulate(pack2(__uint_as_float(cw[m][2 * u]), __uint_as_float(cw[m][2 * u + 1])), qpk[u], m);
            } else {
#pragma unroll
                for (int u = 0; u < NU; ++u)
                    accumulate(pack2(__uint_as_float(cw[m][u] << 16), __uint_as_float(cw[m][u] & 0xffff0000u)),
                               qpk[u], m);
                if (from_word_before)
                    accumulate(pack2(Elem<uint16_t>::widen1(ctail[m]), 0.f), pack2(qlast, 0.f), m);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < (NU > 0 ? 0 : NQC); ++j) {
        float4 q[QF4];
#pragma unroll
        for (int h = 0; h < QF4; ++h) q[h] = qchunk(j, h);
#pragma unroll
        for (int m = 0; m < RPW; ++m) {
            float4 c[QF4];
            Elem<T>::widen(cv[m][j], c);
#pragma unroll
            for (int h = 0; h < QF4; ++h) {
                const unsigned long long q01 = pack2(q[h].x, q[h].y), q23 = pack2(q[h].z, q[h].w);
                const unsigned long long c01 = pack2(c[h].x, c[h].y), c23 = pack2(c[h].z, c[h].w);
                if (acc_dot(MODE)) {
                    acc[VPR * m] = fma2(c01, q01, acc[VPR * m]);
                    acc[VPR * m] = fma2(c23, q23, acc[VPR * m]);
                }
                if (acc_norm(MODE)) {
                    acc[VPR * m + VPR - 1] = fma2(c01, c01, acc[VPR * m + VPR - 1]);
                    acc[VPR * m + VPR - 1] = fma2(c23, c23, acc[VPR * m + VPR - 1]);
                }
            }
        }
    }
    float v[V];
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = sum2(acc[i]);
    int idx;
    const float sum = transpose_reduce<V>(v, lane, &idx);
    if ((lane & (32 / V - 1)) == 0) {
        const int r = warp + 8 * (idx / VPR);
        if (r < n && !skip) tn[(VPR == 2 && (idx & 1) ? kDirectRows : 0) + r] = sum;
    }
    __syncthreads();

    if (G > 1) cluster_wait();  // every CTA of the cluster has initialised its barrier
    bool arrived = false;  // warp-uniform: this warp has arrived at the closing cluster barrier
    if (warp == 0 && !skip) {
        float v[1] = {-INFINITY};
        if (lane < n) v[0] = row_value<COS ? kFusedCos : kFusedDot>(tn[lane], tn[kDirectRows + lane], w);
        float* dst = p.out + qr.row0;
        const bool out_ok = CS_IN_BOUNDS(dst, n * 4ll, p.out, rows_total(p) * 4, kSiteOutCluster);
        if (G == 1) {
            if (out_ok && !softmax_store<1>(v, n, kexp, dst, lane) && lane == 0) record_range(give_up);
        } else {
            float m;
            const float s = exp_rows<1>(v, n, kexp, lane, &m);
            if (lane < G && CS_IN_BOUNDS(xch + rank, 8, xch, kMaxCluster * 8, kSitePeer))
                st_async_peer(peer_addr(xch + rank, static_cast<uint32_t>(lane)), make_float2(m, s),
                              peer_addr(&xbar, static_cast<uint32_t>(lane)));
            const bool ok = wait_phase(smem_u32(&xbar), 0, give_up);
            // Every pair bound for this CTA has landed (or the wait gave up,
            // after which the closing barrier still holds the CTA until all
            // peers have arrived): arrive now, so that the barrier's round
            // trip overlaps the rest of the softmax and the stores.
            __syncwarp();
            cluster_arrive_relaxed();
            arrived = true;
            float M;
            bool flagged;
            const float inv = combine_pairs(xch, G, kexp, lane, &M, &flagged);
            if (ok && flagged) {
                if (lane == 0) record_range(give_up);
            } else if (out_ok && lane < n) {
                dst[lane] = ok ? v[0] * (softmax_term(kexp, m - M) * inv) : qnan();
            }
        }
    }
    if (G > 1) {
        // Leave only when every CTA has received every pair (none in flight
        // into a CTA that has exited).
        __syncwarp();
        if (!arrived) cluster_arrive_relaxed();
        cluster_wait();
    }
}

// ------------------------------------------------------------------ generic kernel

// One CTA per question (G = 1), or each question's rows split over the G
// CTAs of a thread-block cluster (G > 1, uniform K; the rows of CTA r are
// r K / G .. (r + 1) K / G - 1) with the softmax combined through
// distributed shared memory as in the DIRECT plan. One warp per candidate
// row, scalar coalesced loads: any D, any alignment. CL: built for G > 1
// (the one-CTA form carries none of the exchange, so it keeps its
// registers, and its occupancy, low).
template <bool COS, typename T, bool CL>
__global__ void __launch_bounds__(kGenericThreads) generic_kernel(const Problem p, int G) {
    if constexpr (!CL) G = 1;
    __shared__ float lg[kLogitSlots];
    __shared__ float2 xch[kMaxCluster];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ int give_up_flag;
    volatile int* give_up = &give_up_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = kGenericThreads / 32;
    const long long b = G > 1 ? static_cast<long long>(blockIdx.y) : static_cast<long long>(blockIdx.x);
    const int rank = G > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    if (G > 1) {
        if (threadIdx.x == 0) {
            mbar_init(smem_u32(&xbar), 1);
            give_up_flag = 0;
            fence_mbar_init();
            mbar_arrive_expect_tx(smem_u32(&xbar), 8u * G);
        }
        cluster_arrive_relaxed();  // "my barrier exists"; waited on before the first push
    }
    const QRows qr = question_rows(p, b, rank, G);
    const int K = qr.n, D = p.D;
    const float* __restrict__ q = p.Q + static_cast<size_t>(b) * D;
    if (qr.bad && threadIdx.x == 0) atomicOr(&g_status, 4u);
    const bool skip = qr.bad || !CS_IN_BOUNDS(q, D * 4ll, p.Q, p.B * D * 4ll, kSiteGenericQ) ||
                      !CS_IN_BOUNDS(p.out + qr.row0, K * 4ll, p.out, rows_total(p) * 4, kSiteGenericOut);
    if (!CL && skip) return;  // nothing waits on a CTA of its own; a cluster's CTAs all reach its barriers
    float qsq = 0.f;
    if (COS && !skip) {
        float sq = 0.f;
        for (int d = lane; d < D; d += 32) {
            const float v = __ldg(q + d);
            sq = fmaf(v, v, sq);
        }
        qsq = warp_sum(sq);  // whole norm per warp, never summed across warps
    }
    const float w = value_scale(p.w0, qsq, COS);
    const float kexp = p.kexp;
    for (int k = warp; k < K && !skip; k += nwarps) {
        const T* __restrict__ c = static_cast<const T*>(p.C) + static_cast<size_t>(qr.row0 + k) * D;
        if (!CS_IN_BOUNDS(c, D * static_cast<long long>(sizeof(T)), p.C, rows_total(p) * D * static_cast<long long>(sizeof(T)),
                          kSiteGenericC)) {
            if (lane == 0) lg[k] = -INFINITY;
            continue;
        }
        float t0 = 0.f, t1 = 0.f, n0 = 0.f, n1 = 0.f;
        int d = lane;
        for (; d + 32 < D; d += 64) {
            const float c0 = Elem<T>::value(c, d), c1 = Elem<T>::value(c, d + 32);
            t0 = fmaf(c0, __ldg(q + d), t0);
            t1 = fmaf(c1, __ldg(q + d + 32), t1);
            if (COS) {
                n0 = fmaf(c0, c0, n0);
                n1 = fmaf(c1, c1, n1);
            }
        }
        if (d < D) {
            const float c0 = Elem<T>::value(c, d);
            t0 = fmaf(c0, __ldg(q + d), t0);
            if (COS) n0 = fmaf(c0, c0, n0);
        }
        const float t = warp_sum(t0 + t1);
        const float n = COS ? warp_sum(n0 + n1) : 0.f;
        if (lane == 0) lg[k] = row_value<COS ? kFusedCos : kFusedDot>(t, n, w);
    }
    __syncthreads();
    if (G > 1) cluster_wait();  // every CTA of the cluster has initialised its barrier
    bool arrived = false;       // warp-uniform: this warp has arrived at the closing cluster barrier
    if (warp == 0 && !skip) {
        float v[kSlotsPerLane];
#pragma unroll
        for (int j = 0; j < kSlotsPerLane; ++j) v[j] = lane + 32 * j < K ? lg[lane + 32 * j] : -INFINITY;
        float* dst = p.out + qr.row0;
        if constexpr (!CL) {
            // no waits in this form, so a flagged row is a range failure
            if (!softmax_store(v, K, kexp, dst, lane) && lane == 0) atomicOr(&g_status, kDevErrRange);
        } else {
            // this CTA's (max, sum of exp) to every CTA of the cluster
            float m;
            const float s = exp_rows<kSlotsPerLane>(v, K, kexp, lane, &m);
            if (lane < G && CS_IN_BOUNDS(xch + rank, 8, xch, kMaxCluster * 8, kSitePeer))
                st_async_peer(peer_addr(xch + rank, static_cast<uint32_t>(lane)), make_float2(m, s),
                              peer_addr(&xbar, static_cast<uint32_t>(lane)));
            const bool ok = wait_phase(smem_u32(&xbar), 0, give_up);
            // every pair bound for this CTA has landed (or the wait gave up)
            __syncwarp();
            cluster_arrive_relaxed();
            arrived = true;
            float M;
            bool flagged;
            const float inv = combine_pairs(xch, G, kexp, lane, &M, &flagged);
            const float rescale = softmax_term(kexp, m - M) * inv;
            if (ok && flagged) {
                if (lane == 0) record_range(give_up);
            } else {
#pragma unroll
                for (int j = 0; j < kSlotsPerLane; ++j)
                    if (lane + 32 * j < K) dst[lane + 32 * j] = ok ? v[j] * rescale : qnan();
            }
        }
    }
    if (G > 1) {
        // Leave only when every CTA has received every pair.
        __syncwarp();
        if (!arrived) cluster_arrive_relaxed();
        cluster_wait();
    }
}

// Unfused baseline pass 2 (dot): one warp per question, softmax of
// factor * staged over the question's K staged similarities.
__global__ void __launch_bounds__(256) staged_softmax_kernel(const Problem p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long b = static_cast<long long>(blockIdx.x) * 8 + warp;
    if (b >= p.B) return;
    const float w = p.w0;
    const float* t = p.staged + static_cast<size_t>(b) * p.K;
    if (!CS_IN_BOUNDS(t, p.K * 4ll, p.staged, p.B * p.K * 4ll, kSiteStagedSoftmax) ||
        !CS_IN_BOUNDS(p.out + static_cast<size_t>(b) * p.K, p.K * 4ll, p.out, p.B * p.K * 4ll, kSiteStagedSoftmaxOut))
        return;
    float v[kSlotsPerLane];
    load_values<kFusedDot>(t, nullptr, nullptr, p.K, w, lane, v);
    if (!softmax_store(v, p.K, p.kexp, p.out + static_cast<size_t>(b) * p.K, lane) && lane == 0)
        atomicOr(&g_status, kDevErrRange);  // no waits here: a flagged row is a range failure
}

// Self-test of the bounded wait: one thread waits, with the kernels' own
// wait_phase, on an mbarrier nothing will ever arrive at; after limit_ns it
// gives up, sets the device status bit and returns. Nothing is copied into
// shared memory, so nothing is in flight when it leaves.
__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int flag;
    if (threadIdx.x == 0) {
        flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        (void)wait_phase(smem_u32(&bar), 0, reinterpret_cast<volatile int*>(&flag), limit_ns);
    }
}

#ifdef CS_DEBUG_BOUNDS
// Self-test of the bounds checks: one thread checks the range one past the
// end of a 64-byte buffer (arithmetic only: nothing is read or written).
__global__ void selftest_bounds_kernel() {
    __shared__ float buf[16];
    if (threadIdx.x == 0) (void)CS_IN_BOUNDS(buf + 16, 4, buf, sizeof(buf), kSiteSelftest);
}
#endif

// ------------------------------------------------------------------ dispatch

template <int NQC, int MODE, typename T, int MR>
cudaError_t launch_stream_t(const StreamArgs& a, const Plan& plan, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (plan.kind == kPlanCluster) {
        cfg.gridDim = dim3(static_cast<unsigned>(plan.cluster), static_cast<unsigned>(a.p.B), 1);
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    } else {
        cfg.gridDim = dim3(static_cast<unsigned>(plan.ctas), 1, 1);
    }
    return cudaLaunchKernelEx(&cfg, stream_kernel<NQC, MODE, T, MR>, a);
}

// Unaligned rows: built for the fused modes at the full stage size only.
template <int MODE, int MR>
constexpr bool has_unaligned_build() {
    return (MODE == kFusedCos || MODE == kFusedDot) && MR == kMaxRowsPerStage;
}

template <int NQC, int MODE, typename T, int MR>
cudaError_t launch_stream_ua(const StreamArgs& a, const Plan& plan, cudaStream_t stream) {
    if constexpr (has_unaligned_build<MODE, MR>())
        return launch_stream_t<NQC, MODE, T, MR>(a, plan, stream);
    else
        return cudaErrorInvalidValue;
}

template <int NQC, int MODE, typename T, int MR>
const void* stream_fn_ua() {
    if constexpr (has_unaligned_build<MODE, MR>())
        return reinterpret_cast<const void*>(stream_kernel<NQC, MODE, T, MR>);
    else
        return nullptr;
}

template <int MODE, typename T, int MR>
cudaError_t launch_stream_m(const StreamArgs& a, const Plan& plan, cudaStream_t stream) {
    switch (plan.nq4) {
        case kNqcUnaligned: return launch_stream_ua<kNqcUnaligned, MODE, T, MR>(a, plan, stream);
        case unaligned_nqc(4): return launch_stream_ua<unaligned_nqc(4), MODE, T, MR>(a, plan, stream);
        case unaligned_nqc(8): return launch_stream_ua<unaligned_nqc(8), MODE, T, MR>(a, plan, stream);
        case unaligned_nqc(16): return launch_stream_ua<unaligned_nqc(16), MODE, T, MR>(a, plan, stream);
        case 1: return launch_stream_t<1, MODE, T, MR>(a, plan, stream);
        case 2: return launch_stream_t<2, MODE, T, MR>(a, plan, stream);
        case 4: return launch_stream_t<4, MODE, T, MR>(a, plan, stream);
        case 8: return launch_stream_t<8, MODE, T, MR>(a, plan, stream);
        case 0: return launch_stream_t<0, MODE, T, MR>(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int MODE, typename T, int MR>
const void* stream_fn_m(int nqc) {
    switch (nqc) {
        case kNqcUnaligned: return stream_fn_ua<kNqcUnaligned, MODE, T, MR>();
        case unaligned_nqc(4): return stream_fn_ua<unaligned_nqc(4), MODE, T, MR>();
        case unaligned_nqc(8): return stream_fn_ua<unaligned_nqc(8), MODE, T, MR>();
        case unaligned_nqc(16): return stream_fn_ua<unaligned_nqc(16), MODE, T, MR>();
        case 1: return reinterpret_cast<const void*>(stream_kernel<1, MODE, T, MR>);
        case 2: return reinterpret_cast<const void*>(stream_kernel<2, MODE, T, MR>);
        case 4: return reinterpret_cast<const void*>(stream_kernel<4, MODE, T, MR>);
        case 8: return reinterpret_cast<const void*>(stream_kernel<8, MODE, T, MR>);
        case 0: return reinterpret_cast<const void*>(stream_kernel<0, MODE, T, MR>);
    }
    return nullptr;
}

// The row limit of the instantiation that runs stages of R rows in `mode`
// (unaligned plans have only the full-size build).
constexpr int rows_limit(int mode, int R, int nqc) {
    return (mode == kFusedCos || mode == kFusedDot) && R <= kSmallStageRows && nqc >= 0
               ? kSmallStageRows
               : kMaxRowsPerStage;
}

// Kernels exist for every mode over float32 C, and for the fused modes over
// bfloat16 C (nqc 8 is never planned for bfloat16: q would take 64 registers);
// the fused modes also in a short-stage form (mr = kSmallStageRows) and, at
// the full stage size, for unaligned rows (nqc < 0).
const void* stream_fn_for(int nqc, int mode, int c_bf16, int mr) {
    const bool fused = mode == kFusedCos || mode == kFusedDot;
    if (nqc < 0 && (!fused || mr != kMaxRowsPerStage)) return nullptr;
    if (mr == kSmallStageRows) {
        if (!fused || (c_bf16 && nqc == 8)) return nullptr;
        if (c_bf16)
            return mode == kFusedCos ? stream_fn_m<kFusedCos, uint16_t, kSmallStageRows>(nqc)
                                     : stream_fn_m<kFusedDot, uint16_t, kSmallStageRows>(nqc);
        return mode == kFusedCos ? stream_fn_m<kFusedCos, float, kSmallStageRows>(nqc)
                                 : stream_fn_m<kFusedDot, float, kSmallStageRows>(nqc);
    }
    if (mr != kMaxRowsPerStage) return nullptr;
    if (c_bf16) {
        if (nqc == 8) return nullptr;
        switch (mode) {
            case kFusedCos: return stream_fn_m<kFusedCos, uint16_t, kMaxRowsPerStage>(nqc);
            case kFusedDot: return stream_fn_m<kFusedDot, uint16_t, kMaxRowsPerStage>(nqc);
        }
        return nullptr;
    }
    switch (mode) {
        case kFusedCos: return stream_fn_m<kFusedCos, float, kMaxRowsPerStage>(nqc);
        case kFusedDot: return stream_fn_m<kFusedDot, float, kMaxRowsPerStage>(nqc);
        case kRowNorm: return stream_fn_m<kRowNorm, float, kMaxRowsPerStage>(nqc);
        case kRowDot: return stream_fn_m<kRowDot, float, kMaxRowsPerStage>(nqc);
        case kStagedCos: return stream_fn_m<kStagedCos, float, kMaxRowsPerStage>(nqc);
    }
    return nullptr;
}

}  // namespace

cudaError_t launch_stream(const Problem& p, const Plan& plan, int mode, cudaStream_t stream) {
    StreamArgs a;
    a.p = p;
    a.rows_per_stage = plan.rows_per_stage;
    a.stages = plan.stages;
    a.cluster = plan.kind == kPlanCluster ? plan.cluster : 1;
    const long long ctas = plan.kind == kPlanCluster ? 1 : plan.ctas;
    a.q_per_cta = static_cast<int>(p.B / ctas);
    a.q_rem = static_cast<int>(p.B % ctas);
    const bool small = rows_limit(mode, plan.rows_per_stage, plan.nq4) == kSmallStageRows;
    if (p.c_bf16) {
        if (plan.nq4 == 8) return cudaErrorInvalidValue;
        switch (mode) {
            case kFusedCos:
                return small ? launch_stream_m<kFusedCos, uint16_t, kSmallStageRows>(a, plan, stream)
                             : launch_stream_m<kFusedCos, uint16_t, kMaxRowsPerStage>(a, plan, stream);
            case kFusedDot:
                return small ? launch_stream_m<kFusedDot, uint16_t, kSmallStageRows>(a, plan, stream)
                             : launch_stream_m<kFusedDot, uint16_t, kMaxRowsPerStage>(a, plan, stream);
        }
        return cudaErrorInvalidValue;
    }
    switch (mode) {
        case kFusedCos:
            return small ? launch_stream_m<kFusedCos, float, kSmallStageRows>(a, plan, stream)
                         : launch_stream_m<kFusedCos, float, kMaxRowsPerStage>(a, plan, stream);
        case kFusedDot:
            return small ? launch_stream_m<kFusedDot, float, kSmallStageRows>(a, plan, stream)
                         : launch_stream_m<kFusedDot, float, kMaxRowsPerStage>(a, plan, stream);
        case kRowNorm: return launch_stream_m<kRowNorm, float, kMaxRowsPerStage>(a, plan, stream);
        case kRowDot: return launch_stream_m<kRowDot, float, kMaxRowsPerStage>(a, plan, stream);
        case kStagedCos: return launch_stream_m<kStagedCos, float, kMaxRowsPerStage>(a, plan, stream);
    }
    return cudaErrorInvalidValue;
}

template <int MODE, typename T>
const void* direct_fn_m(int nqc) {
    switch (nqc) {
        case 1: return reinterpret_cast<const void*>(direct_kernel<1, MODE, T, 4, false>);
        case 2: return reinterpret_cast<const void*>(direct_kernel<2, MODE, T, 4, false>);
        case 4: return reinterpret_cast<const void*>(direct_kernel<4, MODE, T, 4, false>);
        case kDirectWideNqc:
            return reinterpret_cast<const void*>(direct_kernel<kDirectWideNqc, MODE, T, 2, true>);
        case unaligned_nqc(4): return reinterpret_cast<const void*>(direct_kernel<unaligned_nqc(4), MODE, T, 4, false>);
        case unaligned_nqc(8): return reinterpret_cast<const void*>(direct_kernel<unaligned_nqc(8), MODE, T, 4, false>);
        case unaligned_nqc(16):
            return reinterpret_cast<const void*>(direct_kernel<unaligned_nqc(16), MODE, T, 4, false>);
    }
    return nullptr;
}

const void* direct_fn_for(int nqc, int normalize, int c_bf16) {
    if (c_bf16) return normalize ? direct_fn_m<kFusedCos, uint16_t>(nqc) : direct_fn_m<kFusedDot, uint16_t>(nqc);
    return normalize ? direct_fn_m<kFusedCos, float>(nqc) : direct_fn_m<kFusedDot, float>(nqc);
}

cudaError_t launch_direct(const Problem& p, const Plan& plan, cudaStream_t stream) {
    const void* f = direct_fn_for(plan.nq4, p.normalize, p.c_bf16);
    if (!f || p.B > 65535 || plan.cluster < 1 || plan.cluster > kMaxCluster) return cudaErrorInvalidValue;
    int G = plan.cluster;
    void* args[] = {const_cast<Problem*>(&p), &G};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(static_cast<unsigned>(G), static_cast<unsigned>(p.B), 1);
    cfg.blockDim = dim3(kDirectThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (G > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(G);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, f, args);
}

int max_active_direct_clusters(int cluster, int nq4, int normalize, int c_bf16) {
    const void* f = direct_fn_for(nq4, normalize, c_bf16);
    if (!f) return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(kDirectThreads, 1, 1);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_staged_softmax(const Problem& p, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((p.B + 7) / 8)), block(256);
    staged_softmax_kernel<<<grid, block, 0, stream>>>(p);
    return cudaGetLastError();
}

void (*generic_fn_for(int normalize, int c_bf16, bool clustered))(Problem, int) {
    if (clustered) {
        if (c_bf16) return normalize ? generic_kernel<true, uint16_t, true> : generic_kernel<false, uint16_t, true>;
        return normalize ? generic_kernel<true, float, true> : generic_kernel<false, float, true>;
    }
    if (c_bf16) return normalize ? generic_kernel<true, uint16_t, false> : generic_kernel<false, uint16_t, false>;
    return normalize ? generic_kernel<true, float, false> : generic_kernel<false, float, false>;
}

cudaLaunchConfig_t generic_cluster_config(unsigned G, unsigned B, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G, B, 1);
    cfg.blockDim = dim3(kGenericThreads, 1, 1);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t launch_generic(const Problem& p, int G, cudaStream_t stream) {
    void (*f)(Problem, int) = generic_fn_for(p.normalize, p.c_bf16, G > 1);
    if (G <= 1) {
        f<<<dim3(static_cast<unsigned>(p.B)), dim3(kGenericThreads), 0, stream>>>(p, 1);
        return cudaGetLastError();
    }
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        generic_cluster_config(static_cast<unsigned>(G), static_cast<unsigned>(p.B), stream, attr);
    return cudaLaunchKernelEx(&cfg, f, p, G);
}

int max_active_generic_clusters(int cluster, int normalize, int c_bf16) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = generic_cluster_config(static_cast<unsigned>(cluster), 1, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, generic_fn_for(normalize, c_bf16, true), &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t configure_device_kernels(int smem_optin) {
    for (int cos = 0; cos < 2; ++cos)
        for (int bf = 0; bf < 2; ++bf) {
            const cudaError_t e =
                cudaFuncSetAttribute(generic_fn_for(cos, bf, true), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
    for (int nqc : {1, 2, 4, kDirectWideNqc, unaligned_nqc(4), unaligned_nqc(8), unaligned_nqc(16)})
        for (int cos = 0; cos < 2; ++cos)
            for (int bf = 0; bf < 2; ++bf) {
                const cudaError_t e =
                    cudaFuncSetAttribute(direct_fn_for(nqc, cos, bf), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
            }
    const int nq4s[9] = {1, 2, 4, 8, 0, kNqcUnaligned, unaligned_nqc(4), unaligned_nqc(8), unaligned_nqc(16)};
    for (int bf = 0; bf < 2; ++bf) {
        for (int m = kFusedCos; m <= kStagedCos; ++m) {
            for (int i = 0; i < 9; ++i) {
                for (int mr : {kSmallStageRows, kMaxRowsPerStage}) {
                    const void* f = stream_fn_for(nq4s[i], m, bf, mr);
                    if (!f) continue;
                    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
                    if (e != cudaSuccess) return e;
                    e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (e != cudaSuccess) return e;
                }
            }
        }
    }
    return cudaSuccess;
}

int max_active_clusters(int cluster, size_t smem, int nq4, int normalize, int c_bf16, int rows_per_stage) {
    const int mode = normalize ? kFusedCos : kFusedDot;
    const void* f = stream_fn_for(nq4, mode, c_bf16, rows_limit(mode, rows_per_stage, nq4));
    if (!f) return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Built-in staged array for cs_score_candidates_batch_unfused_noalloc, for
// callers that cannot allocate device memory themselves. It takes 4 MiB on
// every device that loads this library, for the life of the process. Host
// code must not pass the symbol itself to a kernel (on the host it names a
// shadow, not device memory): noalloc_staged_address looks up the real
// device address once per device.
static __device__ __align__(256) float g_noalloc_staged[kNoAllocStagedFloats];

cudaError_t noalloc_staged_address(int device, float** ptr) {
    static std::mutex mu;
    static float* addr[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_staged);
        if (e != cudaSuccess) return e;
        addr[device] = static_cast<float*>(p);
    }
    *ptr = addr[device];
    return cudaSuccess;
}

cudaError_t status_word_address(unsigned** ptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_status);
    if (e == cudaSuccess) *ptr = static_cast<unsigned*>(p);
    return e;
}

bool debug_bounds_build() {
#ifdef CS_DEBUG_BOUNDS
    return true;
#else
    return false;
#endif
}

cudaError_t bounds_site_address(unsigned** ptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_bounds_site);
    if (e == cudaSuccess) *ptr = static_cast<unsigned*>(p);
    return e;
}

cudaError_t read_bounds_site(unsigned* site, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(site, g_bounds_site, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_bounds_site, &zero, sizeof(unsigned));
}

cudaError_t launch_selftest_bounds(cudaStream_t stream) {
#ifdef CS_DEBUG_BOUNDS
    selftest_bounds_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
#else
    (void)stream;
    return cudaErrorNotSupported;
#endif
}

cudaError_t read_device_status(unsigned* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned));
}

}  // namespace cs
