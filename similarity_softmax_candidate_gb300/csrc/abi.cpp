// C ABI of the candidate-scoring library: argument validation, plan choice
// and the single kernel launch per call. See include/candidate_scoring.h for
// the contract of every entry point.
//
// Validation follows the rejected-arguments group of PR #69 "cuda: add a
// fused candidate-scoring kernel for CLM and Kev" (section "Verified on
// hardware"): K above 255, K of zero, D of zero, a zero scale, a negative
// temperature and a null query are errors, not answers. It runs before any
// CUDA call, so a rejected call launches nothing and writes nothing.
#include "candidate_scoring.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

namespace {

using cs::Plan;
using cs::Problem;

// Bytes of candidate rows per bulk-copy stage the planner aims for, and the
// most stages per ring.
constexpr int kStageTargetBytes = 16384;
constexpr int kMaxStages = 32;
// Per-CTA candidate bytes below which splitting a question further over a
// cluster stops paying.
constexpr long long kSplitMinBytes = 16384;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int smem_optin = 0;
    bool proj_ready = false;      // tensor-core projection kernels configured
    unsigned* status = nullptr;   // device address of the status word
    unsigned* bounds = nullptr;   // device address of the bounds word
    std::map<std::pair<int, long long>, int> clusters;  // (cluster, smem|nq4|cos) -> max active
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// The logit factor a = scale / temperature, formed in double precision and
// split into the value scale w0 and exponent scale kexp of softmax_form.cuh
// (both rounded once to float32). Returns CS_ERR_RANGE for |a| > 2^126:
// the form needs kexp finite, and the exact softmax of such logits is an
// argmax that float32 similarities cannot settle anyway. A factor too small
// for float32 gives kexp = 0, which scores every candidate alike, as the
// exact softmax does to within far less than 1e-4.
constexpr double kLog2e = 1.44269504088896340736;  // log2(e)
constexpr double kMaxFactor = 85070591730234615865843651857942052864.0;  // 2^126
constexpr double kHalveBelow = 7.88860905221011805411728565283e-31;    // 2^-100

int logit_form(float scale, float temperature, int normalize, float* w0, float* kexp) {
    const double a = static_cast<double>(scale) / static_cast<double>(temperature);
    const double mag = std::fabs(a);
    if (!(mag <= kMaxFactor)) return CS_ERR_RANGE;
    // the dot halves its values under a tiny factor, so that the difference
    // of two dots stays finite where the factor would not shrink it to 0
    const double w = (!normalize && mag < kHalveBelow) ? 0.5 : 1.0;
    if (w0) *w0 = static_cast<float>(a < 0 ? -w : w);
    if (kexp) *kexp = static_cast<float>(mag * kLog2e / w);
    return CS_OK;
}

// out == nullptr with has_out == false validates everything but the output.
int validate(const float* Q, const void* C, long long B, int K, int D, int normalize, const float* out,
             bool has_out, bool check_scalars, float scale, float temperature, int c_bytes = 4) {
    if (!Q || !C || (has_out && !out)) return CS_ERR_NULL_POINTER;
    if (B <= 0) return CS_ERR_BAD_BATCH;
    if (K <= 0) return CS_ERR_K_ZERO;
    if (K > CS_MAX_K) return CS_ERR_K_TOO_LARGE;
    if (D <= 0) return CS_ERR_D_ZERO;
    if (normalize != 0 && normalize != 1) return CS_ERR_BAD_SIMILARITY;
    if (check_scalars) {
        if (!std::isfinite(scale) || scale == 0.0f) return CS_ERR_BAD_SCALE;
        if (!std::isfinite(temperature) || !(temperature > 0.0f)) return CS_ERR_BAD_TEMPERATURE;
        const int r = logit_form(scale, temperature, normalize, nullptr, nullptr);
        if (r != CS_OK) return r;
    }
    // Elements are read as float32 (bfloat16 for C in the _bf16 entry
    // points): pointers must be aligned to them.
    if ((reinterpret_cast<uintptr_t>(Q) & 3u) || (reinterpret_cast<uintptr_t>(C) & (c_bytes - 1)) ||
        (has_out && (reinterpret_cast<uintptr_t>(out) & 3u)))
        return CS_ERR_MISALIGNED;
    // B*K*D elements, as bytes, must fit comfortably in 64 bits.
    const unsigned long long bk = static_cast<unsigned long long>(B) * static_cast<unsigned long long>(K);
    if (bk > (1ull << 60) / static_cast<unsigned long long>(D)) return CS_ERR_TOO_LARGE;
    if (has_out) {
        const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + bk * 4ull;
        const uintptr_t q0 = reinterpret_cast<uintptr_t>(Q),
                        q1 = q0 + static_cast<unsigned long long>(B) * static_cast<unsigned long long>(D) * 4ull;
        const uintptr_t c0 = reinterpret_cast<uintptr_t>(C),
                        c1 = c0 + bk * static_cast<unsigned long long>(D) * static_cast<unsigned long long>(c_bytes);
        if ((o0 < q1 && q0 < o1) || (o0 < c1 && c0 < o1)) return CS_ERR_ALIAS;
    }
    return CS_OK;
}

// Per-device facts and one-time kernel attributes. Returns a CUDA error.
cudaError_t device_state(DeviceState** st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cs::configure_device_kernels(d.smem_optin);
        if (e != cudaSuccess) return e;
        e = cs::status_word_address(&d.status);
        if (e != cudaSuccess) return e;
        e = cs::bounds_site_address(&d.bounds);
        if (e != cudaSuccess) return e;
        d.proj_ready = cs::configure_proj_kernels(d.smem_optin) == cudaSuccess;
        (void)cudaGetLastError();
        d.ready = true;
    }
    *st = &d;
    return cudaSuccess;
}

int cached_direct_clusters(DeviceState& d, int cluster, int nq4, int normalize, int c_bf16) {
    // nq4 + 16 in bits 2..7 (nq4 is -16, -8, -4, 1, 2, 4 or kDirectWideChunks); bit 62: apart from the stream keys
    const long long key2 = (1ll << 62) | (static_cast<long long>(nq4 + 16) << 2) | (c_bf16 << 1) | normalize;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = d.clusters.find({cluster, key2});
    if (it != d.clusters.end()) return it->second;
    const int n = cs::max_active_direct_clusters(cluster, nq4, normalize, c_bf16);
    d.clusters[{cluster, key2}] = n;
    return n;
}

int cached_generic_clusters(DeviceState& d, int cluster, int normalize, int c_bf16) {
    const long long key2 = (3ll << 61) | (c_bf16 << 1) | normalize;  // apart from the DIRECT and stream keys
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = d.clusters.find({cluster, key2});
    if (it != d.clusters.end()) return it->second;
    const int n = cs::max_active_generic_clusters(cluster, normalize, c_bf16);
    d.clusters[{cluster, key2}] = n;
    return n;
}

int cached_max_clusters(DeviceState& d, int cluster, size_t smem, int nq4, int normalize, int c_bf16, int rows) {
    // nq4 + 16 in bits 2..6 (nq4 is -16, -8, -4, kNqcUnaligned = -1, 0, 1, 2, 4 or 8)
    const long long key2 = (static_cast<long long>(smem) << 12) | (static_cast<long long>(rows) << 8) |
                           (static_cast<long long>(nq4 + 16) << 2) | (c_bf16 << 1) | normalize;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = d.clusters.find({cluster, key2});
    if (it != d.clusters.end()) return it->second;
    const int n = cs::max_active_clusters(cluster, smem, nq4, normalize, c_bf16, rows);
    d.clusters[{cluster, key2}] = n;
    return n;
}

// Bulk copies move whole rows: a row of C and of Q must be a multiple of 16
// bytes and start 16-byte aligned.
bool tma_eligible(const Problem& p) {
    const int per_chunk = 16 / cs::c_elem_bytes(p);
    return (p.D % per_chunk) == 0 && (reinterpret_cast<uintptr_t>(p.Q) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(p.C) % 16) == 0;
}

// 16-byte chunks of a C row each lane handles, when q for them fits in 32
// registers per lane (0: q is read from shared memory instead).
int nq4_for(const Problem& p) {
    const int per_chunk = 16 / cs::c_elem_bytes(p);
    const int dc = p.D / per_chunk;
    const int max_nqc = 32 / per_chunk;  // 8 for float32, 4 for bfloat16
    for (int n = 1; n <= max_nqc; n *= 2)
        if (dc <= 32 * n) return n;
    return 0;
}

// Plan.nq4 for rows the bulk copies take as aligned spans: the unit-wise
// form with the fewest units a lane that covers the row (units: float32
// elements, or whole bfloat16 pairs) with q in registers, else the unit-wise
// form with q in shared memory (kNqcUnaligned).
int unaligned_nq4_for(const Problem& p) {
    const int units = p.c_bf16 ? p.D / 2 : p.D;
    for (int nu : cs::kUnalignedUnits)
        if (units <= 32 * nu) return cs::unaligned_nqc(nu);
    return cs::kNqcUnaligned;
}

// Rows per stage that make a stage of about kStageTargetBytes (1..8).
int stage_rows(long long row_bytes) {
    long long R = kStageTargetBytes / row_bytes;
    if (R < 1) R = 1;
    if (R > cs::kMaxRowsPerStage) R = cs::kMaxRowsPerStage;
    return static_cast<int>(R);
}

// The most stages of R rows of D floats that fit in shared memory, as a
// multiple of the consumer-warp count (at most kMaxStages); 0 if not even
// one stage per consumer warp fits. Stage g lives in slot g % NS and belongs
// to warp g % kConsumerWarps, so with NS a multiple of the warp count every
// slot always has the same owner, which consumes its uses in order: a
// parity wait on a slot can then never see a phase two uses old.
int max_stages(const DeviceState& d, int R, int D, int c_bytes, bool ua) {
    const long long stage_bytes = static_cast<long long>(cs::smem_layout(1, R, D, c_bytes, ua).slot_bytes);
    const size_t fixed = cs::smem_layout(0, R, D, c_bytes, ua).total;
    if (fixed >= static_cast<size_t>(d.smem_optin)) return 0;
    long long ns = static_cast<long long>(d.smem_optin - fixed) / stage_bytes;
    if (ns > kMaxStages) ns = kMaxStages;
    ns -= ns % cs::kConsumerWarps;
    // The barrier array grows by 16 bytes per stage as well.
    while (ns > 0 &&
           cs::smem_layout(static_cast<int>(ns), R, D, c_bytes, ua).total > static_cast<size_t>(d.smem_optin))
        ns -= cs::kConsumerWarps;
    return ns > 0 ? static_cast<int>(ns) : 0;
}

// Ring stages for `need` stages of work: enough for all of it if that fits,
// rounded up to whole rounds of consumer warps.
int ring_stages(long long need, int max_ns) {
    long long ns = (need + cs::kConsumerWarps - 1) / cs::kConsumerWarps * cs::kConsumerWarps;
    return ns < max_ns ? static_cast<int>(ns) : max_ns;
}

// STREAM plan with `ctas` persistent CTAs (0 = one per SM, at most B).
// Picks rows per stage R <= stage_rows(D) that keeps the most bytes in
// flight (larger R on ties). Rows the bulk copies cannot take whole (not
// tma_eligible) are copied as aligned spans (nq4 < 0). Returns
// false if no ring fits.
bool stream_plan(const DeviceState& d, const Problem& p, int ctas, Plan* plan) {
    const int cb = cs::c_elem_bytes(p);
    const bool ua = !tma_eligible(p);
    int R = 0, max_ns = 0;
    long long best = 0;
    for (int r = stage_rows(static_cast<long long>(cb) * p.D); r >= 1; --r) {
        const int ns = max_stages(d, r, p.D, cb, ua);
        const long long bytes = static_cast<long long>(cb) * r * p.D * ns;
        if (bytes > best) {
            best = bytes;
            R = r;
            max_ns = ns;
        }
    }
    if (max_ns == 0) return false;
    if (ctas <= 0) ctas = d.sms;
    if (ctas > p.B) ctas = static_cast<int>(p.B);
    // Stages one CTA ever needs: no point reserving more ring than that.
    const long long qpc = (p.B + ctas - 1) / ctas;
    // Few rows per CTA (one short question): fewer rows per stage, so that
    // every consumer warp gets a stage instead of one warp doing them all.
    if (!p.offsets && qpc * p.K < static_cast<long long>(cs::kConsumerWarps) * R) {
        const int r = static_cast<int>((qpc * p.K + cs::kConsumerWarps - 1) / cs::kConsumerWarps);
        const int ns = max_stages(d, r, p.D, cb, ua);
        if (ns > 0) {
            R = r;
            max_ns = ns;
        }
    }
    const int ns = ring_stages(qpc * ((p.K + R - 1) / R), max_ns);
    plan->kind = cs::kPlanStream;
    plan->cluster = 1;
    plan->ctas = ctas;
    plan->rows_per_stage = R;
    plan->stages = ns;
    plan->nq4 = ua ? unaligned_nq4_for(p) : nq4_for(p);
    plan->smem = cs::smem_layout(ns, R, p.D, cb, ua).total;
    return true;
}

// CLUSTER plan with G CTAs per question: each CTA's rows spread over all
// consumer warps (one stage each) when the ring holds them.
bool cluster_plan(const DeviceState& d, const Problem& p, int G, Plan* plan) {
    const int cb = cs::c_elem_bytes(p);
    const bool ua = !tma_eligible(p);
    const int rows = (p.K + G - 1) / G;
    int R = (rows + cs::kConsumerWarps - 1) / cs::kConsumerWarps;
    const int Rmax = stage_rows(static_cast<long long>(cb) * p.D);
    if (R > Rmax) R = Rmax;
    while (R > 1 && max_stages(d, R, p.D, cb, ua) == 0) --R;  // a ring of 8 stages must fit
    const int max_ns = max_stages(d, R, p.D, cb, ua);
    if (max_ns == 0) return false;
    const int ns = ring_stages((rows + R - 1) / R, max_ns);
    plan->kind = cs::kPlanCluster;
    plan->cluster = G;
    plan->ctas = G * static_cast<int>(p.B);
    plan->rows_per_stage = R;
    plan->stages = ns;
    plan->nq4 = ua ? unaligned_nq4_for(p) : nq4_for(p);
    plan->smem = cs::smem_layout(ns, R, p.D, cb, ua).total;
    return true;
}

// The DIRECT kernel form these rows take: narrow (q in registers, nq4 in
// 1, 2, 4, at most kDirectMaxRows rows per CTA), wide (q in shared memory,
// at most kDirectWideChunks 16-byte chunks of a row per lane, at most
// kDirectWideMaxRows rows per CTA), or for rows the bulk copies cannot take
// whole the 4-byte-unit form (unaligned_nqc, q in registers, at most
// kDirectMaxRows rows per CTA). Returns the plan's nq4 for the form (0: no
// DIRECT form) and the row limit.
int direct_form(const Problem& p, int* max_rows) {
    if (!tma_eligible(p)) {
        // rows in 4-byte units with q in registers (no odd-D bfloat16 form)
        const int nq = unaligned_nq4_for(p);
        if (nq < cs::kNqcUnaligned && !(p.c_bf16 && (p.D & 1))) {
            *max_rows = cs::kDirectMaxRows;
            return nq;
        }
        *max_rows = 0;
        return 0;
    }
    const int nq4 = nq4_for(p);
    if (nq4 == 1 || nq4 == 2 || nq4 == 4) {
        *max_rows = cs::kDirectMaxRows;
        return nq4;
    }
    const long long dc = p.D / (16 / cs::c_elem_bytes(p));
    if (dc <= 32ll * cs::kDirectWideChunks && p.D <= cs::kDirectWideMaxD) {
        *max_rows = cs::kDirectWideMaxRows;
        return cs::kDirectWideChunks;
    }
    *max_rows = 0;
    return 0;
}

// DIRECT plan: G CTAs per question (one CTA if G == 1), each with at most
// the form's row limit of it (a question's longest share for ragged batches
// is ceil(255 / G)).
bool direct_plan(const Problem& p, int G, Plan* plan) {
    int max_rows = 0;
    const int nq4 = direct_form(p, &max_rows);
    if (p.B > 65535 || G < 1 || G > cs::kMaxCluster || G > p.K || nq4 == 0) return false;
    const int kmax = p.offsets ? CS_MAX_K : p.K;
    if ((kmax + G - 1) / G > max_rows) return false;
    plan->kind = cs::kPlanDirect;
    plan->cluster = G;
    plan->ctas = G * static_cast<int>(p.B);
    plan->rows_per_stage = 0;
    plan->stages = 0;
    plan->nq4 = nq4;
    plan->smem = 0;
    return true;
}

// Questions per cluster of the scalar plan for few questions: the largest
// power of two that gives every warp at least one row, every CTA at least
// kSplitMinBytes of rows and keeps all clusters on the GPU at once (1: a CTA
// per question; always 1 for ragged batches).
int generic_cluster_size(DeviceState& d, const Problem& p) {
    if (p.offsets || p.B * 2 > d.sms || p.B > 65535) return 1;
    const long long q_bytes = static_cast<long long>(cs::c_elem_bytes(p)) * p.K * p.D;
    const int warps = cs::kGenericThreads / 32;
    int G = 1;
    while (G * 2 <= cs::kMaxCluster && G * 2 * warps <= p.K && (G * 2) * p.B <= d.sms &&
           q_bytes / (G * 2) >= kSplitMinBytes)
        G *= 2;
    while (G > 1 && cached_generic_clusters(d, G, p.normalize, p.c_bf16) < p.B) G /= 2;
    return G;
}

void generic_plan(const Problem& p, Plan* plan, int G = 1) {
    plan->kind = cs::kPlanGeneric;
    plan->cluster = G;
    plan->ctas = G * static_cast<int>(p.B);
    plan->rows_per_stage = 0;
    plan->stages = 0;
    plan->nq4 = 0;
    plan->smem = 0;
}

// Chooses (or checks a forced) plan. Returns a cs_status. fused: the fused
// readout, which may take the DIRECT plan and copy unaligned rows as aligned
// spans (the unfused baseline's passes may do neither).
int make_plan(DeviceState& d, const Problem& p, int kind, int cluster, int ctas, Plan* plan, bool fused = true) {
    const bool aligned = tma_eligible(p);
    if (kind == cs::kPlanDirect) {
        if (!fused) return CS_ERR_BAD_PLAN;
        if (cluster == 0) {  // fewest CTAs per question that keep each within the row limit
            int max_rows = 0;
            direct_form(p, &max_rows);
            const int kmax = p.offsets ? CS_MAX_K : p.K;
            cluster = 1;
            while (max_rows > 0 && (kmax + cluster - 1) / cluster > max_rows && cluster < cs::kMaxCluster)
                cluster *= 2;
        }
        if (!direct_plan(p, cluster, plan)) return CS_ERR_BAD_PLAN;
        if (cluster > 1 && cached_direct_clusters(d, cluster, plan->nq4, p.normalize, p.c_bf16) < 1)
            return CS_ERR_BAD_PLAN;
        return CS_OK;
    }
    if (kind == cs::kPlanGeneric) {
        if (cluster < 0 || cluster > cs::kMaxCluster) return CS_ERR_BAD_PLAN;
        if (cluster > 1 && (p.offsets || cluster > p.K || p.B > 65535 ||
                            cached_generic_clusters(d, cluster, p.normalize, p.c_bf16) < 1))
            return CS_ERR_BAD_PLAN;
        generic_plan(p, plan, cluster > 1 ? cluster : 1);
        return CS_OK;
    }
    if (kind == cs::kPlanStream) {
        if ((!aligned && !fused) || ctas < 0 || ctas > p.B) return CS_ERR_BAD_PLAN;
        return stream_plan(d, p, ctas, plan) ? CS_OK : CS_ERR_BAD_PLAN;
    }
    if (kind == cs::kPlanCluster) {
        if ((!aligned && !fused) || p.B > 65535 || cluster < 0 || cluster > cs::kMaxCluster || cluster > p.K)
            return CS_ERR_BAD_PLAN;
        if (cluster == 0) {
            cluster = 1;
            while (cluster * 2 <= cs::kMaxCluster && cluster * 2 <= p.K) cluster *= 2;
        }
        if (cluster == 1)  // one CTA per question: the STREAM kernel with B CTAs
            return stream_plan(d, p, static_cast<int>(p.B), plan) ? CS_OK : CS_ERR_BAD_PLAN;
        if (!cluster_plan(d, p, cluster, plan)) return CS_ERR_BAD_PLAN;
        if (cached_max_clusters(d, cluster, plan->smem, plan->nq4, p.normalize, p.c_bf16, plan->rows_per_stage) < 1)
            return CS_ERR_BAD_PLAN;
        return CS_OK;
    }
    // automatic choice
    if (p.B * 2 <= d.sms) {
        // Few questions: split each over a cluster so one question is not
        // confined to one SM (the page's 256-thread lesson, "What it is worth").
        const long long avg_k = p.offsets ? (p.total_rows + p.B - 1) / p.B : p.K;
        const long long q_bytes = static_cast<long long>(cs::c_elem_bytes(p)) * avg_k * p.D;
        int G = 1;
        while (G * 2 <= cs::kMaxCluster && G * 2 <= avg_k && (G * 2) * p.B <= d.sms &&
               q_bytes / (G * 2) >= kSplitMinBytes)
            G *= 2;
        // Short questions (at most kDirectMaxRows rows per CTA): the DIRECT
        // plan, one trip to memory and no ring. The fewest CTAs per question
        // that keep each within the row limit, doubled while the grid stays
        // within half the SMs and each CTA keeps kSplitMinBytes of rows; taken
        // while its clusters run in at most 1.5 waves (the plan sweep on
        // K=255, D=512: 8-CTA clusters beat the cluster plans up to 48
        // questions, 16-CTA ones are best up to 4).
        int max_rows = 0;
        if (fused && direct_form(p, &max_rows) != 0) {
            const int kmax = p.offsets ? CS_MAX_K : p.K;
            int g = 1;
            while ((kmax + g - 1) / g > max_rows && g * 2 <= cs::kMaxCluster && g * 2 <= p.K) g *= 2;
            while (g * 2 <= cs::kMaxCluster && g * 2 <= avg_k && (g * 2) * p.B * 2 <= d.sms &&
                   q_bytes / (g * 2) >= kSplitMinBytes)
                g *= 2;
            if (direct_plan(p, g, plan) &&
                (g == 1 ||
                 3ll * cached_direct_clusters(d, g, plan->nq4, p.normalize, p.c_bf16) >= 2ll * p.B))
                return CS_OK;
        }
        // Otherwise the cluster plans of the stream kernel (rows the bulk
        // copies cannot take whole as aligned spans: one K=255 question of
        // D=2560 one element off in 6.0 us, against 49.6 us on the scalar
        // plan over 16 CTAs).
        for (; (aligned || fused) && G > 1; G /= 2) {
            if (cluster_plan(d, p, G, plan) &&
                cached_max_clusters(d, G, plan->smem, plan->nq4, p.normalize, p.c_bf16, plan->rows_per_stage) >= p.B)
                return CS_OK;
        }
    }
    // A few questions whose rows the bulk copies cannot take whole and
    // neither the DIRECT nor a cluster plan takes: the scalar plan, each
    // question spread over a cluster (latency-bound).
    if (!aligned && p.B * 2 <= d.sms && !p.offsets) {
        generic_plan(p, plan, generic_cluster_size(d, p));
        return CS_OK;
    }
    // Many questions: the bulk-copy stream, aligned rows whole, others as
    // aligned spans (fused readout only: the unfused passes have no
    // unaligned build).
    if ((aligned || fused) && stream_plan(d, p, 0, plan)) return CS_OK;
    // Rows too long for the ring: the scalar plan.
    generic_plan(p, plan, generic_cluster_size(d, p));
    return CS_OK;
}

// The fused readout under `plan`.
int launch_fused(const Problem& p, const Plan& plan, cs_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (plan.kind == cs::kPlanGeneric)
        e = cs::launch_generic(p, plan.cluster, st);
    else if (plan.kind == cs::kPlanDirect)
        e = cs::launch_direct(p, plan, st);
    else
        e = cs::launch_stream(p, plan, p.normalize ? cs::kFusedCos : cs::kFusedDot, st);
    return e == cudaSuccess ? CS_OK : CS_ERR_LAUNCH;
}

int run(const float* Q, const void* C, long long B, int K, int D, int normalize, float scale, float temperature,
        float* out, cs_stream_t stream, int kind, int cluster, int ctas, int c_bf16 = 0) {
    const int v = validate(Q, C, B, K, D, normalize, out, true, true, scale, temperature, c_bf16 ? 2 : 4);
    if (v != CS_OK) return v;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return CS_ERR_LAUNCH;
    Problem p{Q, C, out, B, K, D, normalize, 0.f, 0.f, nullptr, c_bf16, nullptr, 0};
    (void)logit_form(scale, temperature, normalize, &p.w0, &p.kexp);  // validated above
    Plan plan{};
    const int s = make_plan(*d, p, kind, cluster, ctas, &plan);
    if (s != CS_OK) return s;
    return launch_fused(p, plan, stream);
}

bool overlaps(const void* a, unsigned long long abytes, const void* b, unsigned long long bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Ragged batches: question b owns rows offsets[b] .. offsets[b+1]-1 of C and
// of out. The offsets live in device memory, so only what the host knows is
// checked here (B, total_rows, D, pointers, scalars, overlaps); the kernels
// check each question's own offsets.
int run_ragged(const float* Q, const void* C, const long long* offsets, long long B, long long total_rows, int D,
               int normalize, float scale, float temperature, float* out, cs_stream_t stream, int c_bf16) {
    if (!Q || !C || !offsets || !out) return CS_ERR_NULL_POINTER;
    if (B <= 0) return CS_ERR_BAD_BATCH;
    if (total_rows < B) return CS_ERR_K_ZERO;
    if (total_rows > static_cast<long long>(CS_MAX_K) * B) return CS_ERR_K_TOO_LARGE;
    if (D <= 0) return CS_ERR_D_ZERO;
    if (normalize != 0 && normalize != 1) return CS_ERR_BAD_SIMILARITY;
    if (!std::isfinite(scale) || scale == 0.0f) return CS_ERR_BAD_SCALE;
    if (!std::isfinite(temperature) || !(temperature > 0.0f)) return CS_ERR_BAD_TEMPERATURE;
    float w0, kexp;
    if (logit_form(scale, temperature, normalize, &w0, &kexp) != CS_OK) return CS_ERR_RANGE;
    const unsigned long long cb = c_bf16 ? 2ull : 4ull, rows = static_cast<unsigned long long>(total_rows);
    if ((reinterpret_cast<uintptr_t>(Q) & 3u) || (reinterpret_cast<uintptr_t>(C) & (cb - 1)) ||
        (reinterpret_cast<uintptr_t>(out) & 3u) || (reinterpret_cast<uintptr_t>(offsets) & 7u))
        return CS_ERR_MISALIGNED;
    if (rows > (1ull << 60) / static_cast<unsigned long long>(D)) return CS_ERR_TOO_LARGE;
    const unsigned long long out_b = rows * 4ull, q_b = static_cast<unsigned long long>(B) * D * 4ull,
                             c_b = rows * D * cb, o_b = (static_cast<unsigned long long>(B) + 1ull) * 8ull;
    if (overlaps(out, out_b, Q, q_b) || overlaps(out, out_b, C, c_b) || overlaps(out, out_b, offsets, o_b))
        return CS_ERR_ALIAS;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return CS_ERR_LAUNCH;
    Problem p{Q, C, out, B, CS_MAX_K, D, normalize, w0, kexp, nullptr, c_bf16, offsets, total_rows};
    Plan plan{};
    const int s = make_plan(*d, p, cs::kPlanAuto, 0, 0, &plan);
    if (s != CS_OK) return s;
    return launch_fused(p, plan, stream);
}

// The unfused baseline: pass 1 stages one value per row in `staged`, pass 2
// scores from it. Two launches on `stream`.
int run_unfused(const float* Q, const float* C, long long B, int K, int D, int normalize, float scale,
                float temperature, float* staged, float* out, cs_stream_t stream) {
    const int v = validate(Q, C, B, K, D, normalize, out, true, true, scale, temperature);
    if (v != CS_OK) return v;
    if (!staged) return CS_ERR_NULL_POINTER;
    if (reinterpret_cast<uintptr_t>(staged) & 3u) return CS_ERR_MISALIGNED;
    const unsigned long long bk4 = static_cast<unsigned long long>(B) * K * 4ull;
    if (overlaps(staged, bk4, out, bk4) || overlaps(staged, bk4, Q, static_cast<unsigned long long>(B) * D * 4ull) ||
        overlaps(staged, bk4, C, bk4 * static_cast<unsigned long long>(D)))
        return CS_ERR_ALIAS;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return CS_ERR_LAUNCH;
    Problem p{Q, C, out, B, K, D, normalize, 0.f, 0.f, staged, 0, nullptr, 0};
    (void)logit_form(scale, temperature, normalize, &p.w0, &p.kexp);  // validated above
    Plan plan{};
    const int s = make_plan(*d, p, cs::kPlanAuto, 0, 0, &plan, false);
    if (s != CS_OK) return s;
    if (plan.kind == cs::kPlanGeneric) return CS_ERR_BAD_PLAN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cs::launch_stream(p, plan, normalize ? cs::kRowNorm : cs::kRowDot, st);
    if (e == cudaSuccess)
        e = normalize ? cs::launch_stream(p, plan, cs::kStagedCos, st) : cs::launch_staged_softmax(p, st);
    return e == cudaSuccess ? CS_OK : CS_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int cs_abi_version(void) { return 1; }

const char* cs_status_string(int status) {
    switch (status) {
        case CS_OK: return "ok";
        case CS_ERR_NULL_POINTER: return "null pointer (Q, C or out)";
        case CS_ERR_K_ZERO: return "K must be at least 1";
        case CS_ERR_K_TOO_LARGE: return "K exceeds CS_MAX_K (255)";
        case CS_ERR_D_ZERO: return "D must be at least 1";
        case CS_ERR_BAD_SCALE: return "scale must be finite and nonzero";
        case CS_ERR_BAD_TEMPERATURE: return "temperature must be finite and positive";
        case CS_ERR_BAD_BATCH: return "B must be at least 1";
        case CS_ERR_BAD_SIMILARITY: return "normalize must be 0 (dot) or 1 (cosine)";
        case CS_ERR_LAUNCH: return "CUDA launch failed";
        case CS_ERR_ALIAS: return "out overlaps Q or C";
        case CS_ERR_TOO_LARGE: return "B*K*D is too large";
        case CS_ERR_BAD_PLAN: return "requested plan cannot run these arguments";
        case CS_ERR_RANGE: return "|scale / temperature| exceeds 2^126";
        case CS_ERR_MISALIGNED: return "a pointer is not aligned to its element size";
        case CS_ERR_SCRATCH_TOO_SMALL:
            return "B*K exceeds the built-in scratch of the no-allocation entry point (1048576 rows)";
        default: return "unknown status";
    }
}

int cs_score_candidates(const float* q, const float* C, int K, int D, int normalize, float scale, float temperature,
                        float* out, cs_stream_t stream) {
    return run(q, C, 1, K, D, normalize, scale, temperature, out, stream, cs::kPlanAuto, 0, 0);
}

int cs_score_candidates_batch(const float* Q, const float* C, int B, int K, int D, int normalize, float scale,
                              float temperature, float* out, cs_stream_t stream) {
    return run(Q, C, B, K, D, normalize, scale, temperature, out, stream, cs::kPlanAuto, 0, 0);
}

int cs_score_candidates_batch_plan(const float* Q, const float* C, int B, int K, int D, int normalize, float scale,
                                   float temperature, float* out, cs_stream_t stream, int plan, int cluster,
                                   int ctas) {
    if (plan < CS_PLAN_AUTO || plan > CS_PLAN_DIRECT) return CS_ERR_BAD_PLAN;
    return run(Q, C, B, K, D, normalize, scale, temperature, out, stream, plan, cluster, ctas);
}

int cs_score_candidates_batch_unfused(const float* Q, const float* C, int B, int K, int D, int normalize,
                                      float scale, float temperature, float* staged, float* out,
                                      cs_stream_t stream) {
    return run_unfused(Q, C, B, K, D, normalize, scale, temperature, staged, out, stream);
}

int cs_score_candidates_batch_unfused_noalloc(const float* Q, const float* C, int B, int K, int D, int normalize,
                                              float scale, float temperature, float* out, cs_stream_t stream) {
    const int v = validate(Q, C, B, K, D, normalize, out, true, true, scale, temperature);
    if (v != CS_OK) return v;
    if (static_cast<unsigned long long>(B) * static_cast<unsigned long long>(K) > cs::kNoAllocStagedFloats)
        return CS_ERR_SCRATCH_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_LAUNCH;
    float* staged = nullptr;
    if (cs::noalloc_staged_address(dev, &staged) != cudaSuccess) return CS_ERR_LAUNCH;
    return run_unfused(Q, C, B, K, D, normalize, scale, temperature, staged, out, stream);
}

int cs_score_candidates_bf16(const float* q, const uint16_t* C, int K, int D, int normalize, float scale,
                             float temperature, float* out, cs_stream_t stream) {
    return run(q, C, 1, K, D, normalize, scale, temperature, out, stream, cs::kPlanAuto, 0, 0, 1);
}

int cs_score_candidates_batch_bf16(const float* Q, const uint16_t* C, int B, int K, int D, int normalize, float scale,
                                   float temperature, float* out, cs_stream_t stream) {
    return run(Q, C, B, K, D, normalize, scale, temperature, out, stream, cs::kPlanAuto, 0, 0, 1);
}

int cs_score_candidates_ragged(const float* Q, const float* C, const long long* offsets, int B, long long total_rows,
                               int D, int normalize, float scale, float temperature, float* out, cs_stream_t stream) {
    return run_ragged(Q, C, offsets, B, total_rows, D, normalize, scale, temperature, out, stream, 0);
}

int cs_score_candidates_ragged_bf16(const float* Q, const uint16_t* C, const long long* offsets, int B,
                                    long long total_rows, int D, int normalize, float scale, float temperature,
                                    float* out, cs_stream_t stream) {
    return run_ragged(Q, C, offsets, B, total_rows, D, normalize, scale, temperature, out, stream, 1);
}

int cs_query_plan(const float* Q, const float* C, int B, int K, int D, int normalize, int* plan, int* cluster,
                  int* ctas, int* smem_bytes) {
    const int v = validate(Q, C, B, K, D, normalize, nullptr, false, false, 1.f, 1.f);
    if (v != CS_OK) return v;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return CS_ERR_LAUNCH;
    Problem p{Q, C, nullptr, B, K, D, normalize, 1.f, 1.f, nullptr, 0, nullptr, 0};
    Plan pl{};
    const int s = make_plan(*d, p, cs::kPlanAuto, 0, 0, &pl);
    if (s != CS_OK) return s;
    if (plan) *plan = pl.kind;
    if (cluster) *cluster = pl.cluster;
    if (ctas) *ctas = pl.ctas;
    if (smem_bytes) *smem_bytes = static_cast<int>(pl.smem);
    return CS_OK;
}

// Shapes the tensor-core projection kernels take.
int validate_projection(long long rows, int Din, int D) {
    if (rows <= 0 || rows > CS_PROJ_MAX_ROWS) return CS_ERR_BAD_BATCH;
    if (Din <= 0 || D <= 0) return CS_ERR_D_ZERO;
    if (Din % 64 != 0 || (D != 256 && D != 512)) return CS_ERR_BAD_PLAN;
    return CS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cs_project_rows(const uint16_t* H, const uint16_t* W, long long rows, int Din, int D, float* P,
                    cs_stream_t stream) {
    if (!H || !W || !P) return CS_ERR_NULL_POINTER;
    const int v = validate_projection(rows, Din, D);
    if (v != CS_OK) return v;
    if (!aligned16(H) || !aligned16(W) || !aligned16(P)) return CS_ERR_BAD_PLAN;
    const unsigned long long rb = static_cast<unsigned long long>(rows);
    if (overlaps(P, rb * D * 4ull, H, rb * Din * 2ull) || overlaps(P, rb * D * 4ull, W, 2ull * D * Din))
        return CS_ERR_ALIAS;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return CS_ERR_LAUNCH;
    if (!d->proj_ready) return CS_ERR_BAD_PLAN;
    return cs::launch_project_rows(H, W, rows, Din, D, P, d->sms, d->status, d->bounds,
                                   reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? CS_OK
               : CS_ERR_LAUNCH;
}

int cs_project_score_batch(const uint16_t* Hq, const uint16_t* Wq, const uint16_t* Hc, const uint16_t* Wc, int B,
                           int K, int Din, int D, int normalize, float scale, float temperature, float* qproj,
                           float* out, cs_stream_t stream) {
    if (!Hq || !Wq || !Hc || !Wc || !qproj || !out) return CS_ERR_NULL_POINTER;
    if (B <= 0) return CS_ERR_BAD_BATCH;
    if (K <= 0) return CS_ERR_K_ZERO;
    if (K > CS_MAX_K) return CS_ERR_K_TOO_LARGE;
    const int v = validate_projection(static_cast<long long>(B) * K, Din, D);
    if (v != CS_OK) return v;
    if (normalize != 0 && normalize != 1) return CS_ERR_BAD_SIMILARITY;
    if (!std::isfinite(scale) || scale == 0.0f) return CS_ERR_BAD_SCALE;
    if (!std::isfinite(temperature) || !(temperature > 0.0f)) return CS_ERR_BAD_TEMPERATURE;
    float w0, kexp;
    if (logit_form(scale, temperature, normalize, &w0, &kexp) != CS_OK) return CS_ERR_RANGE;
    if (!aligned16(Hq) || !aligned16(Wq) || !aligned16(Hc) || !aligned16(Wc) || !aligned16(qproj))
        return CS_ERR_BAD_PLAN;
    const unsigned long long bk = static_cast<unsigned long long>(B) * K;
    const unsigned long long ob = bk * 4ull, qb = static_cast<unsigned long long>(B) * D * 4ull;
    const void* ins[4] = {Hq, Wq, Hc, Wc};
    const unsigned long long insb[4] = {static_cast<unsigned long long>(B) * Din * 2ull, 2ull * D * Din,
                                        bk * Din * 2ull, 2ull * D * Din};
    for (int i = 0; i < 4; ++i)
        if (overlaps(out, ob, ins[i], insb[i]) || overlaps(qproj, qb, ins[i], insb[i])) return CS_ERR_ALIAS;
    if (overlaps(out, ob, qproj, qb)) return CS_ERR_ALIAS;
    DeviceState* d = nullptr;
    if (device_state(&d) != cudaSuccess) return CS_ERR_LAUNCH;
    if (!d->proj_ready) return CS_ERR_BAD_PLAN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cs::launch_project_rows(Hq, Wq, B, Din, D, qproj, d->sms, d->status, d->bounds, st);
    if (e == cudaSuccess)
        e = cs::launch_project_score(Hc, Wc, qproj, B, K, Din, D, normalize, w0, kexp, out, d->sms, d->status,
                                     d->bounds, st);
    return e == cudaSuccess ? CS_OK : CS_ERR_LAUNCH;
}

int cs_selftest_bounded_wait(int limit_us, cs_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return CS_ERR_BAD_PLAN;
    const cudaError_t e = cs::launch_selftest_wait(static_cast<unsigned long long>(limit_us) * 1000ull,
                                                   reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CS_OK : CS_ERR_LAUNCH;
}

int cs_device_status(unsigned* flags, int clear) {
    if (!flags) return CS_ERR_NULL_POINTER;
    return cs::read_device_status(flags, clear != 0) == cudaSuccess ? CS_OK : CS_ERR_LAUNCH;
}

int cs_debug_bounds_build(void) { return cs::debug_bounds_build() ? 1 : 0; }

int cs_bounds_violation(unsigned* site, int clear) {
    if (!site) return CS_ERR_NULL_POINTER;
    return cs::read_bounds_site(site, clear != 0) == cudaSuccess ? CS_OK : CS_ERR_LAUNCH;
}

int cs_selftest_bounds(cs_stream_t stream) {
    if (!cs::debug_bounds_build()) return CS_ERR_BAD_PLAN;
    return cs::launch_selftest_bounds(reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? CS_OK
                                                                                             : CS_ERR_LAUNCH;
}

}  // extern "C"
