// Fused candidate-scoring kernels for GB300 (sm_103a).
//
// Operation (PR #69 "cuda: add a fused candidate-scoring kernel for CLM and
// Kev", opening table and "What is fused, precisely"): per question b,
//   z_k = scale * sim(q_b, c_k) / temperature,  p = softmax_k(z)
// with sim the cosine (each norm clamped at 1e-8) or the plain dot. Each
// candidate row is read once: its dot with q and its squared norm accumulate
// from the same registers. Logits live only in shared memory.
//
// GB300 design (the page's kernel was one 1024-thread block per question on
// sm_89; none of that is kept beyond "softmax in shared memory"):
//   * stream_kernel -- a warp-specialised CTA: one elected thread issues 1-D
//     bulk copies (cp.async.bulk, TMA engine) of whole candidate rows into a
//     ring of shared-memory stages tracked by mbarriers. Stage g (up to 8
//     rows) belongs to consumer warp g % 8, which computes the dots and
//     squared norms of all its rows from float4 shared loads against q held
//     in registers, then reduces them together with one transposed butterfly
//     of warp shuffles. The per-row cosine and the softmax run later, one
//     lane per row, in the warp that finishes the question.
//       - STREAM plan: persistent, one CTA per SM, each CTA streams a
//         contiguous run of questions, prefetching the next question while a
//         single warp finishes the previous question's softmax.
//       - CLUSTER plan: one thread-block cluster (up to 16 CTAs) per
//         question, the K rows striped over the CTAs; each CTA reduces its
//         rows to (local max, local sum) and the CTAs combine them through
//         distributed shared memory, so a single question uses 16 SMs.
//   * generic_kernel -- scalar loads, any D and any alignment.
// Every on-chip wait is bounded (about 1 s); a CTA that gives up sets a
// device status bit, writes NaN where it could not finish, waits (bounded)
// for its own copies in flight, and exits.
#include "internal.h"

#include <math.h>

namespace cs {

__device__ unsigned int g_status;

namespace {

constexpr float kEps = 1e-8f;                       // norm clamp of the cosine
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s

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

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ float2 ld_peer_f2(const void* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ void consumer_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

// ------------------------------------------------------------------ helpers

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
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* give_up) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*give_up) return false;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*give_up) return false;
        if ((it & 31u) == 0 && globaltimer() - t0 > kWaitLimitNs) {
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

__device__ __forceinline__ float logit_of(float t, float n, float qn, float scale, float temperature, bool cos) {
    float sim = cos ? t / (qn * fmaxf(sqrtf(n), kEps)) : t;
    return scale * sim / temperature;
}

// Logits of rows lane, lane+32, ... (< n) from their dot t and squared norm
// n_sq; -inf beyond n.
template <bool COS>
__device__ __forceinline__ void load_logits(const float* t, const float* n_sq, int n, float qn, float scale,
                                            float temperature, int lane, float (&z)[kLogitSlots / 32]) {
#pragma unroll
    for (int j = 0; j < kLogitSlots / 32; ++j) {
        const int k = lane + 32 * j;
        z[j] = k < n ? logit_of(t[k], COS ? n_sq[k] : 0.f, qn, scale, temperature, COS) : -INFINITY;
    }
}

// Softmax of z over one warp (rows lane + 32 j < n), written to dst[0..n).
__device__ __forceinline__ void softmax_store(float (&z)[kLogitSlots / 32], int n, float* __restrict__ dst,
                                              int lane) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kLogitSlots / 32; ++j) m = fmaxf(m, z[j]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kLogitSlots / 32; ++j) {
        const int k = lane + 32 * j;
        z[j] = k < n ? expf(z[j] - m) : 0.f;
        s += z[j];
    }
    s = warp_sum(s);
#pragma unroll
    for (int j = 0; j < kLogitSlots / 32; ++j) {
        const int k = lane + 32 * j;
        if (k < n) dst[k] = z[j] / s;
    }
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

// ------------------------------------------------------------------ stream kernel

struct StreamArgs {
    Problem p;
    int rows_per_stage;  // R <= kMaxRowsPerStage
    int stages;          // NS
    int cluster;         // G: CTAs per question (1 = STREAM plan)
};

// Dots (and squared norms) of the nr <= kMaxRowsPerStage rows of one stage.
// Lane handles float4 columns lane, lane+32, ...; q comes from registers
// (NQ4 > 0) or from shared memory (NQ4 == 0, large D). Accumulators v hold
// t_r at v[VPR*r] and, for the cosine, the squared norm at v[VPR*r + 1].
template <int NQ4, bool COS>
__device__ __forceinline__ void stage_dots(const float4* __restrict__ st, int nr, int D4, const float4 (&qv)[NQ4 > 0 ? NQ4 : 1],
                                           const float4* __restrict__ q4, int lane,
                                           float (&v)[(COS ? 2 : 1) * kMaxRowsPerStage]) {
    constexpr int VPR = COS ? 2 : 1;
#pragma unroll
    for (int i = 0; i < VPR * kMaxRowsPerStage; ++i) v[i] = 0.f;
    if constexpr (NQ4 > 0) {
#pragma unroll
        for (int j = 0; j < NQ4; ++j) {
            const int i = lane + 32 * j;
            if (i < D4) {
                const float4 q = qv[j];
#pragma unroll
                for (int r = 0; r < kMaxRowsPerStage; ++r) {
                    if (r < nr) {
                        const float4 c = st[r * D4 + i];
                        float t = v[VPR * r];
                        t = fmaf(c.x, q.x, t);
                        t = fmaf(c.y, q.y, t);
                        t = fmaf(c.z, q.z, t);
                        t = fmaf(c.w, q.w, t);
                        v[VPR * r] = t;
                        if (COS) {
                            float n = v[VPR * r + 1];
                            n = fmaf(c.x, c.x, n);
                            n = fmaf(c.y, c.y, n);
                            n = fmaf(c.z, c.z, n);
                            n = fmaf(c.w, c.w, n);
                            v[VPR * r + 1] = n;
                        }
                    }
                }
            }
        }
    } else {
        for (int i = lane; i < D4; i += 32) {
            const float4 q = q4[i];
#pragma unroll
            for (int r = 0; r < kMaxRowsPerStage; ++r) {
                if (r < nr) {
                    const float4 c = st[r * D4 + i];
                    float t = v[VPR * r];
                    t = fmaf(c.x, q.x, t);
                    t = fmaf(c.y, q.y, t);
                    t = fmaf(c.z, q.z, t);
                    t = fmaf(c.w, q.w, t);
                    v[VPR * r] = t;
                    if (COS) {
                        float n = v[VPR * r + 1];
                        n = fmaf(c.x, c.x, n);
                        n = fmaf(c.y, c.y, n);
                        n = fmaf(c.z, c.z, n);
                        n = fmaf(c.w, c.w, n);
                        v[VPR * r + 1] = n;
                    }
                }
            }
        }
    }
}

template <int NQ4, bool COS>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(const StreamArgs args) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int VPR = COS ? 2 : 1;
    constexpr int V = VPR * kMaxRowsPerStage;
    const Problem& p = args.p;
    const int K = p.K, D = p.D, D4 = p.D >> 2;
    const int R = args.rows_per_stage, NS = args.stages, G = args.cluster;
    const SmemLayout L = smem_layout(NS, R, D);
    float* ring = reinterpret_cast<float*>(smem + L.ring);
    float* qbuf = reinterpret_cast<float*>(smem + L.qbuf);
    float* tn = reinterpret_cast<float*>(smem + L.tn);
    float2* xch = reinterpret_cast<float2*>(smem + L.xch);
    volatile int* give_up = reinterpret_cast<volatile int*>(smem + L.flag);
    const uint32_t full0 = smem_u32(smem + L.bars);
    const uint32_t empty0 = full0 + 8u * NS;
    const uint32_t qfull0 = empty0 + 8u * NS;
    const uint32_t qempty0 = qfull0 + 16u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The ring must hold whole rounds of consumer warps (slot s is always
    // owned by warp s % kConsumerWarps) and a stage at most kMaxRowsPerStage
    // rows; the host plans it so. Every CTA sees the same arguments, so a bad
    // plan makes every CTA of every cluster leave here, before any barrier.
    if (NS < kConsumerWarps || NS % kConsumerWarps != 0 || R < 1 || R > kMaxRowsPerStage || 2 * NS + 4 > kStreamThreads) {
        if (threadIdx.x == 0) atomicOr(&g_status, 2u);
        return;
    }

    // Barrier set-up, one barrier per thread: full[s] and empty[s] complete
    // once per use of stage slot s (one producer arrival + the copy's bytes;
    // one arrival of the owning consumer warp), qfull/qempty per q slot.
    {
        const int t = threadIdx.x;
        bool did = false;
        if (t < 2 * NS) {
            mbar_init(full0 + 8u * t, 1);
            did = true;
        } else if (t < 2 * NS + 2) {
            mbar_init(qfull0 + 8u * (t - 2 * NS), 1);
            did = true;
        } else if (t < 2 * NS + 4) {
            mbar_init(qempty0 + 8u * (t - 2 * NS - 2), kConsumerWarps);
            did = true;
        }
        if (t == 0) *give_up = 0;
        if (did) fence_mbar_init();
    }
    __syncthreads();

    // Questions [qb, qe) and candidate rows [klo, khi) of this CTA.
    long long qb, qe;
    int klo, khi;
    if (G > 1) {
        const int rank = static_cast<int>(cluster_ctarank());
        qb = blockIdx.y;
        qe = qb + 1;
        klo = rank * K / G;
        khi = (rank + 1) * K / G;
    } else {
        qb = static_cast<long long>(blockIdx.x) * p.B / gridDim.x;
        qe = static_cast<long long>(blockIdx.x + 1) * p.B / gridDim.x;
        klo = 0;
        khi = K;
    }
    const int nrows = khi - klo;
    const int nst = (nrows + R - 1) / R;
    const uint32_t row_bytes = static_cast<uint32_t>(D) * 4u;
    float qn = 1.f;  // clamped query norm of the current question (cosine)

    if (warp == kConsumerWarps) {
        // ---------------- producer: one elected thread issues every copy
        if (lane == 0) {
            uint32_t gst = 0;
            long long nq = 0;
            for (long long b = qb; b < qe; ++b, ++nq) {
                const uint32_t qs = static_cast<uint32_t>(nq & 1), qpar = static_cast<uint32_t>((nq >> 1) & 1);
                if (!wait_phase(qempty0 + 8u * qs, qpar ^ 1u, give_up)) break;
                mbar_arrive_expect_tx(qfull0 + 8u * qs, row_bytes);
                bulk_g2s(smem_u32(qbuf + qs * D), p.Q + static_cast<size_t>(b) * D, row_bytes, qfull0 + 8u * qs);
                bool stop = false;
                for (int s = 0; s < nst; ++s, ++gst) {
                    const uint32_t slot = gst % NS, par = (gst / NS) & 1u;
                    if (!wait_phase(empty0 + 8u * slot, par ^ 1u, give_up)) { stop = true; break; }
                    const int k0 = klo + s * R;
                    const int nr = min(R, khi - k0);
                    const uint32_t bytes = static_cast<uint32_t>(nr) * row_bytes;
                    mbar_arrive_expect_tx(full0 + 8u * slot, bytes);
                    bulk_g2s(smem_u32(ring + static_cast<size_t>(slot) * R * D),
                             p.C + (static_cast<size_t>(b) * K + k0) * D, bytes, full0 + 8u * slot);
                }
                if (stop) { ++nq; break; }
            }
            if (*give_up) {
                // Let this CTA's copies in flight land before it exits.
                const unsigned long long deadline = globaltimer() + kWaitLimitNs;
                const uint32_t last = gst < static_cast<uint32_t>(NS) ? gst : static_cast<uint32_t>(NS);
                for (uint32_t u = gst - last; u < gst; ++u)
                    wait_phase_until(full0 + 8u * (u % NS), (u / NS) & 1u, deadline);
                const long long qlast = nq < 2 ? nq : 2;
                for (long long u = nq - qlast; u < nq; ++u)
                    wait_phase_until(qfull0 + 8u * static_cast<uint32_t>(u & 1),
                                     static_cast<uint32_t>((u >> 1) & 1), deadline);
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers: stage gst belongs to warp gst % kConsumerWarps
        uint32_t gst = 0;
        long long nq = 0;
        for (long long b = qb; b < qe; ++b, ++nq) {
            const uint32_t qs = static_cast<uint32_t>(nq & 1), qpar = static_cast<uint32_t>((nq >> 1) & 1);
            bool good = wait_phase(qfull0 + 8u * qs, qpar, give_up);
            const float4* q4 = reinterpret_cast<const float4*>(qbuf + qs * D);
            float4 qv[NQ4 > 0 ? NQ4 : 1];
            if constexpr (NQ4 > 0) {
                float sq = 0.f;
#pragma unroll
                for (int j = 0; j < NQ4; ++j) {
                    const int i = lane + 32 * j;
                    qv[j] = i < D4 ? q4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                    if (COS) sq += qv[j].x * qv[j].x + qv[j].y * qv[j].y + qv[j].z * qv[j].z + qv[j].w * qv[j].w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8u * qs);
                // Every warp holds all of q, so this warp-wide sum is the whole
                // norm; it is never added across warps.
                if (COS) qn = fmaxf(sqrtf(warp_sum(sq)), kEps);
            } else if (COS) {
                float sq = 0.f;
                for (int i = lane; i < D4; i += 32) {
                    const float4 x = q4[i];
                    sq += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                }
                qn = fmaxf(sqrtf(warp_sum(sq)), kEps);
            }

            float* tb = tn + (nq & 1) * 2 * kLogitSlots;  // dots
            float* nb = tb + kLogitSlots;                 // squared norms
            for (int s = 0; s < nst; ++s, ++gst) {
                if (static_cast<int>(gst % kConsumerWarps) != warp) continue;
                const uint32_t slot = gst % NS, par = (gst / NS) & 1u;
                const bool ok = wait_phase(full0 + 8u * slot, par, give_up) && good;
                const int k0 = s * R;  // relative to klo
                const int nr = min(R, nrows - k0);
                float v[V];
                stage_dots<NQ4, COS>(reinterpret_cast<const float4*>(ring + static_cast<size_t>(slot) * R * D), nr, D4,
                                     qv, q4, lane, v);
                int idx;
                const float sum = transpose_reduce<V>(v, lane, &idx);
                if ((lane & (32 / V - 1)) == 0) {
                    const int r = idx / VPR;
                    if (r < nr) (VPR == 2 && (idx & 1) ? nb : tb)[k0 + r] = ok ? sum : __int_as_float(0x7fc00000);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8u * slot);
            }
            if constexpr (NQ4 == 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8u * qs);
            }
            consumer_bar_sync();  // every row of question b has its dot (and norm)
            if (G == 1 && warp == static_cast<int>(nq % kConsumerWarps)) {
                float z[kLogitSlots / 32];
                load_logits<COS>(tb, nb, nrows, qn, p.scale, p.temperature, lane, z);
                softmax_store(z, nrows, p.out + static_cast<size_t>(b) * K, lane);
            }
        }
    }

    if (G > 1) {
        // Cluster plan: one question per cluster; combine (local max, local
        // sum of exp) of every CTA through distributed shared memory.
        float z[kLogitSlots / 32];
        if (warp == 0) {
            load_logits<COS>(tn, tn + kLogitSlots, nrows, qn, p.scale, p.temperature, lane, z);
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < kLogitSlots / 32; ++j) m = fmaxf(m, z[j]);
            m = warp_max(m);
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < kLogitSlots / 32; ++j)
                if (lane + 32 * j < nrows) s += expf(z[j] - m);
            s = warp_sum(s);
            if (lane == 0) *xch = make_float2(m, s);
        }
        __syncwarp();
        cluster_sync_all();  // every CTA's (m, s) is visible cluster-wide
        if (warp == 0) {
            float mj = -INFINITY, sj = 0.f;
            if (lane < G) {
                const float2 x = ld_peer_f2(xch, static_cast<uint32_t>(lane));
                mj = x.x;
                sj = x.y;
            }
            const float M = warp_max(mj);
            const float S = warp_sum(lane < G ? sj * expf(mj - M) : 0.f);
            float* dst = p.out + static_cast<size_t>(qb) * K + klo;
#pragma unroll
            for (int j = 0; j < kLogitSlots / 32; ++j) {
                const int k = lane + 32 * j;
                if (k < nrows) dst[k] = expf(z[j] - M) / S;
            }
        }
        __syncwarp();
        cluster_sync_all();  // no CTA leaves while a peer may still read its xch
    }
}

// ------------------------------------------------------------------ generic kernel

// One CTA per question, one warp per candidate row, scalar coalesced loads:
// any D, any alignment.
template <bool COS>
__global__ void __launch_bounds__(kGenericThreads) generic_kernel(const Problem p) {
    __shared__ float lg[kLogitSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = kGenericThreads / 32;
    const long long b = blockIdx.x;
    const int K = p.K, D = p.D;
    const float* __restrict__ q = p.Q + static_cast<size_t>(b) * D;
    float qn = 1.f;
    if (COS) {
        float sq = 0.f;
        for (int d = lane; d < D; d += 32) {
            const float v = __ldg(q + d);
            sq = fmaf(v, v, sq);
        }
        qn = fmaxf(sqrtf(warp_sum(sq)), kEps);  // whole norm per warp, never summed across warps
    }
    for (int k = warp; k < K; k += nwarps) {
        const float* __restrict__ c = p.C + (static_cast<size_t>(b) * K + k) * D;
        float t0 = 0.f, t1 = 0.f, n0 = 0.f, n1 = 0.f;
        int d = lane;
        for (; d + 32 < D; d += 64) {
            const float c0 = __ldg(c + d), c1 = __ldg(c + d + 32);
            t0 = fmaf(c0, __ldg(q + d), t0);
            t1 = fmaf(c1, __ldg(q + d + 32), t1);
            if (COS) {
                n0 = fmaf(c0, c0, n0);
                n1 = fmaf(c1, c1, n1);
            }
        }
        if (d < D) {
            const float c0 = __ldg(c + d);
            t0 = fmaf(c0, __ldg(q + d), t0);
            if (COS) n0 = fmaf(c0, c0, n0);
        }
        const float t = warp_sum(t0 + t1);
        const float n = COS ? warp_sum(n0 + n1) : 0.f;
        if (lane == 0) lg[k] = logit_of(t, n, qn, p.scale, p.temperature, COS);
    }
    __syncthreads();
    if (warp == 0) {
        float z[kLogitSlots / 32];
#pragma unroll
        for (int j = 0; j < kLogitSlots / 32; ++j) z[j] = lane + 32 * j < K ? lg[lane + 32 * j] : -INFINITY;
        softmax_store(z, K, p.out + static_cast<size_t>(b) * K, lane);
    }
}

// ------------------------------------------------------------------ dispatch

template <int NQ4, bool COS>
cudaError_t launch_stream_t(const StreamArgs& a, const Plan& plan, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    if (plan.kind == kPlanCluster) {
        cfg.gridDim = dim3(static_cast<unsigned>(plan.cluster), static_cast<unsigned>(a.p.B), 1);
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(plan.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    } else {
        cfg.gridDim = dim3(static_cast<unsigned>(plan.ctas), 1, 1);
        cfg.attrs = nullptr;
        cfg.numAttrs = 0;
    }
    return cudaLaunchKernelEx(&cfg, stream_kernel<NQ4, COS>, a);
}

template <bool COS>
cudaError_t launch_stream_c(const StreamArgs& a, const Plan& plan, cudaStream_t stream) {
    switch (plan.nq4) {
        case 1: return launch_stream_t<1, COS>(a, plan, stream);
        case 2: return launch_stream_t<2, COS>(a, plan, stream);
        case 4: return launch_stream_t<4, COS>(a, plan, stream);
        case 8: return launch_stream_t<8, COS>(a, plan, stream);
        case 0: return launch_stream_t<0, COS>(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int NQ4, bool COS>
const void* stream_fn() {
    return reinterpret_cast<const void*>(stream_kernel<NQ4, COS>);
}

const void* stream_fn_for(int nq4, int normalize) {
    if (normalize) {
        switch (nq4) {
            case 1: return stream_fn<1, true>();
            case 2: return stream_fn<2, true>();
            case 4: return stream_fn<4, true>();
            case 8: return stream_fn<8, true>();
            case 0: return stream_fn<0, true>();
        }
    } else {
        switch (nq4) {
            case 1: return stream_fn<1, false>();
            case 2: return stream_fn<2, false>();
            case 4: return stream_fn<4, false>();
            case 8: return stream_fn<8, false>();
            case 0: return stream_fn<0, false>();
        }
    }
    return nullptr;
}

}  // namespace

cudaError_t launch_stream(const Problem& p, const Plan& plan, cudaStream_t stream) {
    StreamArgs a;
    a.p = p;
    a.rows_per_stage = plan.rows_per_stage;
    a.stages = plan.stages;
    a.cluster = plan.kind == kPlanCluster ? plan.cluster : 1;
    return p.normalize ? launch_stream_c<true>(a, plan, stream) : launch_stream_c<false>(a, plan, stream);
}

cudaError_t launch_generic(const Problem& p, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(p.B)), block(kGenericThreads);
    if (p.normalize)
        generic_kernel<true><<<grid, block, 0, stream>>>(p);
    else
        generic_kernel<false><<<grid, block, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t configure_device_kernels(int smem_optin) {
    const int nq4s[5] = {1, 2, 4, 8, 0};
    for (int c = 0; c < 2; ++c) {
        for (int i = 0; i < 5; ++i) {
            const void* f = stream_fn_for(nq4s[i], c);
            cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

int max_active_clusters(int cluster, size_t smem, int nq4, int normalize) {
    const void* f = stream_fn_for(nq4, normalize);
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

cudaError_t read_device_status(unsigned* flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_status, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned));
}

}  // namespace cs
