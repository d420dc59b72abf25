// Caller-side projections on the tensor cores, fused with the scoring.
//
// PR #69 "cuda: add a fused candidate-scoring kernel for CLM and Kev" (its
// opening table) scores projected vectors: CLM compares state_head(s) with
// action_head(c), Kev k(h_opts) with q(h_decide); the page leaves those
// projections to the caller. Here they run on the 5th-generation tensor
// cores and the candidate projection feeds the scoring directly from the
// accumulators, so the projected candidates never reach global memory:
//
//   proj_kernel<PLAIN>: P = H W^T, float32 rows written out (the queries).
//   proj_kernel<SCORE>: per question b, the K projected candidate rows
//     c_k = W h_k live only in tensor memory; each becomes its dot with q_b
//     and its squared norm, then a logit, and the question's softmax is
//     written as in the plain scoring path.
//
// H and W are bfloat16, K-major (a row of H and a row of W are both Din
// contiguous elements); accumulation is float32.
//
// GB300 structure: one CTA per SM, 6 warps. The work is cut into units of
// 128 rows x 256 output features (one N half of a 128-row tile). Warp 0 (one
// lane) streams, per unit, the 128-row tile of H and the unit's 256 rows of
// W, 64 columns of Din at a time, with 2-D TMA copies (128-byte swizzle) into
// a 4-stage ring tracked by mbarriers. Warp 1 allocates all 512 columns of
// tensor memory as two 256-column accumulators and (one lane) issues
// tcgen05.mma (M=128, N=256, K=16) into them in turn; tcgen05.commit frees a
// ring stage when its MMAs finish and hands a finished accumulator to the
// epilogue. Warps 2-5 (128 threads, each warp the 32 accumulator rows of its
// TMEM lane quarter) read a unit back with tcgen05.ld while the tensor cores
// fill the other accumulator, and either store it or fold it into dot, norm
// and softmax. Every wait is bounded.
#include "internal.h"
#include "softmax_form.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

namespace cs {
namespace {

constexpr int kTileM = 128;        // accumulator rows (TMEM lanes)
constexpr int kTileK = 64;         // Din columns per ring stage: 128 bytes of bf16, one swizzle row
constexpr int kMmaN = 256;         // N of one tcgen05.mma
constexpr int kMmaK = 16;          // K of one tcgen05.mma (bf16)
// Ring stages of 48 KB.
constexpr int kProjStages = 4;
constexpr int kAccCols = 2 * kMmaN;  // two accumulators of kMmaN columns: all of tensor memory
constexpr int kProjThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpiThreads = 128;
constexpr unsigned long long kProjWaitNs = 1000000000ull;

enum ProjMode { kProjPlain = 0, kProjScore = 1 };

struct ProjArgs {
    long long rows;     // rows of A (PLAIN: rows to project; SCORE: B*K)
    int B, K, Din, D;   // SCORE: B questions of K rows
    int normalize;
    float w0, kexp;     // SCORE: value and exponent scales of the logit factor (softmax_form.cuh)
    const float* qproj; // SCORE: projected queries [B][D]
    float* out;         // PLAIN: [rows][D]; SCORE: [B][K]
    unsigned* status;   // device status word
    unsigned* bounds;   // bounds word (first failing check of a bounds-checked build)
};

#ifdef CS_DEBUG_BOUNDS
// [ptr, ptr + bytes) inside [base, base + extent)? Otherwise record the site
// (first one only) and the status bit, and tell the caller to skip.
__device__ __noinline__ bool check_range(const void* ptr, unsigned long long bytes, const void* base,
                                         unsigned long long extent, unsigned site, unsigned* bounds,
                                         unsigned* status) {
    const unsigned long long x = reinterpret_cast<unsigned long long>(ptr);
    const unsigned long long b = reinterpret_cast<unsigned long long>(base);
    if (x >= b && bytes <= extent && x - b <= extent - bytes) return true;
    atomicCAS(bounds, 0u, site);
    atomicOr(status, kDevErrBounds);
    return false;
}
#define CS_IN_BOUNDS(ptr, bytes, base, extent, site)                                                        \
    check_range((ptr), static_cast<unsigned long long>(bytes), (base), static_cast<unsigned long long>(extent), \
                (site), a.bounds, a.status)
#else
#define CS_IN_BOUNDS(ptr, bytes, base, extent, site) true
#endif

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void bar_init(uint32_t b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool bar_try(uint32_t b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(b), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait; false once this CTA has given up.
__device__ __forceinline__ bool wait_bar(uint32_t b, uint32_t parity, volatile int* give_up, unsigned* status) {
    if (bar_try(b, parity)) return true;
    if (*give_up) return false;
    const unsigned long long t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (bar_try(b, parity)) return true;
        if (*give_up) return false;
        if ((it & 31u) == 0 && gtimer() - t0 > kProjWaitNs) {
            *give_up = 1;
            atomicOr(status, 1u);
            return false;
        }
    }
}
__device__ __forceinline__ void wait_bar_until(uint32_t b, uint32_t parity, unsigned long long deadline) {
    while (!bar_try(b, parity))
        if (gtimer() > deadline) return;
}

// 2-D tiled TMA load: box at (x = column, y = row) of the tensor map.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}


__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for this layout), stride byte offset >> 4 (32-45), version 1
// (46-47), swizzle mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: D float32 (bits 4-5 = 1), A and B
// bfloat16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 128 columns of 16 TMEM lanes (taddr's lane the first), as the .16x256b
// shape spreads them: repetition i gives thread t the columns 8 i + 2 (t % 4)
// and + 1 of lanes t / 4 (v[4 i], v[4 i + 1]) and t / 4 + 8 (v[4 i + 2],
// v[4 i + 3]), so a quad of threads holds 8 consecutive columns of a lane.
__device__ __forceinline__ void tmem_ld_16x256b_x16(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x16.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
        "}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
    uint32_t r[128];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
        "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
        "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
        "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
        "}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
          "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
          "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
          "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
          "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
          "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
          "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
          "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
          "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");  // the wait is in the same statement: no use of r can move above it
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory"); }

__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float wmax(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Shared memory, from a 1024-byte aligned base: ring stages (A tile, then
// the unit's kMmaN rows of W), q (D floats) and 2 x 256 logits (scoring
// kernel only), barriers, TMEM address.
struct ProjLayout {
    uint32_t stage_bytes, a_bytes, ring, q, logits, bars, tmem, flag, total;
};
__host__ __device__ inline ProjLayout proj_layout(int D, int mode) {
    ProjLayout L;
    L.a_bytes = kTileM * kTileK * 2;
    L.stage_bytes = L.a_bytes + kMmaN * kTileK * 2;
    L.ring = 0;
    L.q = L.ring + kProjStages * L.stage_bytes;
    L.logits = L.q + (mode == 1 ? static_cast<uint32_t>(D) * 4 : 0u);  // q and logits: scoring kernel only
    L.bars = L.logits + (mode == 1 ? 2u * 256u * 4u : 0u);
    L.tmem = L.bars + (2 * kProjStages + 4) * 8;
    L.flag = L.tmem + 8;
    L.total = L.flag + 8 + 1024;  // + alignment slack for the base
    return L;
}

template <int MODE>
__global__ void __launch_bounds__(kProjThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                const ProjArgs a) {
    extern __shared__ unsigned char smem_raw[];
    const int D = a.D, nk = a.Din / kTileK, nhalf = D / kMmaN;
    const ProjLayout L = proj_layout(D, MODE);
    const uint32_t raw = su32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sm = smem_raw + (base - raw);
    float* qs = reinterpret_cast<float*>(sm + L.q);
    float* logits = reinterpret_cast<float*>(sm + L.logits);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + L.tmem);
    volatile int* give_up = reinterpret_cast<volatile int*>(sm + L.flag);
    // full/empty per ring stage; accf/acce per accumulator (0: columns
    // 0..255, 1: columns 256..511)
    const uint32_t full0 = base + L.bars, empty0 = full0 + 8u * kProjStages;
    const uint32_t accf0 = empty0 + 8u * kProjStages, acce0 = accf0 + 16u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // work items: PLAIN = 128-row tiles; SCORE = questions of ceil(K/128)
    // tiles; each tile is nhalf units of kMmaN output features
    const int tiles_per_item = MODE == kProjScore ? (a.K + kTileM - 1) / kTileM : 1;
    const long long items = MODE == kProjScore ? a.B : (a.rows + kTileM - 1) / kTileM;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kProjStages; ++s) {
            bar_init(full0 + 8u * s, 1);
            bar_init(empty0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(accf0 + 8u * b, 1);
            bar_init(acce0 + 8u * b, kEpiThreads);
        }
        *give_up = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // the whole warp allocates both accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + L.tmem),
                     "r"(static_cast<uint32_t>(kAccCols)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool stop = false;
            for (long long item = blockIdx.x; item < items && !stop; item += gridDim.x) {
                for (int h = 0; h < tiles_per_item && !stop; ++h) {
                    const long long row0 = MODE == kProjScore ? item * a.K + static_cast<long long>(h) * kTileM
                                                              : item * kTileM;
                    for (int n = 0; n < nhalf && !stop; ++n) {
                        for (int kk = 0; kk < nk; ++kk, ++it) {
                            const uint32_t s = it % kProjStages, ph = (it / kProjStages) & 1u;
                            if (it >= kProjStages && !wait_bar(empty0 + 8u * s, ph ^ 1u, give_up, a.status)) {
                                stop = true;
                                break;
                            }
                            const uint32_t st = base + L.ring + s * L.stage_bytes;
                            bar_expect(full0 + 8u * s, L.stage_bytes);
                            tma_2d(st, &tmA, kk * kTileK, static_cast<int>(row0), full0 + 8u * s);
                            tma_2d(st + L.a_bytes, &tmW, kk * kTileK, n * kMmaN, full0 + 8u * s);
                        }
                    }
                }
            }
            if (*give_up) {  // let issued copies land before the CTA leaves
                const unsigned long long dl = gtimer() + kProjWaitNs;
                const uint32_t first = it > kProjStages ? it - kProjStages : 0;
                for (uint32_t u = first; u < it; ++u)
                    wait_bar_until(full0 + 8u * (u % kProjStages), (u / kProjStages) & 1u, dl);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = mma_idesc(kTileM, kMmaN);
            uint32_t it = 0, unit = 0;
            bool stop = false;
            for (long long item = blockIdx.x; item < items && !stop; item += gridDim.x) {
                for (int h = 0; h < tiles_per_item * nhalf && !stop; ++h, ++unit) {
                    const uint32_t acc = unit & 1u;
                    // the epilogue has read this accumulator's previous unit
                    if (unit >= 2 && !wait_bar(acce0 + 8u * acc, ((unit >> 1) & 1u) ^ 1u, give_up, a.status)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    for (int kk = 0; kk < nk; ++kk, ++it) {
                        const uint32_t s = it % kProjStages, ph = (it / kProjStages) & 1u;
                        if (!wait_bar(full0 + 8u * s, ph, give_up, a.status)) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t st = base + L.ring + s * L.stage_bytes;
                        const uint64_t ad = sw128_desc(st), bd = sw128_desc(st + L.a_bytes);
#pragma unroll
                        for (int k = 0; k < kTileK / kMmaK; ++k)  // +32 bytes per K step inside the swizzled row
                            mma_bf16(tmem + acc * kMmaN, ad + 2u * k, bd + 2u * k, idesc, (kk | k) != 0);
                        mma_commit(empty0 + 8u * s);  // stage free once these MMAs are done
                    }
                    if (stop) break;
                    mma_commit(accf0 + 8u * acc);  // the unit's accumulator is complete
                }
            }
            {  // every issued MMA has finished before TMEM is released
                const unsigned long long dl = gtimer() + kProjWaitNs;
                const uint32_t first = it > kProjStages ? it - kProjStages : 0;
                for (uint32_t u = first; u < it; ++u)
                    wait_bar_until(empty0 + 8u * (u % kProjStages), (u / kProjStages) & 1u, dl);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: thread = accumulator row (TMEM lane)
        const int et = threadIdx.x - 64;                  // 0..127
        const int row = 32 * (warp & 3) + lane;           // TMEM lane this warp may read
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        uint32_t unit = 0;
        long long nq = 0;
        for (long long item = blockIdx.x; item < items; item += gridDim.x, ++nq) {
            float w = 1.f;  // SCORE: the question's value scale (softmax_form.cuh)
            float* lg = logits + (nq & 1) * 256;
            if (MODE == kProjScore) {
                const float* q = a.qproj + static_cast<size_t>(item) * D;
                if (CS_IN_BOUNDS(q, D * 4ll, a.qproj, a.B * D * 4ll, kSiteProjQ))
                    for (int i = et; i < D; i += kEpiThreads) qs[i] = q[i];
                epi_bar_sync();
                float sq = 0.f;
                if (a.normalize)
                    for (int i = lane; i < D; i += 32) sq = fmaf(qs[i], qs[i], sq);
                sq = wsum(sq);
                w = form::value_scale(a.w0, sq, a.normalize != 0);
            }
            for (int h = 0; h < tiles_per_item; ++h) {
                float dot = 0.f, nrm = 0.f;
                bool ok = true;
                for (int n = 0; n < nhalf; ++n, ++unit) {
                    const uint32_t acc = unit & 1u;
                    ok = wait_bar(accf0 + 8u * acc, (unit >> 1) & 1u, give_up, a.status) && ok;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kMmaN; c += 128) {
                        const int col = n * kMmaN + c;  // output feature of the chunk's first column
                        if constexpr (MODE == kProjScore) {
                            float v[128];
                            tmem_ld128(lane_addr + acc * kMmaN + static_cast<uint32_t>(c), v);
                            const float4* q4 = reinterpret_cast<const float4*>(qs + col);
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float4 w = q4[j];
                                dot = fmaf(v[4 * j], w.x, dot);
                                dot = fmaf(v[4 * j + 1], w.y, dot);
                                dot = fmaf(v[4 * j + 2], w.z, dot);
                                dot = fmaf(v[4 * j + 3], w.w, dot);
                                nrm = fmaf(v[4 * j], v[4 * j], nrm);
                                nrm = fmaf(v[4 * j + 1], v[4 * j + 1], nrm);
                                nrm = fmaf(v[4 * j + 2], v[4 * j + 2], nrm);
                                nrm = fmaf(v[4 * j + 3], v[4 * j + 3], nrm);
                            }
                        } else {
                            // the warp's 32 lanes as two halves of 16 read with the
                            // .16x256b shape: a quad of threads holds 8 consecutive
                            // columns of a row, so every store instruction writes
                            // whole 32-byte segments of 8 rows straight from registers
#pragma unroll 1
                            for (int hh = 0; hh < 2; ++hh) {
                                float v[64];
                                tmem_ld_16x256b_x16(lane_addr + (static_cast<uint32_t>(16 * hh) << 16) +
                                                        acc * kMmaN + static_cast<uint32_t>(c),
                                                    v);
                                const long long r0 = item * kTileM + 32 * (warp & 3) + 16 * hh + (lane >> 2);
                                float* p0 = a.out + r0 * D + col + 2 * (lane & 3);
                                float* p1 = p0 + 8ll * D;  // row r0 + 8
                                const bool in0 = r0 < a.rows, in1 = r0 + 8 < a.rows;
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    if (in0 && CS_IN_BOUNDS(p0 + 8 * i, 8, a.out, a.rows * D * 4ll, kSiteProjRows))
                                        *reinterpret_cast<float2*>(p0 + 8 * i) =
                                            ok ? make_float2(v[4 * i], v[4 * i + 1]) : make_float2(NAN, NAN);
                                    if (in1 && CS_IN_BOUNDS(p1 + 8 * i, 8, a.out, a.rows * D * 4ll, kSiteProjRows))
                                        *reinterpret_cast<float2*>(p1 + 8 * i) =
                                            ok ? make_float2(v[4 * i + 2], v[4 * i + 3]) : make_float2(NAN, NAN);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    bar_arrive(acce0 + 8u * acc);  // this thread is done with the accumulator
                }
                if (MODE == kProjScore) {
                    const int k = h * kTileM + row;
                    if (k < a.K) {
                        const float v = a.normalize ? form::cos_value(dot, nrm, w) : form::dot_value(dot, w);
                        lg[k] = ok ? v : form::qnan();
                    }
                }
            }
            if (MODE == kProjScore) {
                epi_bar_sync();  // every logit of the question is in lg
                if (warp == 2) {
                    // softmax of the values (softmax_form.cuh); a flagged row
                    // makes the sum NaN, and the question is skipped unscored
                    float z[8];
                    float m = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int k = lane + 32 * j;
                        z[j] = k < a.K ? lg[k] : -INFINITY;
                        m = fmaxf(m, z[j]);
                    }
                    m = wmax(m);
                    float s = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        z[j] = lane + 32 * j < a.K ? form::softmax_term(a.kexp, z[j] - m) : 0.f;
                        s += z[j];
                    }
                    s = wsum(s);
                    const float inv = 1.0f / s;
                    float* dst = a.out + static_cast<size_t>(item) * a.K;
                    if (isnan(s)) {
                        if (lane == 0 && !*give_up) atomicOr(a.status, kDevErrRange);
                    } else if (CS_IN_BOUNDS(dst, a.K * 4ll, a.out, a.B * a.K * 4ll, kSiteProjOut)) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (lane + 32 * j < a.K) dst[lane + 32 * j] = z[j] * inv;
                    }
                }
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(static_cast<uint32_t>(kAccCols)));
}

// ---------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Tensor map of a row-major matrix [rows][cols] with boxes of box_rows x
// box_cols elements and 128-byte swizzle (box_cols x element size = 128
// bytes); loads read rows past the end as zero.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, int elem_bytes, const void* ptr, unsigned long long rows,
              unsigned long long cols, int box_cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<unsigned long long>(elem_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_bf16_map(CUtensorMap* map, const void* ptr, unsigned long long rows, unsigned long long cols, int box_rows) {
    return make_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, rows, cols, kTileK, box_rows);
}

}  // namespace

size_t proj_smem_bytes(int D) {
    const size_t p = proj_layout(D, kProjPlain).total, s = proj_layout(D, kProjScore).total;
    return p > s ? p : s;
}

cudaError_t configure_proj_kernels(int smem_optin) {
    const int plain = static_cast<int>(proj_layout(512, kProjPlain).total);
    const int score = static_cast<int>(proj_layout(512, kProjScore).total);
    if (plain > smem_optin || score > smem_optin) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(proj_kernel<kProjPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, plain);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(proj_kernel<kProjScore>, cudaFuncAttributeMaxDynamicSharedMemorySize, score);
}

cudaError_t launch_project_rows(const uint16_t* H, const uint16_t* W, long long rows, int Din, int D, float* P,
                                int sms, unsigned* status, unsigned* bounds, cudaStream_t stream) {
    CUtensorMap ma, mw;
    if (!make_bf16_map(&ma, H, rows, Din, kTileM) || !make_bf16_map(&mw, W, D, Din, kMmaN))
        return cudaErrorInvalidValue;
    ProjArgs a{};
    a.rows = rows;
    a.Din = Din;
    a.D = D;
    a.out = P;
    a.status = status;
    a.bounds = bounds;
    const long long tiles = (rows + kTileM - 1) / kTileM;
    const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
    proj_kernel<kProjPlain><<<grid, kProjThreads, proj_layout(D, kProjPlain).total, stream>>>(ma, mw, a);
    return cudaGetLastError();
}

cudaError_t launch_project_score(const uint16_t* Hc, const uint16_t* Wc, const float* qproj, int B, int K, int Din,
                                 int D, int normalize, float w0, float kexp, float* out, int sms,
                                 unsigned* status, unsigned* bounds, cudaStream_t stream) {
    CUtensorMap ma, mw;
    const unsigned long long rows = static_cast<unsigned long long>(B) * K;
    if (!make_bf16_map(&ma, Hc, rows, Din, kTileM) || !make_bf16_map(&mw, Wc, D, Din, kMmaN))
        return cudaErrorInvalidValue;
    ProjArgs a{};
    a.rows = static_cast<long long>(rows);
    a.B = B;
    a.K = K;
    a.Din = Din;
    a.D = D;
    a.normalize = normalize;
    a.w0 = w0;
    a.kexp = kexp;
    a.qproj = qproj;
    a.out = out;
    a.status = status;
    a.bounds = bounds;
    const unsigned grid = static_cast<unsigned>(B < sms ? B : sms);
    proj_kernel<kProjScore><<<grid, kProjThreads, proj_layout(D, kProjScore).total, stream>>>(ma, mw, a);
    return cudaGetLastError();
}

}  // namespace cs
