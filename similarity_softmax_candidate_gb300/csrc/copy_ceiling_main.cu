// cs_copy_ceiling: the practical read ceiling of the streaming kernel's
// access pattern on this GPU, measured with the same geometry and no
// arithmetic.
//
//   cs_copy_ceiling [total_bytes] [stage_bytes] [stages] [lanes] [launches]
//
// One CTA per SM streams its own contiguous share of a device buffer into a
// shared-memory ring of `stages` slots of `stage_bytes` with 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier per slot); `lanes`
// issuing lanes each own the slots l, l + lanes, ... and a consumer lane per
// slot frees it as soon as its copy has landed. The buffer is streamed as
// `launches` back-to-back launches over consecutive slices. Defaults: the
// throughput workload's 8.6 GB, 12 KB stages (6 rows of 512 float32), 16
// stages, 8 lanes, 1 launch -- the stream plan's ring.
//
// Prints one line of JSON with the median GB/s of 5 timed repetitions
// (CUDA events, after 3 warm-up repetitions). Every wait is bounded (1 s);
// a wait that gives up sets a flag, the kernel returns, and the program
// exits with status 3.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

namespace {

__device__ unsigned g_gave_up;

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool phase_done(uint32_t bar, uint32_t parity) {
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

// Wait for a phase until `deadline`; on giving up, raise the CTA's flag.
__device__ bool wait_until(uint32_t bar, uint32_t parity, unsigned long long deadline, volatile int* stop) {
    while (!phase_done(bar, parity)) {
        if (*stop) return false;
        if (now_ns() > deadline) {
            *stop = 1;
            atomicOr(&g_gave_up, 1u);
            return false;
        }
    }
    return true;
}

__global__ void ring_stream(const unsigned char* src, long long per_cta, int stage_bytes, int stages, int lanes) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm);  // [stages]
    uint64_t* empty = full + stages;                   // [stages]
    volatile int* stop = reinterpret_cast<volatile int*>(empty + stages);
    unsigned char* ring = sm + 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * stages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(full + i)));
        *stop = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const unsigned long long deadline = now_ns() + 1000000000ull;
    const unsigned char* base = src + static_cast<long long>(blockIdx.x) * per_cta;
    const long long n = per_cta / stage_bytes;
    if (warp == 0 && lane < lanes) {
        long long issued = 0;
        for (long long g = lane; g < n; g += lanes, ++issued) {
            const uint32_t slot = static_cast<uint32_t>(g % stages), use = static_cast<uint32_t>(g / stages);
            if (use > 0 && !wait_until(saddr(empty + slot), (use - 1) & 1u, deadline, stop)) break;
            const uint32_t fb = saddr(full + slot);
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(stage_bytes)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    saddr(ring + static_cast<size_t>(slot) * stage_bytes)),
                "l"(base + g * stage_bytes), "r"(stage_bytes), "r"(fb)
                : "memory");
        }
        // the copies this lane still has in flight land before the CTA leaves
        const unsigned long long d2 = now_ns() + 1000000000ull;
        const long long per_lane = stages / lanes;
        for (long long m = issued > per_lane ? issued - per_lane : 0; m < issued; ++m) {
            const long long g = lane + static_cast<long long>(lanes) * m;
            const uint32_t slot = static_cast<uint32_t>(g % stages), use = static_cast<uint32_t>(g / stages);
            while (!phase_done(saddr(full + slot), use & 1u) && now_ns() < d2) {
            }
        }
    } else if (warp == 1 && lane < lanes) {
        for (long long g = lane; g < n; g += lanes) {
            const uint32_t slot = static_cast<uint32_t>(g % stages), use = static_cast<uint32_t>(g / stages);
            if (!wait_until(saddr(full + slot), use & 1u, deadline, stop)) break;
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(empty + slot)) : "memory");
        }
    }
}

#define CHECK(x)                                                                 \
    do {                                                                         \
        cudaError_t e_ = (x);                                                    \
        if (e_ != cudaSuccess) {                                                 \
            std::fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_)); \
            std::exit(2);                                                        \
        }                                                                        \
    } while (0)

}  // namespace

int main(int argc, char** argv) {
    const long long total_req = argc > 1 ? std::atoll(argv[1]) : 8606646272ll;
    const int stage_bytes = argc > 2 ? std::atoi(argv[2]) : 12288;
    const int stages = argc > 3 ? std::atoi(argv[3]) : 16;
    const int lanes = argc > 4 ? std::atoi(argv[4]) : 8;
    const int launches = argc > 5 ? std::atoi(argv[5]) : 1;
    int dev = 0, sms = 0, max_smem = 0;
    CHECK(cudaGetDevice(&dev));
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CHECK(cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    // At least 120 KB of shared memory, so that one CTA runs per SM.
    const int smem = std::max(1024 + stages * stage_bytes, 120 * 1024);
    if (stage_bytes <= 0 || stage_bytes % 16 != 0 || stages < 1 || lanes < 1 || lanes > 32 ||
        stages % lanes != 0 || 2 * stages * 8 + 4 > 1024 || smem > max_smem || launches < 1 ||
        total_req <= 0) {
        std::fprintf(stderr, "bad arguments (stage_bytes %% 16, stages %% lanes, ring fits %d bytes)\n", max_smem);
        return 1;
    }
    // Each launch gives every CTA a whole number of stages.
    const long long unit = static_cast<long long>(sms) * stage_bytes * launches;
    const long long total = total_req / unit * unit;
    if (total == 0) {
        std::fprintf(stderr, "total_bytes too small for this geometry\n");
        return 1;
    }
    const long long per_launch = total / launches, per_cta = per_launch / sms;
    unsigned char* buf = nullptr;
    CHECK(cudaMalloc(&buf, static_cast<size_t>(total)));
    CHECK(cudaMemset(buf, 0, static_cast<size_t>(total)));
    CHECK(cudaFuncSetAttribute(ring_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    auto pass = [&]() {
        for (int l = 0; l < launches; ++l)
            ring_stream<<<sms, 64, smem>>>(buf + l * per_launch, per_cta, stage_bytes, stages, lanes);
    };
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    for (int i = 0; i < 3; ++i) pass();
    CHECK(cudaGetLastError());
    CHECK(cudaDeviceSynchronize());
    std::vector<double> gbs;
    for (int r = 0; r < 5; ++r) {
        CHECK(cudaEventRecord(e0));
        for (int i = 0; i < 3; ++i) pass();
        CHECK(cudaEventRecord(e1));
        CHECK(cudaEventSynchronize(e1));
        float ms = 0.f;
        CHECK(cudaEventElapsedTime(&ms, e0, e1));
        gbs.push_back(3.0 * static_cast<double>(total) / (ms * 1e-3) / 1e9);
    }
    std::sort(gbs.begin(), gbs.end());
    unsigned gave_up = 0;
    CHECK(cudaMemcpyFromSymbol(&gave_up, g_gave_up, sizeof(gave_up)));
    std::printf(
        "{\"gbs\": %.1f, \"gbs_min\": %.1f, \"gbs_max\": %.1f, \"total_bytes\": %lld, \"stage_bytes\": %d, "
        "\"stages\": %d, \"lanes\": %d, \"launches\": %d, \"ctas\": %d}\n",
        gbs[2], gbs[0], gbs[4], total, stage_bytes, stages, lanes, launches, sms);
    CHECK(cudaFree(buf));
    return gave_up ? 3 : 0;
}
