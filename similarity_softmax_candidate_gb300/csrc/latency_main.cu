// cs_latency: microseconds per call of the C ABI for one shape, measured
// from native code (no Python between calls), the way a C or C++ caller
// would see it.
//
//   cs_latency <B> <K> <D> <normalize> <calls> [unfused]
//
// Prints one line of JSON, every figure the mean over at least `calls`
// calls (so the timer's resolution is far below it):
//   direct_warm_us    back-to-back calls on the same inputs (L2-warm)
//   direct_cold_us    back-to-back calls, each on its own slice of an input
//                     pool of at least 512 MiB, so every call reads from HBM
//   graph_warm_us     50 calls on the same inputs captured in one graph
//   graph_cold_us     a graph of a read-only L2 flush (a 256 MiB read) and 50
//                     calls on distinct slices, minus a graph of the flush
//                     alone, per call: back-to-back calls reading from HBM
//   isolated_cold_us  as graph_cold_us, with an empty kernel before each
//                     call, minus the same graph without the calls: a call
//                     that starts only when the GPU is otherwise idle (no
//                     overlap with a previous kernel) and reads from HBM
// Inputs are N(0,1)-like values from a fixed integer hash, filled on the
// device. A read-only flush leaves clean lines, so no write-back of
// earlier data lands inside a timed call.
#include "candidate_scoring.h"

#include <cuda_runtime.h>

#include <cstdio>
#include <algorithm>
#include <cstdlib>

namespace {

__global__ void fill_kernel(float* x, size_t n, unsigned seed) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        unsigned h = (unsigned)i * 2654435761u ^ seed;
        h ^= h >> 15;
        h *= 2246822519u;
        h ^= h >> 13;
        x[i] = ((h & 0xffffff) / 16777216.0f - 0.5f) * 3.4641f;  // uniform, unit variance
    }
}

// Reads n floats (evicting whatever L2 held with clean lines); writes only
// if their sum is exactly `never`, which keeps the reads from being removed.
__global__ void flush_read_kernel(const float4* x, size_t n4, float never, float* sink) {
    float acc = 0.f;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = x[i];
        acc += v.x + v.y + v.z + v.w;
    }
    if (acc == never) *sink = acc;
}

__global__ void empty_kernel() {}

#define CHECK(x)                                                                            \
    do {                                                                                    \
        cudaError_t e_ = (x);                                                               \
        if (e_ != cudaSuccess) {                                                            \
            std::fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));            \
            std::exit(2);                                                                   \
        }                                                                                   \
    } while (0)

}  // namespace

int main(int argc, char** argv) {
    if (argc < 6) {
        std::fprintf(stderr, "usage: %s B K D normalize calls [unfused]\n", argv[0]);
        return 1;
    }
    const int B = std::atoi(argv[1]), K = std::atoi(argv[2]), D = std::atoi(argv[3]);
    const int normalize = std::atoi(argv[4]), calls = std::atoi(argv[5]);
    const bool unfused = argc > 6 && std::atoi(argv[6]) != 0;
    if (B < 1 || K < 1 || D < 1 || calls < 1) return 1;
    const float scale = normalize ? 14.285714f : 0.0625f, temperature = 1.0f;

    // One slice = one call's Q, C, out and staged; slices are 256-byte
    // aligned within one pool of at least 512 MiB.
    auto round256 = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t q_b = round256(sizeof(float) * (size_t)B * D), c_b = round256(sizeof(float) * (size_t)B * K * D),
                 o_b = round256(sizeof(float) * (size_t)B * K);
    const size_t slice_b = q_b + c_b + 2 * o_b;
    const size_t pool_min = (size_t)512 << 20;
    const size_t nslices = std::max<size_t>(64, (pool_min + slice_b - 1) / slice_b);
    const int kGraphCalls = 50;
    if (nslices < (size_t)kGraphCalls) return 1;
    char* pool;
    CHECK(cudaMalloc(&pool, slice_b * nslices));
    fill_kernel<<<2048, 256>>>(reinterpret_cast<float*>(pool), slice_b * nslices / sizeof(float), 2u);
    const size_t flush_n = (size_t)256 << 20 >> 2;  // 256 MiB of floats, about twice the L2
    float *flush, *sink;
    CHECK(cudaMalloc(&flush, flush_n * sizeof(float)));
    CHECK(cudaMalloc(&sink, sizeof(float)));
    fill_kernel<<<1024, 256>>>(flush, flush_n, 7u);
    CHECK(cudaDeviceSynchronize());
    cudaStream_t s;
    CHECK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    cs_stream_t cs = reinterpret_cast<cs_stream_t>(s);
    int sms = 0;
    CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));

    auto call = [&](size_t slice) -> int {
        char* b = pool + slice * slice_b;
        const float* Q = reinterpret_cast<const float*>(b);
        const float* C = reinterpret_cast<const float*>(b + q_b);
        float* out = reinterpret_cast<float*>(b + q_b + c_b);
        float* staged = reinterpret_cast<float*>(b + q_b + c_b + o_b);
        if (unfused) return cs_score_candidates_batch_unfused(Q, C, B, K, D, normalize, scale, temperature, staged, out, cs);
        if (B == 1) return cs_score_candidates(Q, C, K, D, normalize, scale, temperature, out, cs);
        return cs_score_candidates_batch(Q, C, B, K, D, normalize, scale, temperature, out, cs);
    };
    auto flush_l2 = [&] {
        flush_read_kernel<<<4 * sms, 512, 0, s>>>(reinterpret_cast<const float4*>(flush), flush_n / 4, -1.2345e30f,
                                                  sink);
    };
    for (int i = 0; i < 20; ++i)
        if (call(0) != CS_OK) {
            std::fprintf(stderr, "call failed\n");
            return 3;
        }
    CHECK(cudaStreamSynchronize(s));

    cudaEvent_t a, b;
    CHECK(cudaEventCreate(&a));
    CHECK(cudaEventCreate(&b));
    // mean ms of body() over 5 repetitions, the best repetition
    auto time_ms = [&](auto&& body) {
        float best = 1e30f;
        for (int rep = 0; rep < 5; ++rep) {
            CHECK(cudaEventRecord(a, s));
            body();
            CHECK(cudaEventRecord(b, s));
            CHECK(cudaEventSynchronize(b));
            float ms = 0.f;
            CHECK(cudaEventElapsedTime(&ms, a, b));
            if (ms < best) best = ms;
        }
        return best;
    };

    const float direct_warm = 1e3f * time_ms([&] { for (int i = 0; i < calls; ++i) call(0); }) / calls;
    const float direct_cold = 1e3f * time_ms([&] { for (int i = 0; i < calls; ++i) call(i % nslices); }) / calls;

    // Graphs: kinds 0 = 50 calls on slice 0; 1 = flush + 50 calls on slices
    // 1..50; 2 = flush alone; 3 = flush + 50 x (empty, call); 4 = flush +
    // 50 x empty.
    auto make_graph = [&](int kind, cudaGraphExec_t* exec) {
        cudaGraph_t g;
        CHECK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
        if (kind != 0) flush_l2();
        for (int i = 0; i < kGraphCalls; ++i) {
            if (kind >= 3) empty_kernel<<<1, 32, 0, s>>>();
            if (kind == 0) call(0);
            if (kind == 1 || kind == 3) call(1 + (size_t)i);
        }
        CHECK(cudaStreamEndCapture(s, &g));
        CHECK(cudaGraphInstantiate(exec, g, 0));
        CHECK(cudaGraphDestroy(g));
    };
    cudaGraphExec_t gx[5];
    for (int k = 0; k < 5; ++k) make_graph(k, &gx[k]);
    for (int i = 0; i < 3; ++i)
        for (int k = 0; k < 5; ++k) CHECK(cudaGraphLaunch(gx[k], s));
    CHECK(cudaStreamSynchronize(s));
    const int reps = calls / kGraphCalls > 0 ? calls / kGraphCalls : 1;
    float t[5];
    for (int k = 0; k < 5; ++k)
        t[k] = time_ms([&] { for (int i = 0; i < reps; ++i) cudaGraphLaunch(gx[k], s); });
    const float per = 1e3f / (reps * kGraphCalls);
    const float graph_warm = t[0] * per, graph_cold = (t[1] - t[2]) * per, isolated_cold = (t[3] - t[4]) * per;
    CHECK(cudaGetLastError());

    std::printf("{\"B\": %d, \"K\": %d, \"D\": %d, \"normalize\": %d, \"unfused\": %d, \"calls\": %d, "
                "\"slices\": %zu, \"pool_mib\": %.1f, \"direct_warm_us\": %.3f, \"direct_cold_us\": %.3f, "
                "\"graph_warm_us\": %.3f, \"graph_cold_us\": %.3f, \"isolated_cold_us\": %.3f, "
                "\"flush_us\": %.3f, \"empty_kernel_us\": %.3f}\n",
                B, K, D, normalize, unfused ? 1 : 0, reps * kGraphCalls, nslices,
                slice_b * (double)nslices / (1 << 20), direct_warm, direct_cold, graph_warm, graph_cold,
                isolated_cold, 1e3f * t[2] / reps, (t[4] - t[2]) * per);
    for (int k = 0; k < 5; ++k) cudaGraphExecDestroy(gx[k]);
    cudaFree(pool);
    cudaFree(flush);
    cudaFree(sink);
    return 0;
}
