// cs_latency: microseconds per call of the C ABI for one shape, measured
// from native code (no Python between calls), the way a C or C++ caller
// would see it.
//
//   cs_latency <B> <K> <D> <normalize> <calls> [unfused]
//
// Prints one line of JSON: direct_us (back-to-back calls, CUDA events around
// `calls` calls), graph1_us (a one-call graph replayed `calls` times) and
// graph50_us (50 calls captured in one graph, replayed; per call). Inputs are
// N(0,1)-like values from a fixed integer hash, filled on the device.
#include "candidate_scoring.h"

#include <cuda_runtime.h>

#include <cstdio>
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

    float *Q, *C, *out, *staged;
    CHECK(cudaMalloc(&Q, sizeof(float) * (size_t)B * D));
    CHECK(cudaMalloc(&C, sizeof(float) * (size_t)B * K * D));
    CHECK(cudaMalloc(&out, sizeof(float) * (size_t)B * K));
    CHECK(cudaMalloc(&staged, sizeof(float) * (size_t)B * K));
    fill_kernel<<<256, 256>>>(Q, (size_t)B * D, 1u);
    fill_kernel<<<1024, 256>>>(C, (size_t)B * K * D, 2u);
    CHECK(cudaDeviceSynchronize());
    cudaStream_t s;
    CHECK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    cs_stream_t cs = reinterpret_cast<cs_stream_t>(s);

    auto call = [&]() -> int {
        if (unfused) return cs_score_candidates_batch_unfused(Q, C, B, K, D, normalize, scale, temperature, staged, out, cs);
        if (B == 1) return cs_score_candidates(Q, C, K, D, normalize, scale, temperature, out, cs);
        return cs_score_candidates_batch(Q, C, B, K, D, normalize, scale, temperature, out, cs);
    };
    for (int i = 0; i < 20; ++i)
        if (call() != CS_OK) {
            std::fprintf(stderr, "call failed\n");
            return 3;
        }
    CHECK(cudaStreamSynchronize(s));

    cudaEvent_t a, b;
    CHECK(cudaEventCreate(&a));
    CHECK(cudaEventCreate(&b));
    auto time_us = [&](auto&& body, int n) {
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
        return 1e3f * best / n;
    };

    const float direct = time_us([&] { for (int i = 0; i < calls; ++i) call(); }, calls);

    auto make_graph = [&](int n, cudaGraphExec_t* exec) {
        cudaGraph_t g;
        CHECK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
        for (int i = 0; i < n; ++i) call();
        CHECK(cudaStreamEndCapture(s, &g));
        CHECK(cudaGraphInstantiate(exec, g, 0));
        CHECK(cudaGraphDestroy(g));
    };
    cudaGraphExec_t g1, g50;
    make_graph(1, &g1);
    make_graph(50, &g50);
    for (int i = 0; i < 5; ++i) {
        CHECK(cudaGraphLaunch(g1, s));
        CHECK(cudaGraphLaunch(g50, s));
    }
    CHECK(cudaStreamSynchronize(s));
    const float graph1 = time_us([&] { for (int i = 0; i < calls; ++i) cudaGraphLaunch(g1, s); }, calls);
    const int reps50 = calls / 50 > 0 ? calls / 50 : 1;
    const float graph50 = time_us([&] { for (int i = 0; i < reps50; ++i) cudaGraphLaunch(g50, s); }, reps50 * 50);

    std::printf("{\"B\": %d, \"K\": %d, \"D\": %d, \"normalize\": %d, \"unfused\": %d, \"calls\": %d, "
                "\"direct_us\": %.3f, \"graph1_us\": %.3f, \"graph50_us\": %.3f}\n",
                B, K, D, normalize, unfused ? 1 : 0, calls, direct, graph1, graph50);
    cudaGraphExecDestroy(g1);
    cudaGraphExecDestroy(g50);
    cudaFree(Q);
    cudaFree(C);
    cudaFree(out);
    cudaFree(staged);
    return 0;
}
