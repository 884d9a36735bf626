// probe.cu -- FP32 FMA-pipe probe: the CUDA cores with no memory traffic.
//
// The FP32 peak of the roofline is computed from the SM count, 128 FP32
// lanes per SM, 2 FLOPs per FMA and the SM clock ("Worklog: optimising GEMM
// on NVIDIA H100", the speed-of-light estimate of the introduction).  This
// kernel measures what the FMA pipes deliver when nothing else competes for
// issue slots, as a cross-check of that figure.
#include <cuda_runtime.h>

#include "internal.h"

namespace gemm {
namespace {

constexpr int kFmaThreads = 256;
constexpr int kChains = 8;   // independent FMA chains per thread (hide the FMA latency)
constexpr int kUnroll = 16;  // steps per loop trip (keeps loop overhead near 1 %)

__device__ float g_fma_sink;

// Every thread advances kChains values x <- x * a + b for `trips` x kUnroll
// steps (a just below 1, b small: the values stay between 0.8 and 1.1), then
// stores their sum only if it equals a value it cannot reach -- the compiler
// cannot prove that, so no FMA is dropped.
__global__ void __launch_bounds__(kFmaThreads) fma_probe_kernel(int64_t trips) {
    float x[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j)
        x[j] = 1.0f + static_cast<float>(threadIdx.x * kChains + j) * 1.0e-7f;
    const float a = 0.9999999f, b = 1.0e-7f;
    for (int64_t t = 0; t < trips; ++t) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int j = 0; j < kChains; ++j) x[j] = fmaf(x[j], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += x[j];
    if (s == 12345.0f) g_fma_sink = s;
}

int sms_of_current_device() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_fma_probe(int64_t trips, cudaStream_t stream, double *flops) {
    if (trips < 1) return cudaErrorInvalidValue;
    // 8 CTAs of 256 threads per SM: 64 warps, 16 per scheduler
    const int grid = sms_of_current_device() * 8;
    fma_probe_kernel<<<grid, kFmaThreads, 0, stream>>>(trips);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *flops = 2.0 * kChains * kUnroll * static_cast<double>(trips) * grid * kFmaThreads;
    return cudaSuccess;
}

}  // namespace gemm
