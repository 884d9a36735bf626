// workspace.cu -- the library's stream-ordered workspace pool.
//
// Kernels that split K across CTAs need a temporary buffer for partial sums.
// It comes from one CUDA memory pool per device, created on first use and
// owned by the library (the device's default pool and its settings are left
// alone).  The pool keeps up to kKeepBytes of freed memory so that repeated
// calls do not go back to the driver.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace gemm {
namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kKeepBytes = 256ull << 20;

struct Pool {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    cudaMemPool_t pool = nullptr;
};
Pool g_pools[kMaxDevices];

cudaError_t device_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    Pool &p = g_pools[dev];
    std::call_once(p.once, [&p, dev] {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        p.err = cudaMemPoolCreate(&p.pool, &props);
        if (p.err != cudaSuccess) return;
        unsigned long long keep = kKeepBytes;
        p.err = cudaMemPoolSetAttribute(p.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    });
    *out = p.pool;
    return p.err;
}

}  // namespace

cudaError_t workspace_alloc(size_t bytes, cudaStream_t stream, void **ptr) {
    cudaMemPool_t pool = nullptr;
    const cudaError_t e = device_pool(&pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

cudaError_t workspace_free(void *ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }

}  // namespace gemm
