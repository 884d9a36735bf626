// workspace.cu -- the library's stream-ordered workspace pool, and the
// split kernels' counters.
//
// Kernels that split K across CTAs need a temporary buffer for partial sums.
// It comes from one CUDA memory pool per device, created on first use and
// owned by the library (the device's default pool and its settings are left
// alone).  The pool keeps up to kKeepBytes of freed memory so that repeated
// calls do not go back to the driver.
//
// The same kernels count the pieces of a split tile.  Their counters live in
// one buffer per (device, stream), zeroed once when it is created: every
// kernel leaves the counters it used at zero when it completes (the last
// piece of a tile resets its counter), so calls on a stream need no clearing
// operation between them -- an extra stream operation between two GEMM
// kernels keeps the second one from starting as the first drains.  Flags
// that pieces wait on are compared with a per-stream generation number that
// grows with every call, so they are never cleared either.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <vector>

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
    // under stream capture the allocation becomes a graph memory node, which
    // comes from the graph's own memory, not from a pool of the library
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &capture);
    if (e != cudaSuccess) return e;
    if (capture != cudaStreamCaptureStatusNone) return cudaMallocAsync(ptr, bytes, stream);
    cudaMemPool_t pool = nullptr;
    if ((e = device_pool(&pool)) != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

cudaError_t workspace_free(void *ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }

namespace {
struct SyncBuf {
    int *counters = nullptr;
    size_t n_counters = 0;
    unsigned *flags = nullptr;
    size_t n_flags = 0;
    unsigned generation = 0;
};
std::mutex g_sync_mutex;
std::unordered_map<uint64_t, SyncBuf> g_sync;  // key: (device, stream)
std::vector<void *> g_sync_retired;            // outgrown buffers, never freed

uint64_t sync_key(int dev, cudaStream_t stream) {
    return (static_cast<uint64_t>(dev) << 56) ^ reinterpret_cast<uintptr_t>(stream);
}

// A zeroed buffer of at least `want` words for one of the regions.  An
// outgrown buffer is kept allocated: a launch enqueued by another host thread
// may still hold its address.
template <typename T>
cudaError_t ensure(T **ptr, size_t *have, size_t want, cudaStream_t stream) {
    if (*have >= want) return cudaSuccess;
    size_t n = *have ? *have : 4096;
    while (n < want) n *= 2;
    void *fresh = nullptr;
    cudaError_t e = cudaMalloc(&fresh, n * sizeof(T));
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(fresh, 0, n * sizeof(T), stream);
    if (e != cudaSuccess) {
        cudaFree(fresh);
        return e;
    }
    if (*ptr != nullptr) g_sync_retired.push_back(*ptr);
    *ptr = static_cast<T *>(fresh);
    *have = n;
    return cudaSuccess;
}
}  // namespace

cudaError_t split_sync(cudaStream_t stream, size_t n_counters, size_t n_flags, int **counters,
                       unsigned **flags, unsigned *generation, void **owned) {
    *owned = nullptr;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &capture);
    if (e != cudaSuccess) return e;
    if (capture != cudaStreamCaptureStatusNone) {
        // one zeroed block per captured launch: [counters][flags]
        const size_t c_bytes = (n_counters * sizeof(int) + 15) & ~static_cast<size_t>(15);
        const size_t bytes = c_bytes + n_flags * sizeof(unsigned);
        void *blk = nullptr;
        if ((e = workspace_alloc(bytes > 0 ? bytes : 16, stream, &blk)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(blk, 0, bytes > 0 ? bytes : 16, stream)) != cudaSuccess) {
            workspace_free(blk, stream);
            return e;
        }
        *owned = blk;
        if (counters) *counters = static_cast<int *>(blk);
        if (flags) *flags = reinterpret_cast<unsigned *>(static_cast<char *>(blk) + c_bytes);
        if (generation) *generation = 1;
        return cudaSuccess;
    }
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_sync_mutex);
    SyncBuf &b = g_sync[sync_key(dev, stream)];
    if ((e = ensure(&b.counters, &b.n_counters, n_counters, stream)) != cudaSuccess) return e;
    if ((e = ensure(&b.flags, &b.n_flags, n_flags, stream)) != cudaSuccess) return e;
    if (++b.generation == 0) {
        // after 2^32 calls on one stream: start the flags over from zero
        e = cudaMemsetAsync(b.flags, 0, b.n_flags * sizeof(unsigned), stream);
        if (e != cudaSuccess) return e;
        b.generation = 1;
    }
    if (counters) *counters = b.counters;
    if (flags) *flags = b.flags;
    if (generation) *generation = b.generation;
    return cudaSuccess;
}

cudaError_t split_sync_reset_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_sync_mutex);
    for (auto &kv : g_sync) {
        if (static_cast<int>(kv.first >> 56) != dev) continue;
        SyncBuf &b = kv.second;
        if (b.counters && (e = cudaMemset(b.counters, 0, b.n_counters * sizeof(int))) != cudaSuccess)
            return e;
        if (b.flags && (e = cudaMemset(b.flags, 0, b.n_flags * sizeof(unsigned))) != cudaSuccess)
            return e;
        b.generation = 0;
    }
    return cudaDeviceSynchronize();
}

}  // namespace gemm
