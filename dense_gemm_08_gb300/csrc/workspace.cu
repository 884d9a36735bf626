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
// kernels keeps the second one from starting as the first drains.
//
// Streams are told apart by the stream's unique id (cudaStreamGetId), not
// by the handle value: cudaStreamPerThread is one handle value for every
// host thread but a different stream in each, and the legacy default stream
// has two handle values (0 and cudaStreamLegacy).
//
// A call holds its stream's entry from SplitSync::acquire until the launch
// is enqueued (SplitSync::release).  So a buffer that a stream outgrows is
// freed in stream order (cudaFreeAsync) after every launch that was given
// it, and any number of host threads may call on one stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <memory>
#include <mutex>
#include <unordered_map>
#include <utility>
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

cudaError_t pool_of(int dev, cudaMemPool_t *out) {
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

cudaError_t device_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return pool_of(dev, out);
}

cudaError_t pool_alloc(size_t bytes, cudaStream_t stream, void **ptr) {
    cudaMemPool_t pool = nullptr;
    cudaError_t e = device_pool(&pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream);
}

}  // namespace

cudaError_t workspace_alloc(size_t bytes, cudaStream_t stream, void **ptr) {
    // under stream capture the allocation becomes a graph memory node, which
    // comes from the graph's own memory, not from a pool of the library
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &capture);
    if (e != cudaSuccess) return e;
    if (capture != cudaStreamCaptureStatusNone) return cudaMallocAsync(ptr, bytes, stream);
    return pool_alloc(bytes, stream, ptr);
}

cudaError_t workspace_free(void *ptr, cudaStream_t stream) { return cudaFreeAsync(ptr, stream); }

namespace {
struct SyncBuf {
    std::mutex m;  // held by a call from acquire until its launch is enqueued
    int dev = 0;
    int *counters = nullptr;
    size_t n_counters = 0;
};

struct KeyHash {
    size_t operator()(const std::pair<int, unsigned long long> &k) const {
        return std::hash<unsigned long long>()(k.second * 0x9E3779B97F4A7C15ull ^
                                               static_cast<unsigned long long>(k.first));
    }
};

// Entries are created on a stream's first split call and never erased (an
// entry is a few words; its buffers are freed by split_sync_release_device).
std::mutex g_map_mutex;
std::unordered_map<std::pair<int, unsigned long long>, std::unique_ptr<SyncBuf>, KeyHash> g_sync;

// Buffer sizes grow in steps of 16 words (64 bytes): a stream holds about
// what its largest split call needed (at most a few KiB).
constexpr size_t kWords = 16;

// A zeroed buffer of at least `want` words, allocated from the pool and
// cleared on `stream`.  The outgrown buffer is freed on `stream`: every
// launch that was given it was enqueued on `stream` before this call (the
// entry is held from acquire to enqueue), so the free runs after them.
template <typename T>
cudaError_t ensure(T **ptr, size_t *have, size_t want, cudaStream_t stream) {
    if (*have >= want) return cudaSuccess;
    const size_t n = (want + kWords - 1) / kWords * kWords;
    void *fresh = nullptr;
    cudaError_t e = pool_alloc(n * sizeof(T), stream, &fresh);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(fresh, 0, n * sizeof(T), stream);
    if (e != cudaSuccess) {
        cudaFreeAsync(fresh, stream);
        return e;
    }
    T *old = *ptr;
    *ptr = static_cast<T *>(fresh);
    *have = n;
    return old != nullptr ? cudaFreeAsync(old, stream) : cudaSuccess;
}

// Frees the buffers of every entry of `dev` after the device has finished
// all work (the caller holds g_map_mutex).  Entries are locked first, so no
// call can enqueue a launch with these counters meanwhile.
cudaError_t release_device_locked(int dev) {
    std::vector<std::unique_lock<std::mutex>> held;
    for (auto &kv : g_sync)
        if (kv.first.first == dev) held.emplace_back(kv.second->m);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    for (auto &kv : g_sync) {
        SyncBuf &b = *kv.second;
        if (b.dev != dev) continue;
        if (b.counters != nullptr) {
            const cudaError_t ef = cudaFreeAsync(b.counters, cudaStreamLegacy);
            if (e == cudaSuccess) e = ef;
        }
        b.counters = nullptr;
        b.n_counters = 0;
    }
    const cudaError_t es = cudaStreamSynchronize(cudaStreamLegacy);
    return e != cudaSuccess ? e : es;
}
}  // namespace

cudaError_t SplitSync::acquire(cudaStream_t stream, size_t n_counters) {
    stream_ = stream;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &capture);
    if (e != cudaSuccess) return e;
    if (capture != cudaStreamCaptureStatusNone) {
        // one zeroed block of counters per captured launch
        size_t bytes = n_counters * sizeof(int);
        if (bytes == 0) bytes = 16;
        void *blk = nullptr;
        if ((e = workspace_alloc(bytes, stream, &blk)) != cudaSuccess) return e;
        owned_ = blk;
        if ((e = cudaMemsetAsync(blk, 0, bytes, stream)) != cudaSuccess) return e;
        counters = static_cast<int *>(blk);
        return cudaSuccess;
    }
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    unsigned long long id = 0;
    if ((e = cudaStreamGetId(stream, &id)) != cudaSuccess) return e;
    SyncBuf *b = nullptr;
    {
        std::lock_guard<std::mutex> map_lock(g_map_mutex);
        std::unique_ptr<SyncBuf> &slot = g_sync[{dev, id}];
        if (!slot) {
            slot.reset(new SyncBuf);
            slot->dev = dev;
        }
        b = slot.get();
    }
    lock_ = std::unique_lock<std::mutex>(b->m);
    if ((e = ensure(&b->counters, &b->n_counters, n_counters, stream)) != cudaSuccess) return e;
    counters = b->counters;
    return cudaSuccess;
}

cudaError_t SplitSync::release() {
    cudaError_t e = cudaSuccess;
    if (owned_ != nullptr) {
        e = workspace_free(owned_, stream_);
        owned_ = nullptr;
    }
    if (lock_.owns_lock()) lock_.unlock();
    return e;
}

SplitSync::~SplitSync() { release(); }

cudaError_t split_sync_release_device() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> map_lock(g_map_mutex);
    return release_device_locked(dev);
}

cudaError_t memory_info(MemoryInfo *out) {
    *out = MemoryInfo{};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> map_lock(g_map_mutex);
        for (auto &kv : g_sync) {
            if (kv.first.first != dev) continue;
            std::lock_guard<std::mutex> entry_lock(kv.second->m);
            const SyncBuf &b = *kv.second;
            const uint64_t bytes = b.n_counters * sizeof(int);
            if (bytes == 0) continue;
            ++out->split_streams;
            out->split_bytes += bytes;
        }
    }
    cudaMemPool_t pool = nullptr;
    if ((e = pool_of(dev, &pool)) != cudaSuccess) return e;
    unsigned long long used = 0, reserved = 0;
    if ((e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &used)) != cudaSuccess)
        return e;
    if ((e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &reserved)) !=
        cudaSuccess)
        return e;
    out->pool_used_bytes = used;
    out->pool_reserved_bytes = reserved;
    return cudaSuccess;
}

cudaError_t release_memory() {
    cudaError_t e = split_sync_release_device();
    if (e != cudaSuccess) return e;
    cudaMemPool_t pool = nullptr;
    if ((e = device_pool(&pool)) != cudaSuccess) return e;
    return cudaMemPoolTrimTo(pool, 0);
}

}  // namespace gemm
