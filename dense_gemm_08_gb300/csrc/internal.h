// internal.h -- what the host dispatcher and the kernel launchers share.
//
// After normalisation every kernel sees D as row-major M x N; op(A) and op(B)
// keep their own storage order, described by whether K is the contiguous
// ("K-major") dimension.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace gemm {

struct Problem {
    int64_t M, N, K;
    float alpha, beta;
    const void *A;
    int64_t lda;
    bool a_kmajor;  // A(i, k) at A[i * lda + k]; else A[i + k * lda]
    const void *B;
    int64_t ldb;
    bool b_kmajor;  // B(k, j) at B[k + j * ldb]; else B[k * ldb + j]
    const float *C;  // read only if beta != 0; row-major, ldc
    int64_t ldc;
    float *D;  // row-major, ldd (holds BF16 bit patterns when d_bf16)
    int64_t ldd;
    // Fused epilogue: D = act(alpha * AB + beta * C + bias), stored as FP32 or
    // BF16.  bias has one value per column of D (per row when bias_per_row).
    const float *bias = nullptr;
    bool bias_per_row = false;
    int act = 0;  // 0 none, 1 ReLU, 2 GELU (tanh form)
    bool d_bf16 = false;
};

enum class InType { F32, BF16, F16 };

// Programmatic dependent launch.  The library's kernels are launched with
// the programmatic-stream-serialization attribute, so a kernel may be
// scheduled while the kernel before it on the stream is still finishing.
// Each kernel does its on-chip set-up, then calls pdl_wait() -- which
// returns once the previous kernel has completed and its memory operations
// are visible -- before it touches global memory, and pdl_launch_dependents()
// to let the next launch be scheduled (its CTAs start as this grid's CTAs
// leave their SMs).  Without a programmatic dependency both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The launch attribute that allows it.
inline void set_pdl_attribute(cudaLaunchAttribute *attr) {
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
}

// Temporary device workspace from a library-owned, stream-ordered memory pool
// (one per device, kept warm between calls): memory handed out on `stream`
// and returned on `stream` once the kernels enqueued before the free are done.
cudaError_t workspace_alloc(size_t bytes, cudaStream_t stream, void **ptr);
cudaError_t workspace_free(void *ptr, cudaStream_t stream);
// The split kernels' counters for one launch on `stream` (current device):
// after acquire, `counters` has at least n_counters ints that are zero.
//   Eager calls get the stream's persistent buffer and enqueue nothing
//   (except when the buffer grows): every kernel returns the counters it used
//   to zero, and calls on one stream run in order, so they may share them
//   (other streams have their own).  The stream's entry stays held until
//   release(), which the caller invokes once its launch is enqueued, so an
//   outgrown buffer is freed after every launch given it, whichever host
//   threads make the calls.
//   Under stream capture a graph may be replayed on any stream, at the same
//   time as other work: the call gets a fresh zeroed block of graph memory
//   instead, freed in stream order by release().
class SplitSync {
   public:
    SplitSync() = default;
    SplitSync(const SplitSync &) = delete;
    SplitSync &operator=(const SplitSync &) = delete;
    ~SplitSync();
    cudaError_t acquire(cudaStream_t stream, size_t n_counters);
    cudaError_t release();
    int *counters = nullptr;

   private:
    cudaStream_t stream_ = nullptr;
    void *owned_ = nullptr;              // captured launch: its block
    std::unique_lock<std::mutex> lock_;  // eager launch: the stream's entry
};
// Frees every stream's split counters on the current device after
// synchronising it (the next split call on a stream creates zeroed ones).
// Used after a bounded wait ran out, when counters may be left mid-count.
cudaError_t split_sync_release_device();

// What the library holds on the current device between calls.
struct MemoryInfo {
    uint64_t split_streams = 0;        // streams with split counters
    uint64_t split_bytes = 0;          // bytes of those counters
    uint64_t pool_used_bytes = 0;      // pool memory in use (counters, pending workspace)
    uint64_t pool_reserved_bytes = 0;  // pool memory held from the driver
};
cudaError_t memory_info(MemoryInfo *out);
// split_sync_release_device, then the pool returns all its free memory.
cudaError_t release_memory();

// Each launcher enqueues one kernel on `stream`, returns the CUDA error of
// the launch and sets *name to the kernel's static name.
cudaError_t launch_simt(const Problem &p, InType in, cudaStream_t stream, const char **name);
cudaError_t launch_scale_c(const Problem &p, cudaStream_t stream, const char **name);

// FP32 problems with few 64 x 64 tiles: each tile's K range split over the
// CTAs of a cluster and reduced through distributed shared memory
// (sgemm_cluster.cu).  sgemm_cluster_size returns the cluster size (2, 4 or
// 8) to use for `p` on a GPU of `sms` SMs, or 0 when the kernel does not fit.
int sgemm_cluster_size(const Problem &p, int sms);
cudaError_t launch_sgemm_cluster(const Problem &p, int cl, cudaStream_t stream,
                                 const char **name);

// Scratch supplied in place of pool memory (gemm_f32_noalloc): `counters`
// holds n_counters ints that are zero between calls (every kernel returns
// the counters it used to zero), `part` holds part_bytes for partial sums.
struct FixedScratch {
    int *counters;
    size_t n_counters;
    void *part;
    size_t part_bytes;
};
// The library's fixed scratch array (sgemm_simt.cu): kFixedScratchBytes in
// all, the first kFixedCounterBytes of it counters, the rest partial sums.
constexpr size_t kFixedScratchBytes = size_t(32) << 20;
constexpr size_t kFixedCounterBytes = size_t(16) << 10;
// The current device's fixed scratch.  The first call on a device looks up
// the array's address and zeroes its counters (waiting for that on
// `stream`); it fails under stream capture.
cudaError_t fixed_scratch(FixedScratch *out, cudaStream_t stream);

// The FP32 path of gemm_f32 (A, B FP32; K > 0, alpha != 0): the small-M
// kernel for M <= kSkinnyMaxM, else the cluster kernel where it fits, else
// the CUDA-core kernel in the tile configuration that suits the shape.
// With `fixed`, the split pieces use it instead of pool memory and the
// stream's counters (the same kernel and work split either way).
cudaError_t launch_f32(const Problem &p, cudaStream_t stream, const char **name,
                       const FixedScratch *fixed = nullptr);
// Scratch launch_f32 takes for `p`: partial-sum bytes and counters (both 0
// when no tile is split).
void f32_scratch_needs(const Problem &p, size_t *part_bytes, size_t *n_counters);

// Tensor-core (tcgen05) path for BF16 or FP16 inputs.  Returns
// cudaErrorNotSupported (without launching) when the operands cannot be
// described by TMA.
bool tc_eligible(const Problem &p);
cudaError_t launch_tc(const Problem &p, InType in, cudaStream_t stream, const char **name);
// Reads and clears the tensor-core kernel's device status word (after a sync).
cudaError_t tc_read_and_clear_status(cudaStream_t stream, int *status);

// GEMMs with at most kSkinnyMaxM rows (after the column-major D
// normalisation): a kernel that streams op(B) once (skinny.cu).
constexpr int64_t kSkinnyMaxM = 8;
bool skinny_eligible(const Problem &p);
cudaError_t launch_skinny(const Problem &p, InType in, cudaStream_t stream, const char **name,
                          const FixedScratch *fixed = nullptr);
void skinny_scratch_needs(const Problem &p, InType in, size_t *part_bytes, size_t *n_counters);

// Peak probes (no memory traffic).  Each enqueues one kernel on `stream` and
// stores the FLOPs it performs in *flops.
//   launch_tc_probe: one CTA per SM (cta_group 1) or one CTA pair per two
//     SMs (cta_group 2) issuing n_mma back-to-back BF16 tcgen05.mma each.
//   launch_fma_probe: 8 CTAs of 256 threads per SM, each thread 8 chains of
//     16 x trips dependent FP32 FMAs.
cudaError_t launch_tc_probe(int cta_group, int64_t n_mma, cudaStream_t stream, double *flops);
cudaError_t launch_fma_probe(int64_t trips, cudaStream_t stream, double *flops);
// One CTA waiting on an mbarrier that nothing completes: its bounded wait
// gives up after timeout_ns and sets the tensor-core status word.
cudaError_t launch_wait_probe(uint64_t timeout_ns, cudaStream_t stream);

}  // namespace gemm
