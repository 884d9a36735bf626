// internal.h -- what the host dispatcher and the kernel launchers share.
//
// After normalisation every kernel sees D as row-major M x N; op(A) and op(B)
// keep their own storage order, described by whether K is the contiguous
// ("K-major") dimension.
#pragma once

#include <cstdint>
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

// Temporary device workspace from a library-owned, stream-ordered memory pool
// (one per device, kept warm between calls): memory handed out on `stream`
// and returned on `stream` once the kernels enqueued before the free are done.
cudaError_t workspace_alloc(size_t bytes, cudaStream_t stream, void **ptr);
cudaError_t workspace_free(void *ptr, cudaStream_t stream);
// The split kernels' counters and flags for one launch on `stream` (current
// device): at least n_counters ints that are zero and n_flags unsigned flags
// that are below *generation, the number this launch writes to a flag.
//   Eager calls get the stream's persistent buffers and enqueue nothing:
//   every kernel returns the counters it used to zero, and calls on one
//   stream run in order, so they may share them (calls on other streams
//   have their own).  *owned = nullptr.
//   Under stream capture a graph may be replayed on any stream, at the same
//   time as other work, with the generation fixed at capture: the call gets a
//   fresh zeroed block from the pool instead (*owned = its address, generation
//   1), which the caller frees in stream order after its launch.
cudaError_t split_sync(cudaStream_t stream, size_t n_counters, size_t n_flags, int **counters,
                       unsigned **flags, unsigned *generation, void **owned);
// After a bounded wait ran out (counters may be left mid-count): zero every
// stream's counters and flags of the current device (synchronises the device).
cudaError_t split_sync_reset_device();

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

// FP32 CUDA-core path whose split-tile workspace is a fixed file-scope device
// array of kFixedScratchBytes instead of pool memory (nothing is allocated).
constexpr size_t kFixedScratchBytes = size_t(32) << 20;
// Workspace the FP32 CUDA-core path needs for `p` (0 if it splits no tile).
size_t simt_f32_scratch_bytes(const Problem &p);
cudaError_t launch_simt_fixed_scratch(const Problem &p, cudaStream_t stream, const char **name);

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
cudaError_t launch_skinny(const Problem &p, InType in, cudaStream_t stream, const char **name);

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
