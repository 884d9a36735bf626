/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Both entry points compute, on the GPU,
 *
 *     D = alpha * op(A) * op(B) + beta * C
 *
 * the general matrix multiplication of "GEMM on NVIDIA GPUs: from naive
 * kernel to tiled pipeline", section 1 "GEMM definition": op(A) is M x K,
 * op(B) is K x N, C and D are M x N, and
 *
 *     D_ij = alpha * sum_{k<K} A_ik * B_kj + beta * C_ij.
 *
 * "op" (identity or transpose) is expressed as the storage order of each
 * operand, which is exactly the BLAS "trans" flag:
 *
 *     GEMM_ROW_MAJOR:  X(r, q) is stored at X[r * ld + q]
 *     GEMM_COL_MAJOR:  X(r, q) is stored at X[r + q * ld]
 *
 * where (r, q) index the LOGICAL matrix: A(i, k), B(k, j), C(i, j), D(i, j).
 * C and D share one order.  Leading dimensions are in elements.
 *
 * Common contract of gemm_f32 and gemm_bf16_f32acc
 * -------------------------------------------------
 * Ownership: A, B, C and D are device pointers owned by the caller (for
 *   example torch CUDA tensors).  The library keeps no pointer after the call
 *   returns; tensor maps travel by value in the launch parameters.
 *   Workspace: a kernel may split the K range of some tiles across CTAs (to
 *   keep every SM busy).  Such a kernel takes a temporary workspace for the
 *   partial sums (a few tens of MiB at most) from a memory pool the library
 *   owns, one per device, allocated and freed in stream order on `stream`.
 *   The pool keeps up to 256 MiB of freed memory for later calls.  Kernels
 *   that split a tile's K range over the CTAs of one thread-block cluster
 *   (small tensor-core and FP32 problems) add the partial sums in the
 *   cluster's shared memory and take neither workspace nor counters.
 *   Split counters: the split pieces count themselves in small counters that
 *   the library keeps per (device, stream) -- streams told apart by their
 *   unique id, so cudaStreamPerThread is a different stream in each host
 *   thread -- and that every kernel returns to zero, so no call clears them.
 *   They take what the largest split call on the stream needed (64 bytes
 *   to a few KiB) and come from the same pool.  A stream's counters that
 *   a larger problem outgrows are freed in stream order.  What a device
 *   holds is reported by gemm_memory_info(); gemm_release_memory() frees it.
 *   Graph capture: while `stream` is being captured, each call takes fresh
 *   counters and workspace as graph memory.  The graph may therefore be
 *   replayed on any stream, beside other calls.
 *   Threads: any number of host threads may call at once, on one stream or
 *   on several.  A call holds its stream's counters from the moment it takes
 *   them until its kernel is enqueued, so calls on one stream are enqueued
 *   one after another.
 * Asynchrony: the work is enqueued on `stream` (0 = the legacy default
 *   stream) and the call returns without waiting for it.  The caller keeps
 *   the buffers alive until the stream has passed the call.
 * Shapes: M, N, K >= 0 and each <= 2^31 - 1, and M * N <= 2^43 (no device
 *   holds a larger D).  M == 0 or N == 0 is a no-op that returns GEMM_OK
 *   without touching any pointer.  K == 0 or alpha == 0 gives
 *   D = beta * C (A and B are not read).
 * beta == 0: C is never read and may be NULL (BLAS convention; C traffic
 *   only counts when beta != 0 in "GEMM on NVIDIA GPUs", section 2, "GEMM
 *   arithmetic intensity").  C == D with the same ldc/ldd is allowed
 *   (in-place update).  Any other overlap of D with A, B or C is undefined.
 * Leading dimensions: lda >= max(1, K) if A is row-major, >= max(1, M) if
 *   column-major; ldb >= max(1, N) row-major / max(1, K) column-major;
 *   ldc, ldd >= max(1, N) row-major / max(1, M) column-major.
 * Alignment: pointers must be aligned to their element size.  Any leading
 *   dimension is accepted; wide loads and TMA are used when pointers and
 *   leading dimensions allow it, narrower guarded accesses otherwise.  This
 *   never changes the result beyond the stated tolerances and is never an
 *   error.
 * Edges: any M, N, K is handled; tiles past the matrix edge read zeros and
 *   never store outside D.
 * Errors: argument errors return synchronously before any launch and leave
 *   D untouched.  A launch failure returns GEMM_ERR_LAUNCH.  A device without
 *   sm_103 support returns GEMM_ERR_UNSUPPORTED_DEVICE (no CPU fallback
 *   exists).  The tensor-core kernel bounds every wait on its pipeline
 *   barriers; if one runs out it records GEMM_ERR_TIMEOUT in a per-device
 *   status word, read by gemm_last_device_status().  Nothing is printed.
 */
#ifndef DENSE_GEMM_08_GB300_GEMM_H
#define DENSE_GEMM_08_GB300_GEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_order_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,     /* bad shape, leading dimension, order, NULL or misaligned pointer */
    GEMM_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not sm_103 */
    GEMM_ERR_LAUNCH = 3,            /* the CUDA runtime refused the launch */
    GEMM_ERR_TIMEOUT = 4,           /* a bounded device-side wait ran out (see gemm_last_device_status) */
    GEMM_ERR_INTERNAL = 5           /* a CUDA runtime or driver call failed (e.g. tensor-map encoding) */
} gemm_status_t;

/* One BF16 number as its raw 16-bit pattern (the upper half of an FP32). */
typedef uint16_t gemm_bf16_t;

/* One IEEE 754 binary16 (FP16) number as its raw 16-bit pattern. */
typedef uint16_t gemm_f16_t;

/*
 * gemm_f32 -- FP32 inputs, FP32 arithmetic on the CUDA cores (no TF32),
 * FP32 output.  The kernel tiles D into CTA tiles staged through shared
 * memory, each thread accumulates an 8 x 8 register block with FP32 FMA
 * ("Worklog: optimising GEMM on NVIDIA H100", kernels 2-6: shared-memory
 * tiling, register tiling, vectorised loads, warp tiling).
 *
 *   M, N, K        logical sizes of op(A) (M x K), op(B) (K x N), C/D (M x N)
 *   alpha, beta    scalars (FP32)
 *   A, lda, order_a   device pointer to op(A)'s storage, its leading dimension, its order
 *   B, ldb, order_b   same for op(B)
 *   C, ldc         device pointer to C (read only if beta != 0), leading dimension
 *   D, ldd         device pointer to D (written), leading dimension
 *   order_cd       storage order of both C and D
 *   stream         CUDA stream the kernel is enqueued on
 *
 * Accuracy: |D - D_ref| <= 1e-5 * sum_k |alpha A_ik B_kj| + 1e-6 * |beta C_ij|
 * against the exact result; bit-exact when every partial sum is an integer
 * below 2^24 and alpha = 1, beta = 0.
 */
gemm_status_t gemm_f32(int64_t M, int64_t N, int64_t K, float alpha,
                       const float *A, int64_t lda, gemm_order_t order_a,
                       const float *B, int64_t ldb, gemm_order_t order_b,
                       float beta, const float *C, int64_t ldc,
                       float *D, int64_t ldd, gemm_order_t order_cd,
                       cudaStream_t stream);

/*
 * gemm_bf16_f32acc -- BF16 inputs, FP32 accumulation, FP32 C and D.
 *
 * The tensor-core path (tcgen05.mma with the accumulator in tensor memory,
 * "GEMM on NVIDIA GPUs", section 4 "Tensor Core pipeline"; TMA-fed
 * multi-stage shared-memory ring with a producer/consumer split,
 * "Worklog: optimising GEMM on NVIDIA H100", kernels 7-9) runs when A and B
 * are 16-byte aligned and lda, ldb are multiples of 8 elements.  Otherwise a
 * CUDA-core kernel with the same results contract runs.  Arguments as for
 * gemm_f32; A and B point to BF16 bit patterns.
 *
 * Accuracy: |D - D_ref| <= 4e-3 * sum_k |alpha A_ik B_kj| + 1e-6 against the
 * exact result over the same BF16 inputs; bit-exact when every partial sum
 * is an integer below 2^24 and alpha = 1, beta = 0.
 */
gemm_status_t gemm_bf16_f32acc(int64_t M, int64_t N, int64_t K, float alpha,
                               const gemm_bf16_t *A, int64_t lda, gemm_order_t order_a,
                               const gemm_bf16_t *B, int64_t ldb, gemm_order_t order_b,
                               float beta, const float *C, int64_t ldc,
                               float *D, int64_t ldd, gemm_order_t order_cd,
                               cudaStream_t stream);

/*
 * gemm_f16_f32acc -- FP16 inputs, FP32 accumulation, FP32 C and D.
 *
 * The FP16-input, FP32-accumulate GEMM measured in "High-Performance FP16
 * General Matrix Multiplication on NVIDIA Ada Lovelace via CUTLASS and
 * WMMA" (methodology and results: FP16 -> FP32 at M = N = K = 8192), on the
 * same tcgen05 kernels as gemm_bf16_f32acc (kind::f16 with the FP16 operand
 * format) and the same CUDA-core fallback.  Arguments, contract and
 * accuracy bound as for gemm_bf16_f32acc; A and B point to binary16 bit
 * patterns.
 */
gemm_status_t gemm_f16_f32acc(int64_t M, int64_t N, int64_t K, float alpha,
                              const gemm_f16_t *A, int64_t lda, gemm_order_t order_a,
                              const gemm_f16_t *B, int64_t ldb, gemm_order_t order_b,
                              float beta, const float *C, int64_t ldc,
                              float *D, int64_t ldd, gemm_order_t order_cd,
                              cudaStream_t stream);

/*
 * gemm_f32_noalloc -- gemm_f32 for callers that cannot allocate device
 * memory.  The GEMM pages have no counterpart to this entry point.  It is
 * for code that must not call the CUDA allocator: code running under a
 * device-memory budget fixed in advance, code inside an allocator's own
 * callbacks, or code on a path where an allocation could block or fail.
 *
 * Arguments, results and accuracy are those of gemm_f32, and it picks the
 * same kernel with the same work split (the small-M kernel for M <= 8, the
 * cluster kernel for small problems, the CUDA-core kernel's tile
 * configurations otherwise).  The only difference: when that kernel splits
 * the K range of some tiles, the split pieces' counters and partial sums go
 * to a fixed 32 MiB array compiled into the library (a file-scope __device__
 * array that every device holding the library keeps until the process
 * exits) instead of pool memory and the stream's counters.  So the call
 * allocates nothing: no cudaMalloc, no cudaFree, no pool.
 *
 * Limits and rules:
 *   - The first 16 KiB of the array hold the counters, the rest (32 MiB -
 *     16 KiB) the partial sums.  A problem whose split needs more is refused
 *     with GEMM_ERR_INVALID_VALUE before anything is enqueued (gemm_f32
 *     handles it).  Problems that split no tile need no scratch.
 *   - The first call on each device sets up the array: it looks up that
 *     device's address of it (cudaGetSymbolAddress), zeroes the counters on
 *     `stream` and waits for that.  Make that first call before any stream
 *     capture on that device (under capture it returns GEMM_ERR_INTERNAL).
 *   - Every kernel leaves the counters it used at zero, so later calls clear
 *     nothing.  All calls on a device share the one array, and it keeps what
 *     the last call left in it.  Calls whose work overlaps on the GPU
 *     (different streams, no ordering between them) race on the array and
 *     give wrong results: order them on one stream or with events.
 */
gemm_status_t gemm_f32_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                               const float *A, int64_t lda, gemm_order_t order_a,
                               const float *B, int64_t ldb, gemm_order_t order_b,
                               float beta, const float *C, int64_t ldc,
                               float *D, int64_t ldd, gemm_order_t order_cd,
                               cudaStream_t stream);

/*
 * gemm_bf16_f32acc_ex -- gemm_bf16_f32acc with a fused epilogue:
 *
 *     D = act(alpha * op(A) * op(B) + beta * C + bias)
 *
 * stored as FP32 or as BF16 (round to nearest even), all in the same kernel
 * ("GEMM on NVIDIA GPUs", section 4 "Epilogue": alpha, beta, bias,
 * activation and dtype conversion in the epilogue, no extra round trip;
 * BF16 output as in "Worklog: optimising GEMM on NVIDIA H100", kernels 7-9).
 *
 *   epilogue->bias        N FP32 values, bias[j] added to column j of D, or
 *                         NULL for none (device pointer, 4-byte aligned)
 *   epilogue->activation  GEMM_ACT_NONE, GEMM_ACT_RELU (max(x, 0)) or
 *                         GEMM_ACT_GELU (tanh form:
 *                         0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))))
 *   epilogue->d_type      GEMM_D_F32 (D is float) or GEMM_D_BF16 (D holds
 *                         gemm_bf16_t; its pointer must be 2-byte aligned)
 *
 * epilogue == NULL means no bias, no activation, FP32 D (= gemm_bf16_f32acc).
 * C stays FP32; with a BF16 D, C and D must not overlap.  Everything else
 * as for gemm_bf16_f32acc.  Accuracy: the bound of gemm_bf16_f32acc on the
 * pre-activation value, times 1.13 for GELU (its largest slope) plus
 * 1e-6 |x|, plus 2^-8 |D| for BF16 rounding (half an ulp at 8 significant
 * bits).
 */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 } gemm_activation_t;
typedef enum { GEMM_D_F32 = 0, GEMM_D_BF16 = 1 } gemm_d_type_t;
typedef struct {
    const float *bias;
    gemm_activation_t activation;
    gemm_d_type_t d_type;
} gemm_epilogue_t;

gemm_status_t gemm_bf16_f32acc_ex(int64_t M, int64_t N, int64_t K, float alpha,
                                  const gemm_bf16_t *A, int64_t lda, gemm_order_t order_a,
                                  const gemm_bf16_t *B, int64_t ldb, gemm_order_t order_b,
                                  float beta, const float *C, int64_t ldc,
                                  void *D, int64_t ldd, gemm_order_t order_cd,
                                  const gemm_epilogue_t *epilogue, cudaStream_t stream);

/* Static English description of a status code; never NULL. */
const char *gemm_status_string(gemm_status_t status);

/*
 * gemm_last_device_status -- synchronises `stream`, then reads and clears
 * the current device's status word.  Returns GEMM_OK, or GEMM_ERR_TIMEOUT if
 * a tensor-core launch on this device gave up a bounded wait since the last
 * read (its D is then incomplete), or GEMM_ERR_INTERNAL if the read itself
 * failed.  After a timeout it also synchronises the device and frees every
 * stream's split counters (the counts of finished K pieces that each stream
 * keeps between calls, and that a kernel which gave up may have left
 * mid-count); the next split call on a stream starts from zeroed ones.  Read
 * it after a timeout before the next call on this device.
 */
gemm_status_t gemm_last_device_status(cudaStream_t stream);

/*
 * What the library holds on the current device between calls (the split
 * counters of each stream and the workspace pool; see "Split counters" and
 * "Workspace" above).  Nothing in the pages corresponds to this: it is the
 * accounting of this library's own memory.
 *   split_streams        streams of this device that hold split counters
 *   split_bytes          bytes of those counters
 *   pool_used_bytes      pool memory in use: the split counters, plus the
 *                        workspace of calls the GPU has not finished yet
 *   pool_reserved_bytes  pool memory held from the driver (in use or kept
 *                        for reuse, at most 256 MiB beyond what is in use)
 * Returns GEMM_ERR_INVALID_VALUE for a NULL info, GEMM_ERR_INTERNAL if a
 * CUDA query failed.
 */
typedef struct {
    uint64_t split_streams;
    uint64_t split_bytes;
    uint64_t pool_used_bytes;
    uint64_t pool_reserved_bytes;
} gemm_memory_info_t;
gemm_status_t gemm_memory_info(gemm_memory_info_t *info);

/*
 * gemm_release_memory -- synchronises the current device, frees the split
 * counters of every stream on it and returns the pool's free memory to the
 * driver.  Later calls take what they need again.  Call it when no other
 * host thread is calling the library on this device.
 */
gemm_status_t gemm_release_memory(void);

/*
 * gemm_last_kernel -- name of the kernel the calling host thread's most
 * recent successful gemm_* call enqueued ("" if it enqueued none, e.g. for
 * M == 0).  Static string; for tests and launch accounting.
 */
const char *gemm_last_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_08_GB300_GEMM_H */
