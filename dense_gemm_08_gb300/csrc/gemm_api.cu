// gemm_api.cu -- the C ABI of include/gemm.h: argument checks, layout
// normalisation and dispatch to the kernels.
//
// Normalisation: kernels only produce row-major D.  A column-major D is the
// row-major Dᵀ = op(B)ᵀ op(A)ᵀ (transpose identity of the GEMM definition,
// "GEMM on NVIDIA GPUs", section 1), so the call is rewritten with M and N
// swapped, A and B exchanged and each operand's storage order flipped.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gemm.h"
#include "gemm_probe.h"
#include "internal.h"

#define GEMM_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local const char *t_last_kernel = "";

constexpr int64_t kMaxDim = 0x7fffffff;

bool is_order(gemm_order_t o) { return o == GEMM_ROW_MAJOR || o == GEMM_COL_MAJOR; }

bool aligned(const void *p, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(p) % bytes) == 0;
}

int64_t need_ld(gemm_order_t order, int64_t rows, int64_t cols) {
    const int64_t v = order == GEMM_ROW_MAJOR ? cols : rows;
    return v > 1 ? v : 1;
}

// Every rule of the contract in gemm.h, checked before any CUDA call.
gemm_status_t validate(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                       gemm_order_t oa, const void *B, int64_t ldb, gemm_order_t ob, float beta,
                       const float *C, int64_t ldc, const void *D, int64_t ldd, gemm_order_t ocd,
                       size_t in_bytes, size_t d_bytes = sizeof(float)) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return GEMM_ERR_INVALID_VALUE;
    if (!is_order(oa) || !is_order(ob) || !is_order(ocd)) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    // a D of more than 2^43 elements exceeds any device's memory (the
    // kernels' tile indices are 32-bit on that assumption)
    if (M * N > (int64_t(1) << 43)) return GEMM_ERR_INVALID_VALUE;
    if (D == nullptr || !aligned(D, d_bytes) || ldd < need_ld(ocd, M, N))
        return GEMM_ERR_INVALID_VALUE;
    if (beta != 0.f && (C == nullptr || !aligned(C, sizeof(float)) || ldc < need_ld(ocd, M, N)))
        return GEMM_ERR_INVALID_VALUE;
    if (K > 0 && alpha != 0.f) {
        if (A == nullptr || B == nullptr || !aligned(A, in_bytes) || !aligned(B, in_bytes))
            return GEMM_ERR_INVALID_VALUE;
        if (lda < need_ld(oa, M, K) || ldb < need_ld(ob, K, N)) return GEMM_ERR_INVALID_VALUE;
    }
    return GEMM_OK;
}

gemm::Problem normalise(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                        gemm_order_t oa, const void *B, int64_t ldb, gemm_order_t ob, float beta,
                        const float *C, int64_t ldc, float *D, int64_t ldd, gemm_order_t ocd) {
    gemm::Problem p;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = beta != 0.f ? C : nullptr;
    p.ldc = ldc;
    p.D = D;
    p.ldd = ldd;
    if (ocd == GEMM_ROW_MAJOR) {
        p.M = M;
        p.N = N;
        p.A = A;
        p.lda = lda;
        p.a_kmajor = oa == GEMM_ROW_MAJOR;  // A(i,k) at A[i*lda + k]
        p.B = B;
        p.ldb = ldb;
        p.b_kmajor = ob == GEMM_COL_MAJOR;  // B(k,j) at B[k + j*ldb]
    } else {
        // Dᵀ (N x M, row-major with ldd) = op(B)ᵀ op(A)ᵀ.
        // A' = op(B)ᵀ: A'(j,k) = B(k,j); K-major iff B(k,j) is at B[j*ldb + k], i.e. B column-major.
        // B' = op(A)ᵀ: B'(k,i) = A(i,k); K-major iff A(i,k) is at A[k + i*lda], i.e. A row-major.
        p.M = N;
        p.N = M;
        p.A = B;
        p.lda = ldb;
        p.a_kmajor = ob == GEMM_COL_MAJOR;
        p.B = A;
        p.ldb = lda;
        p.b_kmajor = oa == GEMM_ROW_MAJOR;
    }
    return p;
}

// The library carries sm_103a code only.
gemm_status_t check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_UNSUPPORTED_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    return (major == 10 && minor == 3) ? GEMM_OK : GEMM_ERR_UNSUPPORTED_DEVICE;
}

gemm_status_t finish(cudaError_t e, const char *name) {
    if (e == cudaSuccess) {
        t_last_kernel = name;
        return GEMM_OK;
    }
    return (e == cudaErrorInvalidValue || e == cudaErrorSymbolNotFound) ? GEMM_ERR_INTERNAL
                                                                          : GEMM_ERR_LAUNCH;
}

}  // namespace

GEMM_API gemm_status_t gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                int64_t lda, gemm_order_t order_a, const float *B, int64_t ldb,
                                gemm_order_t order_b, float beta, const float *C, int64_t ldc,
                                float *D, int64_t ldd, gemm_order_t order_cd,
                                cudaStream_t stream) {
    t_last_kernel = "";
    gemm_status_t st = validate(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D,
                                ldd, order_cd, sizeof(float));
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    if ((st = check_device()) != GEMM_OK) return st;
    const gemm::Problem p = normalise(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                                      ldc, D, ldd, order_cd);
    const char *name = "";
    cudaError_t e;
    if (K == 0 || alpha == 0.f)
        e = gemm::launch_scale_c(p, stream, &name);
    else
        e = gemm::launch_f32(p, stream, &name);
    return finish(e, name);
}

GEMM_API gemm_status_t gemm_bf16_f32acc(int64_t M, int64_t N, int64_t K, float alpha,
                                        const gemm_bf16_t *A, int64_t lda, gemm_order_t order_a,
                                        const gemm_bf16_t *B, int64_t ldb, gemm_order_t order_b,
                                        float beta, const float *C, int64_t ldc, float *D,
                                        int64_t ldd, gemm_order_t order_cd, cudaStream_t stream) {
    t_last_kernel = "";
    gemm_status_t st = validate(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D,
                                ldd, order_cd, sizeof(gemm_bf16_t));
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    if ((st = check_device()) != GEMM_OK) return st;
    const gemm::Problem p = normalise(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                                      ldc, D, ldd, order_cd);
    const char *name = "";
    cudaError_t e;
    if (K == 0 || alpha == 0.f)
        e = gemm::launch_scale_c(p, stream, &name);
    else if (gemm::tc_eligible(p))
        e = gemm::launch_tc(p, gemm::InType::BF16, stream, &name);
    else if (gemm::skinny_eligible(p))
        e = gemm::launch_skinny(p, gemm::InType::BF16, stream, &name);
    else
        e = gemm::launch_simt(p, gemm::InType::BF16, stream, &name);
    return finish(e, name);
}

GEMM_API gemm_status_t gemm_f16_f32acc(int64_t M, int64_t N, int64_t K, float alpha,
                                       const gemm_f16_t *A, int64_t lda, gemm_order_t order_a,
                                       const gemm_f16_t *B, int64_t ldb, gemm_order_t order_b,
                                       float beta, const float *C, int64_t ldc, float *D,
                                       int64_t ldd, gemm_order_t order_cd, cudaStream_t stream) {
    t_last_kernel = "";
    gemm_status_t st = validate(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D,
                                ldd, order_cd, sizeof(gemm_f16_t));
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    if ((st = check_device()) != GEMM_OK) return st;
    const gemm::Problem p = normalise(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                                      ldc, D, ldd, order_cd);
    const char *name = "";
    cudaError_t e;
    if (K == 0 || alpha == 0.f)
        e = gemm::launch_scale_c(p, stream, &name);
    else if (gemm::tc_eligible(p))
        e = gemm::launch_tc(p, gemm::InType::F16, stream, &name);
    else if (gemm::skinny_eligible(p))
        e = gemm::launch_skinny(p, gemm::InType::F16, stream, &name);
    else
        e = gemm::launch_simt(p, gemm::InType::F16, stream, &name);
    return finish(e, name);
}

GEMM_API gemm_status_t gemm_bf16_f32acc_ex(int64_t M, int64_t N, int64_t K, float alpha,
                                           const gemm_bf16_t *A, int64_t lda,
                                           gemm_order_t order_a, const gemm_bf16_t *B,
                                           int64_t ldb, gemm_order_t order_b, float beta,
                                           const float *C, int64_t ldc, void *D, int64_t ldd,
                                           gemm_order_t order_cd, const gemm_epilogue_t *epilogue,
                                           cudaStream_t stream) {
    t_last_kernel = "";
    gemm_epilogue_t ep{nullptr, GEMM_ACT_NONE, GEMM_D_F32};
    if (epilogue != nullptr) ep = *epilogue;
    if (ep.activation != GEMM_ACT_NONE && ep.activation != GEMM_ACT_RELU &&
        ep.activation != GEMM_ACT_GELU)
        return GEMM_ERR_INVALID_VALUE;
    if (ep.d_type != GEMM_D_F32 && ep.d_type != GEMM_D_BF16) return GEMM_ERR_INVALID_VALUE;
    const bool d_bf16 = ep.d_type == GEMM_D_BF16;
    gemm_status_t st = validate(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D,
                                ldd, order_cd, sizeof(gemm_bf16_t),
                                d_bf16 ? sizeof(gemm_bf16_t) : sizeof(float));
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    if (ep.bias != nullptr && !aligned(ep.bias, sizeof(float))) return GEMM_ERR_INVALID_VALUE;
    if ((st = check_device()) != GEMM_OK) return st;
    gemm::Problem p = normalise(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc,
                                static_cast<float *>(D), ldd, order_cd);
    p.bias = ep.bias;
    p.bias_per_row = order_cd == GEMM_COL_MAJOR;  // columns of D are rows of the stored Dᵀ
    p.act = static_cast<int>(ep.activation);
    p.d_bf16 = d_bf16;
    const char *name = "";
    cudaError_t e;
    if (K == 0 || alpha == 0.f)
        e = gemm::launch_scale_c(p, stream, &name);
    else if (gemm::tc_eligible(p))
        e = gemm::launch_tc(p, gemm::InType::BF16, stream, &name);
    else if (gemm::skinny_eligible(p))
        e = gemm::launch_skinny(p, gemm::InType::BF16, stream, &name);
    else
        e = gemm::launch_simt(p, gemm::InType::BF16, stream, &name);
    return finish(e, name);
}

GEMM_API gemm_status_t gemm_f32_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                        const float *A, int64_t lda, gemm_order_t order_a,
                                        const float *B, int64_t ldb, gemm_order_t order_b,
                                        float beta, const float *C, int64_t ldc, float *D,
                                        int64_t ldd, gemm_order_t order_cd, cudaStream_t stream) {
    t_last_kernel = "";
    gemm_status_t st = validate(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C, ldc, D,
                                ldd, order_cd, sizeof(float));
    if (st != GEMM_OK || M == 0 || N == 0) return st;
    if ((st = check_device()) != GEMM_OK) return st;
    const gemm::Problem p = normalise(M, N, K, alpha, A, lda, order_a, B, ldb, order_b, beta, C,
                                      ldc, D, ldd, order_cd);
    const char *name = "";
    cudaError_t e;
    if (K == 0 || alpha == 0.f) {
        e = gemm::launch_scale_c(p, stream, &name);
    } else {
        // gemm_f32's kernel and work split, with its split pieces in the
        // fixed array: refuse before anything is enqueued if they do not fit
        size_t part = 0, counters = 0;
        gemm::f32_scratch_needs(p, &part, &counters);
        if (part > gemm::kFixedScratchBytes - gemm::kFixedCounterBytes ||
            counters > gemm::kFixedCounterBytes / sizeof(int))
            return GEMM_ERR_INVALID_VALUE;
        gemm::FixedScratch fixed{};
        if (gemm::fixed_scratch(&fixed, stream) != cudaSuccess) return GEMM_ERR_INTERNAL;
        e = gemm::launch_f32(p, stream, &name, &fixed);
    }
    return finish(e, name);
}

GEMM_API const char *gemm_status_string(gemm_status_t status) {
    switch (status) {
        case GEMM_OK: return "success";
        case GEMM_ERR_INVALID_VALUE: return "invalid argument (shape, leading dimension, order, NULL or misaligned pointer)";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "the current CUDA device is not sm_103";
        case GEMM_ERR_LAUNCH: return "kernel launch failed";
        case GEMM_ERR_TIMEOUT: return "a bounded wait in the tensor-core kernel ran out";
        case GEMM_ERR_INTERNAL: return "internal CUDA runtime or driver error";
    }
    return "unknown status";
}

GEMM_API gemm_status_t gemm_last_device_status(cudaStream_t stream) {
    int status = 0;
    if (gemm::tc_read_and_clear_status(stream, &status) != cudaSuccess) return GEMM_ERR_INTERNAL;
    if (status) {
        // a kernel that gave up may have left split counters mid-count
        if (gemm::split_sync_release_device() != cudaSuccess) return GEMM_ERR_INTERNAL;
        return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

GEMM_API gemm_status_t gemm_memory_info(gemm_memory_info_t *info) {
    if (info == nullptr) return GEMM_ERR_INVALID_VALUE;
    *info = gemm_memory_info_t{0, 0, 0, 0};
    const gemm_status_t dev = check_device();
    if (dev != GEMM_OK) return dev;
    gemm::MemoryInfo m;
    if (gemm::memory_info(&m) != cudaSuccess) return GEMM_ERR_INTERNAL;
    info->split_streams = m.split_streams;
    info->split_bytes = m.split_bytes;
    info->pool_used_bytes = m.pool_used_bytes;
    info->pool_reserved_bytes = m.pool_reserved_bytes;
    return GEMM_OK;
}

GEMM_API gemm_status_t gemm_release_memory(void) {
    const gemm_status_t dev = check_device();
    if (dev != GEMM_OK) return dev;
    return gemm::release_memory() == cudaSuccess ? GEMM_OK : GEMM_ERR_INTERNAL;
}

GEMM_API const char *gemm_last_kernel(void) { return t_last_kernel; }

// ------------------------------------------------------------ peak probes
GEMM_API gemm_status_t gemm_probe_tc_bf16(int cta_group, int64_t n_mma, double *flops,
                                          cudaStream_t stream) {
    t_last_kernel = "";
    if ((cta_group != 1 && cta_group != 2) || n_mma < 1 || n_mma > (int64_t(1) << 40) ||
        flops == nullptr)
        return GEMM_ERR_INVALID_VALUE;
    const gemm_status_t dev = check_device();
    if (dev != GEMM_OK) return dev;
    return finish(gemm::launch_tc_probe(cta_group, n_mma, stream, flops),
                  cta_group == 2 ? "tc_probe<pair>" : "tc_probe");
}

GEMM_API gemm_status_t gemm_probe_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
    t_last_kernel = "";
    if (timeout_ns < 1000 || timeout_ns > 10ull * 1000 * 1000 * 1000) return GEMM_ERR_INVALID_VALUE;
    const gemm_status_t dev = check_device();
    if (dev != GEMM_OK) return dev;
    return finish(gemm::launch_wait_probe(timeout_ns, stream), "wait_probe");
}

GEMM_API gemm_status_t gemm_probe_fma_f32(int64_t trips, double *flops, cudaStream_t stream) {
    t_last_kernel = "";
    if (trips < 1 || trips > (int64_t(1) << 40) || flops == nullptr) return GEMM_ERR_INVALID_VALUE;
    const gemm_status_t dev = check_device();
    if (dev != GEMM_OK) return dev;
    return finish(gemm::launch_fma_probe(trips, stream, flops), "fma_probe");
}
