// skinny.cu -- GEMM with a handful of rows: M <= 8 (after a column-major D
// has been turned into the row-major D^T problem).
//
// With M <= 8 the work is a few dot products per element of op(B): the time
// is reading op(B) from HBM once ("GEMM on NVIDIA GPUs", section 2: the
// arithmetic intensity 2MNK / bytes falls to about M FLOPs per byte of B, far
// below the ridge point; "Understanding roofline and tiling", section 8).  A
// tiled GEMM kernel would spend 127 of every 128 tile rows on padding and
// keep too few bytes in flight to stream B, so these shapes take this kernel
// instead: every byte of op(B) is read once, with wide coalesced loads and
// 16 of them in flight per thread (kept packed in registers until used).
//
// Work unit = (column block, K slice); one CTA per unit.
//   B N-contiguous (B(k, j) at B[k * ldb + j]): a CTA covers 128 columns;
//     lane l of warp w owns columns 4l .. 4l + 3 and rows k = k0 + w, k0 + w +
//     8, ... of the slice; the 8 warps' sums are added in warp order through
//     shared memory.
//   B K-contiguous (B(k, j) at B[k + j * ldb]): a CTA covers 16 columns,
//     2 per warp; lane l owns the 16-byte runs of k at k0 + V l + 32 V i of
//     each column (V = elements per 16 bytes); the lanes' sums are added by a
//     fixed shuffle tree.
// op(A) rows of the slice (up to 4096 / M elements of K) are staged in
// shared memory as FP32.  With several
// K slices, each writes its sums to a workspace and counts itself per column
// block; the last slice to be counted adds the slices in K order and writes
// D (no CTA waits for another; the result does not depend on arrival order).
// The epilogue is the library's: D = act(alpha * AB + beta * C + bias),
// FP32 or BF16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"

namespace gemm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStageFloats = 4096;  // A staging: MS rows x (4096 / MS) elements of K, 16 KiB

template <int MS>
__host__ __device__ constexpr int slice_max() {
    return kStageFloats / MS;  // K elements per slice
}

// ---- element conversion: FP32, BF16 bit patterns or FP16, widened exactly ----
template <typename T>
__device__ __forceinline__ float widen(T x);
template <>
__device__ __forceinline__ float widen<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ float widen<uint16_t>(uint16_t x) {
    return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

// Element e of a raw 32-bit word holding one FP32 or two 16-bit values.
template <typename T>
__device__ __forceinline__ float word_elem(uint32_t w, int e) {
    if constexpr (std::is_same<T, float>::value) {
        return __uint_as_float(w);
    } else if constexpr (std::is_same<T, uint16_t>::value) {
        return __uint_as_float(e == 0 ? (w << 16) : (w & 0xffff0000u));
    } else {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(e == 0 ? w : w >> 16)));
    }
}

// Raw vectors: 4 elements along N (B N-contiguous), 16 bytes along K
// (B K-contiguous).  Kept packed in registers until they are multiplied.
template <typename T>
struct Raw4 {  // 4 elements
    static constexpr int WORDS = 4 * sizeof(T) / 4;
    uint32_t w[WORDS];
    __device__ __forceinline__ void load(const T *p) {
        if constexpr (WORDS == 4) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
            w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
        } else {
            const uint2 q = __ldg(reinterpret_cast<const uint2 *>(p));
            w[0] = q.x; w[1] = q.y;
        }
    }
    __device__ __forceinline__ float get(int i) const {
        return sizeof(T) == 4 ? word_elem<T>(w[i], 0) : word_elem<T>(w[i / 2], i % 2);
    }
};

struct Raw16 {  // 16 bytes
    uint32_t w[4];
    __device__ __forceinline__ void load(const void *p) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    }
};

template <typename T>
__device__ __forceinline__ float raw16_get(const Raw16 &r, int i) {
    return sizeof(T) == 4 ? word_elem<T>(r.w[i], 0) : word_elem<T>(r.w[i / 2], i % 2);
}

// Pack a scalar element into raw word slot i (guarded loads build raw vectors too).
template <typename T>
__device__ __forceinline__ void put_elem(uint32_t *w, int i, T x) {
    if constexpr (sizeof(T) == 4) {
        w[i] = __float_as_uint(widen<T>(x));
    } else {
        const uint32_t h = *reinterpret_cast<const unsigned short *>(&x);
        w[i / 2] = (i % 2) ? ((w[i / 2] & 0xffffu) | (h << 16)) : ((w[i / 2] & 0xffff0000u) | h);
    }
}

struct SkinnyArgs {
    Problem p;
    int64_t n_cb;   // column blocks
    int64_t ks;     // K elements per slice
    int n_slices;
    bool vec_b;     // B's rows (N-contiguous) or columns (K-contiguous) allow wide loads
    float *ws;      // [n_slices][M][N] partial sums (n_slices > 1)
    int *ws_count;  // [n_cb] slices counted per column block (zero between calls)
};

__device__ __forceinline__ float a_elem(const Problem &p, int m, int64_t k, int in_type) {
    const int64_t off = p.a_kmajor ? m * p.lda + k : m + k * p.lda;
    if (in_type == 0) return __ldg(static_cast<const float *>(p.A) + off);
    if (in_type == 1) return widen<uint16_t>(__ldg(static_cast<const uint16_t *>(p.A) + off));
    return __half2float(static_cast<const __half *>(p.A)[off]);
}

// Stage rows 0..M-1 of op(A), K range [k0, k0 + len), in a_s[m * SL + kk],
// and zeros in [len, len rounded up to 8): the 16-byte runs of the
// K-contiguous kernel read up to there (against zeros of B; stale values
// there could be NaN).
template <typename T, int SL>
__device__ __forceinline__ void stage_a(const Problem &p, float *a_s, int64_t k0, int len) {
    constexpr int in_type =
        std::is_same<T, float>::value ? 0 : (std::is_same<T, uint16_t>::value ? 1 : 2);
    const int M = static_cast<int>(p.M);
    const int pad = (len + 7) / 8 * 8 - len;  // len + pad <= SL: SL is a multiple of 8
    for (int idx = threadIdx.x; idx < M * pad; idx += kThreads)
        a_s[(idx / pad) * SL + len + idx % pad] = 0.f;
    for (int idx = threadIdx.x; idx < M * len; idx += kThreads) {
        // consecutive threads walk A's contiguous dimension
        int m, kk;
        if (p.a_kmajor) {
            m = idx / len;
            kk = idx % len;
        } else {
            kk = idx / M;
            m = idx % M;
        }
        a_s[m * SL + kk] = a_elem(p, m, k0 + kk, in_type);
    }
}

// D(m, j) = act(alpha * v + beta * C(m, j) + bias), stored as FP32 or BF16.
__device__ __forceinline__ void store_d(const Problem &p, int m, int64_t j, float v) {
    float o = p.alpha * v;
    if (p.beta != 0.f) o = fmaf(p.beta, p.C[m * p.ldc + j], o);
    if (p.bias != nullptr) o += p.bias_per_row ? p.bias[m] : p.bias[j];
    o = apply_activation(o, p.act);
    if (p.d_bf16)
        reinterpret_cast<uint16_t *>(p.D)[m * p.ldd + j] = to_bf16_bits(o);
    else
        p.D[m * p.ldd + j] = o;
}

// The unit's sums out[m * NB + jj] (columns j0 + jj) -> D, directly or
// through the K-slice workspace.
template <int NB>
__device__ __forceinline__ void finish_unit(const SkinnyArgs &a, const float *out, int64_t cb,
                                            int slice, int64_t j0) {
    const Problem &p = a.p;
    const int M = static_cast<int>(p.M);
    const int total = M * NB;
    if (a.n_slices == 1) {
        for (int idx = threadIdx.x; idx < total; idx += kThreads) {
            const int m = idx / NB, jj = idx % NB;
            if (j0 + jj < p.N) store_d(p, m, j0 + jj, out[idx]);
        }
        return;
    }
    __shared__ int s_last;
    for (int idx = threadIdx.x; idx < total; idx += kThreads) {
        const int m = idx / NB, jj = idx % NB;
        if (j0 + jj < p.N)
            __stcg(&a.ws[(static_cast<int64_t>(slice) * M + m) * p.N + j0 + jj], out[idx]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&a.ws_count[cb], 1) == a.n_slices - 1;
    __syncthreads();
    if (!s_last) return;
    if (threadIdx.x == 0) a.ws_count[cb] = 0;  // every slice counted: ready for the next call
    __threadfence();
    for (int idx = threadIdx.x; idx < total; idx += kThreads) {
        const int m = idx / NB, jj = idx % NB;
        const int64_t j = j0 + jj;
        if (j >= p.N) continue;
        float v = 0.f;
        for (int s = 0; s < a.n_slices; ++s)  // K order
            v += __ldcg(&a.ws[(static_cast<int64_t>(s) * M + m) * p.N + j]);
        store_d(p, m, j, v);
    }
}

// ------------------------------------------------ B N-contiguous: 128 columns
constexpr int kBnCols = 128;
constexpr int kBnRows = 16;  // rows of B in flight per warp

template <typename T, int MS>
__global__ void __launch_bounds__(kThreads) skinny_bn_kernel(const SkinnyArgs a) {
    constexpr int NB = kBnCols, SL = slice_max<MS>();
    static_assert(kWarps * NB <= MS * SL, "the warps' sums reuse the A staging");
    __shared__ __align__(16) float a_s[MS * SL];
    __shared__ __align__(16) float out[MS * NB];
    const Problem &p = a.p;
    const T *__restrict__ B = static_cast<const T *>(p.B);
    pdl_wait();  // the previous kernel on the stream is done with its memory
    pdl_launch_dependents();
    const int64_t cb = blockIdx.x % a.n_cb;
    const int slice = static_cast<int>(blockIdx.x / a.n_cb);
    const int64_t k0 = slice * a.ks;
    const int len = static_cast<int>(p.K - k0 < a.ks ? p.K - k0 : a.ks);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t j0 = cb * NB;
    const int64_t j = j0 + lane * 4;
    stage_a<T, SL>(p, a_s, k0, len);
    __syncthreads();

    float acc[MS][4];
#pragma unroll
    for (int m = 0; m < MS; ++m)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[m][c] = 0.f;
    const bool wide = a.vec_b && j + 3 < p.N;
    const T *base = B + k0 * p.ldb + j;
    // rows kk = warp, warp + 8, ... of the slice, kBnRows loads in flight
    for (int kk0 = warp; kk0 < len; kk0 += kWarps * kBnRows) {
        Raw4<T> b[kBnRows];
#pragma unroll
        for (int u = 0; u < kBnRows; ++u) {
            const int kk = kk0 + u * kWarps;
            const T *row = base + static_cast<int64_t>(kk) * p.ldb;
            if (kk < len && wide) {
                b[u].load(row);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    put_elem<T>(b[u].w, c, (kk < len && j + c < p.N) ? row[c] : T(0));
            }
        }
#pragma unroll
        for (int u = 0; u < kBnRows; ++u) {
            const int kk = kk0 + u * kWarps;
            if (kk < len) {
#pragma unroll
                for (int m = 0; m < MS; ++m) {
                    const float av = a_s[m * SL + kk];
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(av, b[u].get(c), acc[m][c]);
                }
            }
        }
    }
    // the 8 warps' sums, row by row, added in warp order (through the A
    // staging, which every warp has finished reading)
    float *red = a_s;
#pragma unroll
    for (int m = 0; m < MS; ++m) {
        __syncthreads();
#pragma unroll
        for (int c = 0; c < 4; ++c) red[warp * NB + lane * 4 + c] = acc[m][c];
        __syncthreads();
        if (threadIdx.x < NB) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) v += red[w * NB + threadIdx.x];
            out[m * NB + threadIdx.x] = v;
        }
    }
    __syncthreads();
    finish_unit<NB>(a, out, cb, slice, j0);
}

// ------------------------------------------------ B K-contiguous: 16 columns
constexpr int kBkColsPerWarp = 2;
constexpr int kBkRuns = 8;  // 16-byte runs in flight per column per lane

template <typename T, int MS>
__global__ void __launch_bounds__(kThreads) skinny_bk_kernel(const SkinnyArgs a) {
    constexpr int CPW = kBkColsPerWarp, NB = kWarps * CPW, SL = slice_max<MS>();
    constexpr int V = 16 / sizeof(T);  // elements per 16-byte run
    __shared__ __align__(16) float a_s[MS * SL];
    __shared__ __align__(16) float out[MS * NB];
    const Problem &p = a.p;
    const T *__restrict__ B = static_cast<const T *>(p.B);
    pdl_wait();  // the previous kernel on the stream is done with its memory
    pdl_launch_dependents();
    const int64_t cb = blockIdx.x % a.n_cb;
    const int slice = static_cast<int>(blockIdx.x / a.n_cb);
    const int64_t k0 = slice * a.ks;
    const int len = static_cast<int>(p.K - k0 < a.ks ? p.K - k0 : a.ks);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t j0 = cb * NB;
    stage_a<T, SL>(p, a_s, k0, len);
    __syncthreads();

    float acc[MS][CPW];
#pragma unroll
    for (int m = 0; m < MS; ++m)
#pragma unroll
        for (int c = 0; c < CPW; ++c) acc[m][c] = 0.f;
    const T *col[CPW];
    bool live[CPW];
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
        const int64_t jc = j0 + warp * CPW + c;
        live[c] = jc < p.N;
        col[c] = B + (live[c] ? jc : 0) * p.ldb + k0;
    }
    for (int kk0 = lane * V; kk0 < len; kk0 += 32 * V * kBkRuns) {
        Raw16 b[kBkRuns][CPW];
#pragma unroll
        for (int r = 0; r < kBkRuns; ++r) {
            const int kk = kk0 + r * 32 * V;
#pragma unroll
            for (int c = 0; c < CPW; ++c) {
                if (live[c] && a.vec_b && kk + V <= len) {
                    b[r][c].load(col[c] + kk);
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        put_elem<T>(b[r][c].w, e, (live[c] && kk + e < len) ? col[c][kk + e] : T(0));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kBkRuns; ++r) {
            const int kk = kk0 + r * 32 * V;
            if (kk < len) {
#pragma unroll
                for (int m = 0; m < MS; ++m) {
#pragma unroll
                    for (int e4 = 0; e4 < V; e4 += 4) {
                        // zeros of B past len meet the zeros staged after A's slice
                        const float4 q = *reinterpret_cast<const float4 *>(&a_s[m * SL + kk + e4]);
                        const float av[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int c = 0; c < CPW; ++c)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                acc[m][c] = fmaf(av[e], raw16_get<T>(b[r][c], e4 + e), acc[m][c]);
                    }
                }
            }
        }
    }
    // lanes' sums by a fixed shuffle tree
#pragma unroll
    for (int m = 0; m < MS; ++m)
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            float v = acc[m][c];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) out[m * NB + warp * CPW + c] = v;
        }
    __syncthreads();
    finish_unit<NB>(a, out, cb, slice, j0);
}

int sm_count_now() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

bool is_aligned(const void *ptr, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) % bytes) == 0;
}

template <typename T, int MS>
cudaError_t launch_ms(const SkinnyArgs &a, unsigned grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl_attribute(&attr[0]);
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.p.b_kmajor) return cudaLaunchKernelEx(&cfg, skinny_bk_kernel<T, MS>, a);
    return cudaLaunchKernelEx(&cfg, skinny_bn_kernel<T, MS>, a);
}

template <typename T>
cudaError_t launch_t(const SkinnyArgs &a, unsigned grid, cudaStream_t stream) {
    const int64_t M = a.p.M;
    if (M <= 1) return launch_ms<T, 1>(a, grid, stream);
    if (M <= 2) return launch_ms<T, 2>(a, grid, stream);
    if (M <= 4) return launch_ms<T, 4>(a, grid, stream);
    return launch_ms<T, 8>(a, grid, stream);
}

}  // namespace

bool skinny_eligible(const Problem &p) { return p.M >= 1 && p.M <= kSkinnyMaxM && p.K > 0; }


namespace {
// The launch plan: column blocks, K slices (a.n_cb, a.ks, a.n_slices) and
// wide-load eligibility for `p`.
SkinnyArgs plan_skinny(const Problem &p, InType in) {
    const int64_t esz = in == InType::F32 ? 4 : 2;
    SkinnyArgs a;
    a.p = p;
    const int64_t nb = p.b_kmajor ? kWarps * kBkColsPerWarp : kBnCols;
    a.n_cb = (p.N + nb - 1) / nb;
    // wide loads: 16 bytes along K (K-contiguous B) or 4 elements along N
    const int64_t vb = p.b_kmajor ? 16 : 4 * esz;
    a.vec_b = is_aligned(p.B, static_cast<size_t>(vb)) && (p.ldb * esz) % vb == 0;
    // K slices: no longer than the A staging holds; enough units for about
    // two CTAs per SM, but slices of at least 512 elements of K
    const int64_t ms = p.M <= 1 ? 1 : p.M <= 2 ? 2 : p.M <= 4 ? 4 : 8;
    const int64_t max_len = kStageFloats / ms;
    const int64_t target = 2 * static_cast<int64_t>(sm_count_now());
    int64_t slices = (target + a.n_cb - 1) / a.n_cb;
    const int64_t by_len = (p.K + 511) / 512;
    if (slices > by_len) slices = by_len;
    const int64_t min_slices = (p.K + max_len - 1) / max_len;
    if (slices < min_slices) slices = min_slices;
    if (slices < 1) slices = 1;
    // slices start on whole 16-byte runs of a warp (K-contiguous) or on 8 rows
    const int64_t quantum = p.b_kmajor ? 32 * (16 / esz) : 8;
    int64_t ks = (p.K + slices - 1) / slices;
    ks = (ks + quantum - 1) / quantum * quantum;
    if (ks > max_len) ks = max_len;
    a.ks = ks;
    a.n_slices = static_cast<int>((p.K + ks - 1) / ks);
    a.ws = nullptr;
    a.ws_count = nullptr;
    return a;
}
}  // namespace

void skinny_scratch_needs(const Problem &p, InType in, size_t *part_bytes, size_t *n_counters) {
    *part_bytes = 0;
    *n_counters = 0;
    if (!skinny_eligible(p)) return;
    const SkinnyArgs a = plan_skinny(p, in);
    if (a.n_slices <= 1) return;
    *part_bytes = static_cast<size_t>(a.n_slices) * p.M * p.N * sizeof(float);
    *n_counters = static_cast<size_t>(a.n_cb);
}

cudaError_t launch_skinny(const Problem &p, InType in, cudaStream_t stream, const char **name,
                          const FixedScratch *fixed) {
    if (!skinny_eligible(p)) return cudaErrorInvalidValue;
    SkinnyArgs a = plan_skinny(p, in);
    const int64_t grid = a.n_cb * a.n_slices;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;

    void *ws = nullptr;
    SplitSync sync;  // the stream's split counters, held until the launch is enqueued
    if (a.n_slices > 1) {
        const size_t part = static_cast<size_t>(a.n_slices) * p.M * p.N * sizeof(float);
        if (fixed != nullptr) {
            // the caller's scratch: counters zero between calls (the last
            // slice of a column block resets its own)
            if (part > fixed->part_bytes || static_cast<size_t>(a.n_cb) > fixed->n_counters)
                return cudaErrorInvalidValue;
            a.ws_count = fixed->counters;
            a.ws = static_cast<float *>(fixed->part);
        } else {
            // partial sums from the pool; counters from the stream's split
            // counters (zero; the last slice of a column block resets its own)
            cudaError_t e = sync.acquire(stream, static_cast<size_t>(a.n_cb));
            if (e != cudaSuccess) return e;
            a.ws_count = sync.counters;
            e = workspace_alloc(part, stream, &ws);
            if (e != cudaSuccess) return e;
            a.ws = static_cast<float *>(ws);
        }
    }
    const unsigned g = static_cast<unsigned>(grid);
    cudaError_t e;
    if (in == InType::F32) {
        e = launch_t<float>(a, g, stream);
        *name = p.b_kmajor ? "skinny<f32,B:K>" : "skinny<f32,B:N>";
    } else if (in == InType::F16) {
        e = launch_t<__half>(a, g, stream);
        *name = p.b_kmajor ? "skinny<f16,B:K>" : "skinny<f16,B:N>";
    } else {
        e = launch_t<uint16_t>(a, g, stream);
        *name = p.b_kmajor ? "skinny<bf16,B:K>" : "skinny<bf16,B:N>";
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (ws != nullptr) {
        const cudaError_t ef = workspace_free(ws, stream);
        if (e == cudaSuccess) e = ef;
    }
    const cudaError_t er = sync.release();
    return e != cudaSuccess ? e : er;
}

}  // namespace gemm
