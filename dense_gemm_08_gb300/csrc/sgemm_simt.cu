// sgemm_simt.cu -- CUDA-core GEMM: FP32 FMA arithmetic, no tensor cores.
//
// Serves gemm_f32 (FP32 inputs) and the BF16 inputs that TMA cannot
// describe (BF16 values are widened exactly to FP32 when they are staged in
// shared memory; their products are exact in FP32).
//
// Structure (the CUDA-core steps of "Worklog: optimising GEMM on NVIDIA
// H100": kernel 2 shared-memory tiling, kernels 3-4 register tiling,
// kernel 5 vectorised loads with A transposed and padded in shared memory,
// kernel 6 warp tiling; "GEMM on NVIDIA GPUs", section 3 "Tiled GEMM" and
// section 4 "Register blocking", "Load-compute overlap"):
//   * a CTA owns a BM x BN tile of D and walks K in slices of BK;
//   * each slice of op(A) and op(B) is staged in shared memory as [BK][MN]
//     (K-major operands are transposed on the way in, so every thread reads
//     its A and B fragments with 16-byte loads);
//   * shared memory is double-buffered: the next slice is fetched into
//     registers while the current one is multiplied, then written to the
//     other buffer -- one barrier per slice;
//   * each thread accumulates a TM x TN register block built of 4 x 4 quads
//     spread over the warp tile, so fragment loads are conflict-free
//     broadcasts;
//   * the epilogue applies D = alpha * acc + beta * C (C read only when
//     beta != 0) with 16-byte accesses where alignment allows;
//   * tiles past the edge of the matrix load zeros and store nothing
//     outside D ("GEMM on NVIDIA GPUs", section 3 tiled kernel guards).
#include <cuda_bf16.h>

#include "internal.h"

namespace gemm {
namespace {

template <int BM_, int BN_, int BK_, int WM_, int WN_, int LM_, int LN_, int QM_, int QN_,
          int MINB_>
struct SimtCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static constexpr int WM = WM_, WN = WN_;  // warps along M and N
    static constexpr int LM = LM_, LN = LN_;  // lanes along M and N in a warp
    static constexpr int QM = QM_, QN = QN_;  // 4-wide quads per thread along M and N
    static constexpr int NT = WM * WN * 32;
    static constexpr int TM = 4 * QM, TN = 4 * QN;     // register block per thread
    static constexpr int WTM = TM * LM, WTN = TN * LN;  // warp tile
    static constexpr int PAD = 4;                       // keeps rows 16-byte aligned
    static constexpr int SA = BM + PAD, SB = BN + PAD;  // shared row strides (floats)
    static constexpr int MINB = MINB_;
    static constexpr int SLOTS_A = BM * BK / (4 * NT);  // 4-element vectors per thread
    static constexpr int SLOTS_B = BN * BK / (4 * NT);
    static_assert(LM * LN == 32, "a warp is 32 lanes");
    static_assert(WTM * WM == BM && WTN * WN == BN, "warps must tile the CTA tile");
    static_assert(SLOTS_A * 4 * NT == BM * BK && SLOTS_B * 4 * NT == BN * BK,
                  "loads must split evenly over the threads");
    static_assert(BK % 4 == 0, "K slices hold whole vectors");
};

// 128 x 128 x 8 tile, 256 threads, 8 x 8 per thread, two CTAs per SM.
using BigCfg = SimtCfg<128, 128, 8, 2, 4, 8, 4, 2, 2, 2>;
// 64 x 64 x 16 tile, 256 threads, 4 x 4 per thread: more CTAs for small problems.
using SmallCfg = SimtCfg<64, 64, 16, 2, 4, 8, 4, 1, 1, 1>;

// ---- element access: FP32 values or BF16 bit patterns, widened to FP32 ----
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static __device__ __forceinline__ float one(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float4 four(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
};

template <>
struct Elem<uint16_t> {
    // a BF16 value is the upper half of an FP32 bit pattern
    static __device__ __forceinline__ float one(const uint16_t *p) {
        return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
    }
    static __device__ __forceinline__ float4 four(const uint16_t *p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
};

// Fetch this thread's share of one BK-slice of an operand X into registers.
// X(mn, k) is at X[mn * ld + k] when KMAJ, else at X[mn + k * ld].
// Each share is SLOTS vectors of 4 consecutive elements along X's contiguous
// dimension.  `vec`: 16-byte (FP32) / 8-byte (BF16) vector loads are aligned.
// `guard`: the slice may cross the matrix edge (out-of-range elements are 0).
template <typename T, bool KMAJ, int EXT, int BK, int NT, int SLOTS>
__device__ __forceinline__ void fetch_slice(float4 (&r)[SLOTS], const T *__restrict__ X,
                                            int64_t ld, int64_t mn0, int64_t k0, int64_t mn_lim,
                                            int64_t k_lim, bool vec, bool guard) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int v = static_cast<int>(threadIdx.x) + s * NT;
        int mn, kk;
        if (KMAJ) {
            mn = v / (BK / 4);
            kk = (v % (BK / 4)) * 4;
        } else {
            kk = v / (EXT / 4);
            mn = (v % (EXT / 4)) * 4;
        }
        const int64_t gm = mn0 + mn, gk = k0 + kk;
        const T *ptr = KMAJ ? X + gm * ld + gk : X + gk * ld + gm;
        // elements of the vector step along the contiguous dimension
        const int64_t lead = KMAJ ? gk : gm, lead_lim = KMAJ ? k_lim : mn_lim;
        const bool row_ok = KMAJ ? (gm < mn_lim) : (gk < k_lim);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!guard) {
            if (vec) {
                x = Elem<T>::four(ptr);
            } else {
                x.x = Elem<T>::one(ptr);
                x.y = Elem<T>::one(ptr + 1);
                x.z = Elem<T>::one(ptr + 2);
                x.w = Elem<T>::one(ptr + 3);
            }
        } else if (row_ok) {
            if (vec && lead + 3 < lead_lim) {
                x = Elem<T>::four(ptr);
            } else {
                if (lead + 0 < lead_lim) x.x = Elem<T>::one(ptr);
                if (lead + 1 < lead_lim) x.y = Elem<T>::one(ptr + 1);
                if (lead + 2 < lead_lim) x.z = Elem<T>::one(ptr + 2);
                if (lead + 3 < lead_lim) x.w = Elem<T>::one(ptr + 3);
            }
        }
        r[s] = x;
    }
}

// Write the fetched share into shared memory laid out as [BK][EXT + PAD].
template <bool KMAJ, int EXT, int BK, int NT, int SLOTS, int STRIDE>
__device__ __forceinline__ void stage_slice(float *__restrict__ xs, const float4 (&r)[SLOTS]) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
        const int v = static_cast<int>(threadIdx.x) + s * NT;
        if (KMAJ) {  // transpose: four K values of one row go to four shared rows
            const int mn = v / (BK / 4), kk = (v % (BK / 4)) * 4;
            xs[(kk + 0) * STRIDE + mn] = r[s].x;
            xs[(kk + 1) * STRIDE + mn] = r[s].y;
            xs[(kk + 2) * STRIDE + mn] = r[s].z;
            xs[(kk + 3) * STRIDE + mn] = r[s].w;
        } else {
            const int kk = v / (EXT / 4), mn = (v % (EXT / 4)) * 4;
            *reinterpret_cast<float4 *>(&xs[kk * STRIDE + mn]) = r[s];
        }
    }
}

struct SimtArgs {
    Problem p;
    bool vec_a, vec_b;  // vector global loads of A / B are aligned
    bool vec_c, vec_d;  // 16-byte accesses of C / D rows are aligned
    int64_t tiles_m, tiles_n;
};

constexpr int kGroupM = 8;  // grouped raster: 8 tile-rows share each B column panel

template <typename Cfg, typename T, bool AK, bool BKM>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MINB) sgemm_simt_kernel(const SimtArgs args) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, NT = Cfg::NT;
    constexpr int TM = Cfg::TM, TN = Cfg::TN, SA = Cfg::SA, SB = Cfg::SB;
    __shared__ __align__(16) float As[2][BK * SA];
    __shared__ __align__(16) float Bs[2][BK * SB];

    const Problem &p = args.p;
    const T *__restrict__ A = static_cast<const T *>(p.A);
    const T *__restrict__ B = static_cast<const T *>(p.B);

    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int wm = warp / Cfg::WN, wn = warp % Cfg::WN;
    const int tr = lane / Cfg::LN, tc = lane % Cfg::LN;
    const int a_off = wm * Cfg::WTM + tr * 4;  // first row of this thread's quads
    const int b_off = wn * Cfg::WTN + tc * 4;  // first column of this thread's quads

    const int64_t n_tiles = args.tiles_m * args.tiles_n;
    const int64_t n_k = (p.K + BK - 1) / BK;

    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        // grouped rasterisation along M
        const int64_t width = kGroupM * args.tiles_n;
        const int64_t first_m = (t / width) * kGroupM;
        const int64_t rest_m = args.tiles_m - first_m;
        const int64_t gsz = rest_m < kGroupM ? rest_m : kGroupM;
        const int64_t tm = first_m + (t % width) % gsz;
        const int64_t tn = (t % width) / gsz;
        const int64_t m0 = tm * BM, n0 = tn * BN;
        const bool edge_mn = (m0 + BM > p.M) || (n0 + BN > p.N);

        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

        float4 ra[Cfg::SLOTS_A], rb[Cfg::SLOTS_B];
        {
            const bool guard = edge_mn || (BK > p.K);
            fetch_slice<T, AK, BM, BK, NT, Cfg::SLOTS_A>(ra, A, p.lda, m0, 0, p.M, p.K,
                                                         args.vec_a, guard);
            fetch_slice<T, BKM, BN, BK, NT, Cfg::SLOTS_B>(rb, B, p.ldb, n0, 0, p.N, p.K,
                                                          args.vec_b, guard);
            stage_slice<AK, BM, BK, NT, Cfg::SLOTS_A, SA>(As[0], ra);
            stage_slice<BKM, BN, BK, NT, Cfg::SLOTS_B, SB>(Bs[0], rb);
        }
        __syncthreads();

        for (int64_t kt = 0; kt < n_k; ++kt) {
            const int cur = static_cast<int>(kt & 1);
            const bool more = kt + 1 < n_k;
            if (more) {
                const int64_t k0 = (kt + 1) * BK;
                const bool guard = edge_mn || (k0 + BK > p.K);
                fetch_slice<T, AK, BM, BK, NT, Cfg::SLOTS_A>(ra, A, p.lda, m0, k0, p.M, p.K,
                                                             args.vec_a, guard);
                fetch_slice<T, BKM, BN, BK, NT, Cfg::SLOTS_B>(rb, B, p.ldb, n0, k0, p.N, p.K,
                                                              args.vec_b, guard);
            }
            const float *as = As[cur];
            const float *bs = Bs[cur];
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                float a[TM], b[TN];
#pragma unroll
                for (int q = 0; q < Cfg::QM; ++q) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(&as[k * SA + a_off + q * Cfg::LM * 4]);
                    a[q * 4 + 0] = v.x;
                    a[q * 4 + 1] = v.y;
                    a[q * 4 + 2] = v.z;
                    a[q * 4 + 3] = v.w;
                }
#pragma unroll
                for (int q = 0; q < Cfg::QN; ++q) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(&bs[k * SB + b_off + q * Cfg::LN * 4]);
                    b[q * 4 + 0] = v.x;
                    b[q * 4 + 1] = v.y;
                    b[q * 4 + 2] = v.z;
                    b[q * 4 + 3] = v.w;
                }
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            if (more) {
                stage_slice<AK, BM, BK, NT, Cfg::SLOTS_A, SA>(As[cur ^ 1], ra);
                stage_slice<BKM, BN, BK, NT, Cfg::SLOTS_B, SB>(Bs[cur ^ 1], rb);
            }
            __syncthreads();
        }

        // epilogue: D = alpha * acc + beta * C
        const bool use_c = p.beta != 0.f;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int64_t gr = m0 + a_off + (i / 4) * Cfg::LM * 4 + (i % 4);
            if (gr >= p.M) continue;
            float *drow = p.D + gr * p.ldd;
            const float *crow = use_c ? p.C + gr * p.ldc : nullptr;
#pragma unroll
            for (int q = 0; q < Cfg::QN; ++q) {
                const int64_t gc = n0 + b_off + q * Cfg::LN * 4;
                float o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) o[j] = p.alpha * acc[i][q * 4 + j];
                const bool full = gc + 3 < p.N;
                if (use_c) {
                    if (full && args.vec_c) {
                        // plain load: C may be D itself (in-place update)
                        const float4 c = *reinterpret_cast<const float4 *>(crow + gc);
                        o[0] = fmaf(p.beta, c.x, o[0]);
                        o[1] = fmaf(p.beta, c.y, o[1]);
                        o[2] = fmaf(p.beta, c.z, o[2]);
                        o[3] = fmaf(p.beta, c.w, o[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (gc + j < p.N) o[j] = fmaf(p.beta, crow[gc + j], o[j]);
                    }
                }
                if (full && args.vec_d) {
                    *reinterpret_cast<float4 *>(drow + gc) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (gc + j < p.N) drow[gc + j] = o[j];
                }
            }
        }
    }
}

bool aligned(const void *ptr, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) % bytes) == 0;
}

template <typename Cfg, typename T>
cudaError_t launch_cfg(const Problem &p, cudaStream_t stream, const char **name) {
    SimtArgs args;
    args.p = p;
    constexpr size_t vbytes = 4 * sizeof(T);
    args.vec_a = aligned(p.A, vbytes) && (p.lda % 4 == 0);
    args.vec_b = aligned(p.B, vbytes) && (p.ldb % 4 == 0);
    args.vec_c = p.beta != 0.f && aligned(p.C, 16) && (p.ldc % 4 == 0);
    args.vec_d = aligned(p.D, 16) && (p.ldd % 4 == 0);
    args.tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    args.tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int64_t tiles = args.tiles_m * args.tiles_n;
    const unsigned grid = static_cast<unsigned>(tiles < 0x7fffffff ? tiles : 0x7fffffff);
    const bool f32 = sizeof(T) == 4;
    if (p.a_kmajor && p.b_kmajor) {
        sgemm_simt_kernel<Cfg, T, true, true><<<grid, Cfg::NT, 0, stream>>>(args);
        *name = f32 ? "sgemm_simt<f32,A:K,B:K>" : "sgemm_simt<bf16,A:K,B:K>";
    } else if (p.a_kmajor) {
        sgemm_simt_kernel<Cfg, T, true, false><<<grid, Cfg::NT, 0, stream>>>(args);
        *name = f32 ? "sgemm_simt<f32,A:K,B:N>" : "sgemm_simt<bf16,A:K,B:N>";
    } else if (p.b_kmajor) {
        sgemm_simt_kernel<Cfg, T, false, true><<<grid, Cfg::NT, 0, stream>>>(args);
        *name = f32 ? "sgemm_simt<f32,A:M,B:K>" : "sgemm_simt<bf16,A:M,B:K>";
    } else {
        sgemm_simt_kernel<Cfg, T, false, false><<<grid, Cfg::NT, 0, stream>>>(args);
        *name = f32 ? "sgemm_simt<f32,A:M,B:N>" : "sgemm_simt<bf16,A:M,B:N>";
    }
    return cudaGetLastError();
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

__global__ void scale_c_kernel(const Problem p) {
    // D = beta * C (beta may be 0: then C is not read and D = 0)
    const int64_t total = p.M * p.N;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = e / p.N, j = e % p.N;
        const float c = p.beta != 0.f ? p.beta * p.C[i * p.ldc + j] : 0.f;
        p.D[i * p.ldd + j] = c;
    }
}

}  // namespace

cudaError_t launch_simt(const Problem &p, InType in, cudaStream_t stream, const char **name) {
    // Large tiles when they give at least one CTA per SM, small ones otherwise.
    const int64_t big_tiles = ((p.M + BigCfg::BM - 1) / BigCfg::BM) *
                              ((p.N + BigCfg::BN - 1) / BigCfg::BN);
    const bool big = big_tiles >= sm_count();
    if (in == InType::F32)
        return big ? launch_cfg<BigCfg, float>(p, stream, name)
                   : launch_cfg<SmallCfg, float>(p, stream, name);
    return big ? launch_cfg<BigCfg, uint16_t>(p, stream, name)
               : launch_cfg<SmallCfg, uint16_t>(p, stream, name);
}

cudaError_t launch_scale_c(const Problem &p, cudaStream_t stream, const char **name) {
    const int64_t total = p.M * p.N;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    scale_c_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
    *name = "scale_c";
    return cudaGetLastError();
}

}  // namespace gemm
