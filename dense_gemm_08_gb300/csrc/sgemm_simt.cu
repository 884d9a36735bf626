// sgemm_simt.cu -- CUDA-core GEMM: FP32 FMA arithmetic, no tensor cores.
//
// Serves gemm_f32 (FP32 inputs) and the BF16 / FP16 inputs that TMA cannot
// describe (BF16 and FP16 values are widened exactly to FP32 when they are
// staged in shared memory; their products are exact in FP32).
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
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "epilogue.cuh"
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

// 128 x 256 x 16 tile, 256 threads, 16 x 8 per thread (warp tile 64 x 64 of
// 4 x 8 lanes), one CTA per SM: 128 FMAs per 6 fragment loads.  Of the
// 8 x 16 and 16 x 8 blocks with the same loads, 16 x 8 ran 2.5 % faster on
// GB300 (FP32 4096^3: 56.9 against 55.6 TFLOP/s).
using BigCfg = SimtCfg<128, 256, 16, 2, 4, 4, 8, 4, 2, 1>;
// 64 x 64 x 16 tile, 256 threads, 4 x 4 per thread: more CTAs for small problems.
using SmallCfg = SimtCfg<64, 64, 16, 2, 4, 8, 4, 1, 1, 1>;
// FP32 only: 128 x 128 x 16 tile, 8 x 8 per thread, for problems with too few
// 128 x 256 tiles or a short K; and 256 x 64 x 16, 8 x 8 per thread, for a D
// at most 64 columns wide.  Measured on GB300 against the two above: FP32
// 127 x 8191 x 4096 29.4 -> 40.2 TFLOP/s (128 x 128), 4095 x 4097 x 1000
// 38.6 -> 40.5 (128 x 128), 16384 x 64 x 8192 32.7 -> 46.5 (256 x 64).
using WideCfg = SimtCfg<128, 128, 16, 2, 4, 8, 4, 2, 2, 1>;
using TallCfg = SimtCfg<256, 64, 16, 4, 2, 8, 4, 2, 2, 1>;

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

template <>
struct Elem<__half> {
    // IEEE binary16 widened exactly to FP32
    static __device__ __forceinline__ float one(const __half *p) { return __half2float(p[0]); }
    static __device__ __forceinline__ float4 four(const __half *p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
};

// Per-thread view of one operand's slices.  X(mn, k) is at X[mn * ld + k]
// when KMAJ, else at X[mn + k * ld].  The thread owns SLOTS vectors of 4
// consecutive elements along X's contiguous dimension in every BK-slice; their
// addresses at k = 0 are computed once per tile, and each slice moves them by
// `kstep` elements.
template <typename T, bool KMAJ, int EXT, int BK, int NT, int SLOTS>
struct SliceLoader {
    const T *p0[SLOTS];
    int64_t kstep;

    __device__ __forceinline__ static void coords(int s, int &mn, int &kk) {
        const int v = static_cast<int>(threadIdx.x) + s * NT;
        if (KMAJ) {
            mn = v / (BK / 4);
            kk = (v % (BK / 4)) * 4;
        } else {
            kk = v / (EXT / 4);
            mn = (v % (EXT / 4)) * 4;
        }
    }

    __device__ __forceinline__ void init(const T *X, int64_t ld, int64_t mn0) {
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            int mn, kk;
            coords(s, mn, kk);
            p0[s] = KMAJ ? X + (mn0 + mn) * ld + kk : X + static_cast<int64_t>(kk) * ld + mn0 + mn;
        }
        kstep = KMAJ ? BK : BK * ld;
    }

    // Interior slice with aligned vectors: one wide load per slot.
    __device__ __forceinline__ void fetch_fast(float4 (&r)[SLOTS], int64_t kt) const {
        const int64_t off = kt * kstep;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) r[s] = Elem<T>::four(p0[s] + off);
    }

    // Any slice: per-element guards (out-of-range elements are 0); wide loads
    // only when `vec` says they are aligned.
    __device__ __forceinline__ void fetch_guarded(float4 (&r)[SLOTS], int64_t kt, int64_t mn0,
                                                  int64_t mn_lim, int64_t k_lim,
                                                  bool vec) const {
        const int64_t off = kt * kstep;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            int mn, kk;
            coords(s, mn, kk);
            const int64_t gm = mn0 + mn, gk = kt * BK + kk;
            const T *ptr = p0[s] + off;
            // elements of the vector step along the contiguous dimension
            const int64_t lead = KMAJ ? gk : gm, lead_lim = KMAJ ? k_lim : mn_lim;
            const bool row_ok = KMAJ ? (gm < mn_lim) : (gk < k_lim);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row_ok) {
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
};

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

// Two FP32 multiply-adds in one instruction (fma.rn.f32x2): each half is an
// fmaf of its own, rounded the same way.  Pairs are 64-bit registers, low
// half first.
__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t dup2(float x) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

struct SimtArgs {
    Problem p;
    bool vec_a, vec_b;  // vector global loads of A / B are aligned
    bool vec_c, vec_d;  // 16-byte accesses of C / FP32 D rows are aligned
    bool vec_d16;       // 8-byte accesses of BF16 D rows are aligned
    int64_t tiles_m, tiles_n;
    // Stream-K tail: tiles [0, full_tiles) are computed whole, one per CTA;
    // the remaining tail_tiles x n_k slice-iterations are dealt out evenly, in
    // order, to sk_ctas CTAs.  A CTA holding only part of a tile's K range
    // stores its partial sums in ws_part (slot = its position among the
    // tile's contributors, which are in K order) and counts itself in
    // ws_count; the last contributor adds the partials in that order and
    // writes D.
    int64_t full_tiles, tail_iters;
    int sk_ctas, max_contrib;
    float *ws_part;
    int *ws_count;
};

constexpr int kGroupM = 8;  // grouped raster: 8 tile-rows share each B column panel

// EPI: the fused epilogue (bias, activation, BF16 D) is compiled in.  The
// plain kernels leave it out: their code stays as small as the alpha/beta
// epilogue needs, which the instruction cache of the fully unrolled K loop
// rewards.
template <typename Cfg, typename T, bool AK, bool BKM, bool EPI>
__global__ void __launch_bounds__(Cfg::NT, Cfg::MINB) sgemm_simt_kernel(const SimtArgs args) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, NT = Cfg::NT;
    constexpr int TM = Cfg::TM, TN = Cfg::TN, SA = Cfg::SA, SB = Cfg::SB;
    __shared__ __align__(16) float As[2][BK * SA];
    __shared__ __align__(16) float Bs[2][BK * SB];

    const Problem &p = args.p;
    const T *__restrict__ A = static_cast<const T *>(p.A);
    const T *__restrict__ B = static_cast<const T *>(p.B);
    pdl_wait();  // the previous kernel on the stream is done with its memory
    pdl_launch_dependents();

    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int wm = warp / Cfg::WN, wn = warp % Cfg::WN;
    const int tr = lane / Cfg::LN, tc = lane % Cfg::LN;
    const int a_off = wm * Cfg::WTM + tr * 4;  // first row of this thread's quads
    const int b_off = wn * Cfg::WTN + tc * 4;  // first column of this thread's quads

    const int64_t n_k = (p.K + BK - 1) / BK;
    __shared__ int s_last;  // this CTA completed a split tile

    const int64_t n_units = args.full_tiles + args.sk_ctas;
    // first stream-K CTA whose range holds tail iteration x
    auto owner = [&](int64_t x) -> int64_t {
        return ((x + 1) * args.sk_ctas - 1) / args.tail_iters;
    };
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
      int64_t it = 0, it_end = 1;  // tail iterations of this unit (stream-K units only)
      if (u >= args.full_tiles) {
          const int64_t c = u - args.full_tiles;
          it = c * args.tail_iters / args.sk_ctas;
          it_end = (c + 1) * args.tail_iters / args.sk_ctas;
      }
      while (it < it_end) {
        // this step: one tile and a K range of it
        int64_t t = u, kt_begin = 0, kt_end = n_k;
        int contrib = 0, n_contrib = 1;
        if (u >= args.full_tiles) {
            const int64_t tl = it / n_k;
            kt_begin = it % n_k;
            kt_end = kt_begin + (it_end - it);
            if (kt_end > n_k) kt_end = n_k;
            t = args.full_tiles + tl;
            const int64_t c0 = owner(tl * n_k), c1 = owner(tl * n_k + n_k - 1);
            contrib = static_cast<int>(u - args.full_tiles - c0);
            n_contrib = static_cast<int>(c1 - c0 + 1);
            it += kt_end - kt_begin;
        } else {
            it = it_end;  // whole tile
        }
        const int split = n_contrib > 1 ? contrib : -1;
        // grouped rasterisation along M
        const int64_t width = kGroupM * args.tiles_n;
        const int64_t first_m = (t / width) * kGroupM;
        const int64_t rest_m = args.tiles_m - first_m;
        const int64_t gsz = rest_m < kGroupM ? rest_m : kGroupM;
        const int64_t tm = first_m + (t % width) % gsz;
        const int64_t tn = (t % width) / gsz;
        const int64_t m0 = tm * BM, n0 = tn * BN;
        const bool edge_mn = (m0 + BM > p.M) || (n0 + BN > p.N);

        // accumulators as row pairs (2p, 2p + 1) for the paired FMAs; unpacked
        // into acc[TM][TN] after the K loop
        uint64_t acc2[TM / 2][TN];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc2[i][j] = 0ull;

        SliceLoader<T, AK, BM, BK, NT, Cfg::SLOTS_A> la;
        SliceLoader<T, BKM, BN, BK, NT, Cfg::SLOTS_B> lb;
        la.init(A, p.lda, m0);
        lb.init(B, p.ldb, n0);
        // interior tiles with aligned operands take the unguarded wide loads
        const bool fast_mn = !edge_mn && args.vec_a && args.vec_b;
        const int64_t full_slices = p.K / BK;  // slices entirely inside K

        float4 ra[Cfg::SLOTS_A], rb[Cfg::SLOTS_B];
        auto fetch = [&](int64_t kt) {
            if (fast_mn && kt < full_slices) {
                la.fetch_fast(ra, kt);
                lb.fetch_fast(rb, kt);
            } else {
                la.fetch_guarded(ra, kt, m0, p.M, p.K, args.vec_a);
                lb.fetch_guarded(rb, kt, n0, p.N, p.K, args.vec_b);
            }
        };
        if (kt_begin < kt_end) {  // CTA-uniform
        fetch(kt_begin);
        stage_slice<AK, BM, BK, NT, Cfg::SLOTS_A, SA>(As[0], ra);
        stage_slice<BKM, BN, BK, NT, Cfg::SLOTS_B, SB>(Bs[0], rb);
        __syncthreads();

        for (int64_t kt = kt_begin; kt < kt_end; ++kt) {
            const int cur = static_cast<int>((kt - kt_begin) & 1);
            const bool more = kt + 1 < kt_end;
            if (more) fetch(kt + 1);  // lands in registers while this slice is multiplied
            const float *as = As[cur];
            const float *bs = Bs[cur];
            // fragments double-buffered in registers: slice row k + 1 is read
            // from shared memory while row k is multiplied.  A's fragment is
            // read as row pairs (a quad of rows = two pairs), B's values are
            // duplicated into pairs as they are read (a step ahead of their
            // use): one paired FMA updates rows 2p, 2p + 1.
            uint64_t a[2][TM / 2];
            uint64_t bd[2][TN];
            auto load_frag = [&](int buf, int k) {
#pragma unroll
                for (int q = 0; q < Cfg::QM; ++q) {
                    const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(
                        &as[k * SA + a_off + q * Cfg::LM * 4]);
                    a[buf][q * 2 + 0] = v.x;
                    a[buf][q * 2 + 1] = v.y;
                }
#pragma unroll
                for (int q = 0; q < Cfg::QN; ++q) {
                    const float4 v =
                        *reinterpret_cast<const float4 *>(&bs[k * SB + b_off + q * Cfg::LN * 4]);
                    bd[buf][q * 4 + 0] = dup2(v.x);
                    bd[buf][q * 4 + 1] = dup2(v.y);
                    bd[buf][q * 4 + 2] = dup2(v.z);
                    bd[buf][q * 4 + 3] = dup2(v.w);
                }
            };
            load_frag(0, 0);
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                if (k + 1 < BK) load_frag((k + 1) & 1, k + 1);
#pragma unroll
                for (int j = 0; j < TN; ++j)
#pragma unroll
                    for (int i = 0; i < TM / 2; ++i) fma2(acc2[i][j], a[k & 1][i], bd[k & 1][j]);
            }
            if (more) {
                stage_slice<AK, BM, BK, NT, Cfg::SLOTS_A, SA>(As[cur ^ 1], ra);
                stage_slice<BKM, BN, BK, NT, Cfg::SLOTS_B, SB>(Bs[cur ^ 1], rb);
            }
            __syncthreads();
        }
        }
        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) unpack2(acc2[i][j], acc[2 * i][j], acc[2 * i + 1][j]);

        if (split >= 0) {
            // Every contributor of a split tile stores its partial sums (each
            // thread its own TM x TN block), then counts itself; the last one
            // adds all partials in K order -- the same order whatever the
            // arrival order, so the result is deterministic -- and runs the
            // epilogue.
            const int64_t slot = t - args.full_tiles;
            float *tile_ws = args.ws_part + slot * args.max_contrib * (BM * BN);
            float4 *mine = reinterpret_cast<float4 *>(tile_ws + split * (BM * BN) +
                                                      threadIdx.x * (TM * TN));
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j4 = 0; j4 < TN / 4; ++j4)
                    __stcg(&mine[i * (TN / 4) + j4],
                           make_float4(acc[i][j4 * 4 + 0], acc[i][j4 * 4 + 1],
                                       acc[i][j4 * 4 + 2], acc[i][j4 * 4 + 3]));
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0)
                s_last = atomicAdd(&args.ws_count[slot], 1) == n_contrib - 1;
            __syncthreads();
            if (!s_last) continue;  // CTA-uniform
            __threadfence();
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
            for (int sp = 0; sp < n_contrib; ++sp) {
                const float4 *part = reinterpret_cast<const float4 *>(
                    tile_ws + sp * (BM * BN) + threadIdx.x * (TM * TN));
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j4 = 0; j4 < TN / 4; ++j4) {
                        const float4 v = __ldcg(&part[i * (TN / 4) + j4]);
                        acc[i][j4 * 4 + 0] += v.x;
                        acc[i][j4 * 4 + 1] += v.y;
                        acc[i][j4 * 4 + 2] += v.z;
                        acc[i][j4 * 4 + 3] += v.w;
                    }
            }
            if (threadIdx.x == 0) args.ws_count[slot] = 0;  // ready for the next call
        }

        // epilogue: D = act(alpha * acc + beta * C + bias), FP32 or BF16
        const bool use_c = p.beta != 0.f;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int64_t gr = m0 + a_off + (i / 4) * Cfg::LM * 4 + (i % 4);
            if (gr >= p.M) continue;
            float *drow = p.D + gr * p.ldd;
            uint16_t *drow16 = reinterpret_cast<uint16_t *>(p.D) + gr * p.ldd;
            const float *crow = use_c ? p.C + gr * p.ldc : nullptr;
            const float row_bias =
                (EPI && p.bias != nullptr && p.bias_per_row) ? p.bias[gr] : 0.f;
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
                if (EPI && p.bias != nullptr) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        o[j] += p.bias_per_row ? row_bias : (gc + j < p.N ? p.bias[gc + j] : 0.f);
                }
                if (EPI && p.act != kActNone) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) o[j] = apply_activation(o[j], p.act);
                }
                if (EPI && p.d_bf16) {
                    if (full && args.vec_d16) {
                        *reinterpret_cast<uint2 *>(drow16 + gc) =
                            make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (gc + j < p.N) drow16[gc + j] = to_bf16_bits(o[j]);
                    }
                } else if (full && args.vec_d) {
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
}

bool aligned(const void *ptr, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) % bytes) == 0;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

// How to cut the work into CTA units.  With S resident CTAs and T tiles, the
// last T mod S tiles would run as a partial wave on a fraction of the SMs.
// Instead their K-slice iterations are dealt out evenly to S CTAs (a
// stream-K tail; when T < S every tile is dealt out), so every SM finishes at
// about the same time ("GEMM on NVIDIA GPUs", section 5: split-K / Stream-K
// for short M/N and tile tails).
struct SplitPlan {
    int64_t full_tiles, tail_tiles, tail_iters;
    int sk_ctas, max_contrib;
};

template <typename Cfg>
SplitPlan plan_split(const Problem &p, int64_t tiles) {
    const int64_t slots = static_cast<int64_t>(sm_count()) * Cfg::MINB;
    const int64_t n_k = (p.K + Cfg::BK - 1) / Cfg::BK;
    SplitPlan plan{tiles, 0, 0, 0, 1};
    const int64_t rem = tiles % slots;
    if (rem == 0) return plan;
    const int64_t tail_tiles = rem;
    const int64_t iters = tail_tiles * n_k;
    // at least 4 slices per CTA; no point in fewer CTAs than tail tiles
    int64_t ctas = slots;
    if (ctas > iters / 4) ctas = iters / 4;
    if (ctas <= tail_tiles) return plan;  // nothing to gain: keep whole tiles
    plan.full_tiles = tiles - tail_tiles;
    plan.tail_tiles = tail_tiles;
    plan.tail_iters = iters;
    plan.sk_ctas = static_cast<int>(ctas);
    // contributors of tile tl: owner(first iteration) .. owner(last iteration)
    auto owner = [&](int64_t x) { return ((x + 1) * ctas - 1) / iters; };
    int64_t maxc = 1;
    for (int64_t tl = 0; tl < tail_tiles; ++tl) {
        const int64_t c = owner(tl * n_k + n_k - 1) - owner(tl * n_k) + 1;
        if (c > maxc) maxc = c;
    }
    plan.max_contrib = static_cast<int>(maxc);
    return plan;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Scratch the split plan of config Cfg takes for `p`: partial-sum bytes and
// counters (one per dealt-out tile).
template <typename Cfg>
void split_needs(const Problem &p, size_t *part_bytes, size_t *n_counters) {
    const int64_t tiles = ((p.M + Cfg::BM - 1) / Cfg::BM) * ((p.N + Cfg::BN - 1) / Cfg::BN);
    const SplitPlan plan = plan_split<Cfg>(p, tiles);
    *part_bytes = plan.tail_tiles == 0
                      ? 0
                      : align256(static_cast<size_t>(plan.tail_tiles) * plan.max_contrib *
                                 Cfg::BM * Cfg::BN * sizeof(float));
    *n_counters = static_cast<size_t>(plan.tail_tiles);
}

// Only BF16 inputs reach the fused epilogue (gemm_bf16_f32acc_ex); the other
// input types are built without it.
template <typename Cfg, typename T, bool AK, bool BKM>
cudaError_t launch_kernel(bool epi, unsigned grid, const SimtArgs &args, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl_attribute(&attr[0]);
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(Cfg::NT, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (std::is_same<T, uint16_t>::value) {
        if (epi) return cudaLaunchKernelEx(&cfg, sgemm_simt_kernel<Cfg, T, AK, BKM, true>, args);
    } else {
        if (epi) return cudaErrorInvalidValue;
    }
    return cudaLaunchKernelEx(&cfg, sgemm_simt_kernel<Cfg, T, AK, BKM, false>, args);
}

template <typename Cfg, typename T>
cudaError_t launch_cfg(const Problem &p, cudaStream_t stream, const char **name,
                       const FixedScratch *fixed = nullptr) {
    SimtArgs args;
    args.p = p;
    constexpr size_t vbytes = 4 * sizeof(T);
    args.vec_a = aligned(p.A, vbytes) && (p.lda % 4 == 0);
    args.vec_b = aligned(p.B, vbytes) && (p.ldb % 4 == 0);
    args.vec_c = p.beta != 0.f && aligned(p.C, 16) && (p.ldc % 4 == 0);
    args.vec_d = aligned(p.D, 16) && (p.ldd % 4 == 0);
    args.vec_d16 = aligned(p.D, 8) && (p.ldd % 4 == 0);
    args.tiles_m = (p.M + Cfg::BM - 1) / Cfg::BM;
    args.tiles_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int64_t tiles = args.tiles_m * args.tiles_n;
    const SplitPlan plan = plan_split<Cfg>(p, tiles);
    args.full_tiles = plan.full_tiles;
    args.tail_iters = plan.tail_iters > 0 ? plan.tail_iters : 1;
    args.sk_ctas = plan.sk_ctas;
    args.max_contrib = plan.max_contrib;
    args.ws_part = nullptr;
    args.ws_count = nullptr;
    const int64_t units = plan.full_tiles + plan.sk_ctas;

    // workspace for the dealt-out tiles: partial sums, then one counter per tile
    void *ws = nullptr;
    SplitSync sync;  // the stream's split counters, held until the launch is enqueued
    if (plan.tail_tiles > 0) {
        const size_t part_bytes = align256(static_cast<size_t>(plan.tail_tiles) *
                                           plan.max_contrib * Cfg::BM * Cfg::BN * sizeof(float));
        if (fixed != nullptr) {
            // no allocation: the caller's scratch, whose counters are zero
            // between calls (the last contributor of a tile resets its own)
            if (part_bytes > fixed->part_bytes ||
                static_cast<size_t>(plan.tail_tiles) > fixed->n_counters)
                return cudaErrorInvalidValue;
            args.ws_part = static_cast<float *>(fixed->part);
            args.ws_count = fixed->counters;
        } else {
            // partial sums from the pool; counters from the stream's split
            // counters (zero; the last contributor of a tile resets its own)
            cudaError_t e = sync.acquire(stream, static_cast<size_t>(plan.tail_tiles));
            if (e != cudaSuccess) return e;
            args.ws_count = sync.counters;
            e = workspace_alloc(part_bytes, stream, &ws);
            if (e != cudaSuccess) return e;
            args.ws_part = static_cast<float *>(ws);
        }
    }

    const unsigned grid = static_cast<unsigned>(units < 0x7fffffff ? units : 0x7fffffff);
    const int kind = sizeof(T) == 4 ? 0 : (std::is_same<T, __half>::value ? 2 : 1);
    static const char *const names[3][4] = {
        {"sgemm_simt<f32,A:K,B:K>", "sgemm_simt<f32,A:K,B:N>", "sgemm_simt<f32,A:M,B:K>",
         "sgemm_simt<f32,A:M,B:N>"},
        {"sgemm_simt<bf16,A:K,B:K>", "sgemm_simt<bf16,A:K,B:N>", "sgemm_simt<bf16,A:M,B:K>",
         "sgemm_simt<bf16,A:M,B:N>"},
        {"sgemm_simt<f16,A:K,B:K>", "sgemm_simt<f16,A:K,B:N>", "sgemm_simt<f16,A:M,B:K>",
         "sgemm_simt<f16,A:M,B:N>"}};
    const bool epi = p.bias != nullptr || p.act != kActNone || p.d_bf16;
    cudaError_t e = cudaSuccess;
    if (p.a_kmajor && p.b_kmajor) {
        e = launch_kernel<Cfg, T, true, true>(epi, grid, args, stream);
        *name = names[kind][0];
    } else if (p.a_kmajor) {
        e = launch_kernel<Cfg, T, true, false>(epi, grid, args, stream);
        *name = names[kind][1];
    } else if (p.b_kmajor) {
        e = launch_kernel<Cfg, T, false, true>(epi, grid, args, stream);
        *name = names[kind][2];
    } else {
        e = launch_kernel<Cfg, T, false, false>(epi, grid, args, stream);
        *name = names[kind][3];
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (ws != nullptr) {
        const cudaError_t ef = workspace_free(ws, stream);
        if (e == cudaSuccess) e = ef;
    }
    const cudaError_t er = sync.release();
    return e != cudaSuccess ? e : er;
}

__global__ void scale_c_kernel(const Problem p) {
    // D = act(beta * C + bias) (beta may be 0: then C is not read)
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = p.M * p.N;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = e / p.N, j = e % p.N;
        float c = p.beta != 0.f ? p.beta * p.C[i * p.ldc + j] : 0.f;
        if (p.bias != nullptr) c += p.bias_per_row ? p.bias[i] : p.bias[j];
        c = apply_activation(c, p.act);
        if (p.d_bf16)
            reinterpret_cast<uint16_t *>(p.D)[i * p.ldd + j] = to_bf16_bits(c);
        else
            p.D[i * p.ldd + j] = c;
    }
}

}  // namespace

namespace {
// The FP32 kernel choice for K > 0, alpha != 0 (shared by gemm_f32 and
// gemm_f32_noalloc).
enum class F32Kernel { Skinny, Cluster, Tall, Big, Wide, Small };

F32Kernel choose_f32(const Problem &p, int *cluster) {
    auto tiles = [&p](int64_t bm, int64_t bn) {
        return ((p.M + bm - 1) / bm) * ((p.N + bn - 1) / bn);
    };
    const int64_t sms = sm_count();
    *cluster = 0;
    // M <= 8: the small-M kernel streams op(B) once
    if (skinny_eligible(p)) return F32Kernel::Skinny;
    // few 64 x 64 tiles and a K that splits into 2-8 short slices: the
    // cluster kernel (its pieces add up in shared memory, not through a
    // global-memory workspace)
    const int cl = sgemm_cluster_size(p, static_cast<int>(sms));
    if (cl > 0) {
        *cluster = cl;
        return F32Kernel::Cluster;
    }
    // otherwise a D of at most 64 columns takes 256 x 64 tiles; 128 x 256
    // tiles when there are two waves of them and K is long enough to carry
    // their epilogue; else 128 x 128 tiles if there are enough of them for
    // the stream-K tail to spread; else 64 x 64
    if (p.N <= TallCfg::BN) return F32Kernel::Tall;
    if (tiles(BigCfg::BM, BigCfg::BN) >= 2 * sms && p.K >= 2048) return F32Kernel::Big;
    if (tiles(WideCfg::BM, WideCfg::BN) * 4 >= sms) return F32Kernel::Wide;
    return F32Kernel::Small;
}
}  // namespace

cudaError_t launch_f32(const Problem &p, cudaStream_t stream, const char **name,
                       const FixedScratch *fixed) {
    int cl = 0;
    switch (choose_f32(p, &cl)) {
        case F32Kernel::Skinny: return launch_skinny(p, InType::F32, stream, name, fixed);
        case F32Kernel::Cluster: return launch_sgemm_cluster(p, cl, stream, name);
        case F32Kernel::Tall: return launch_cfg<TallCfg, float>(p, stream, name, fixed);
        case F32Kernel::Big: return launch_cfg<BigCfg, float>(p, stream, name, fixed);
        case F32Kernel::Wide: return launch_cfg<WideCfg, float>(p, stream, name, fixed);
        case F32Kernel::Small: break;
    }
    return launch_cfg<SmallCfg, float>(p, stream, name, fixed);
}

void f32_scratch_needs(const Problem &p, size_t *part_bytes, size_t *n_counters) {
    int cl = 0;
    *part_bytes = 0;
    *n_counters = 0;
    switch (choose_f32(p, &cl)) {
        case F32Kernel::Skinny: skinny_scratch_needs(p, InType::F32, part_bytes, n_counters); return;
        case F32Kernel::Cluster: return;  // pieces meet in distributed shared memory
        case F32Kernel::Tall: split_needs<TallCfg>(p, part_bytes, n_counters); return;
        case F32Kernel::Big: split_needs<BigCfg>(p, part_bytes, n_counters); return;
        case F32Kernel::Wide: split_needs<WideCfg>(p, part_bytes, n_counters); return;
        case F32Kernel::Small: break;
    }
    split_needs<SmallCfg>(p, part_bytes, n_counters);
}

cudaError_t launch_simt(const Problem &p, InType in, cudaStream_t stream, const char **name) {
    if (in == InType::F32) return launch_f32(p, stream, name);
    const bool big = ((p.M + BigCfg::BM - 1) / BigCfg::BM) * ((p.N + BigCfg::BN - 1) / BigCfg::BN) >=
                     sm_count();
    if (in == InType::F16)
        return big ? launch_cfg<BigCfg, __half>(p, stream, name)
                   : launch_cfg<SmallCfg, __half>(p, stream, name);
    return big ? launch_cfg<BigCfg, uint16_t>(p, stream, name)
               : launch_cfg<SmallCfg, uint16_t>(p, stream, name);
}

// ----------------------------------------------------- fixed scratch array
// For callers that cannot allocate device memory (gemm_f32_noalloc): the
// split pieces' counters and partial sums live in this file-scope array
// instead of pool memory.  Every device that loads the library holds it
// until the process exits.  In host code the name g_fixed_scratch is only a
// host-side stand-in for the array, not a device address: the device
// address is looked up per device with cudaGetSymbolAddress (with that
// device current) and passed to the kernels.  Layout: kFixedCounterBytes of
// counters, then partial sums.  The counters are zeroed at set-up, and every
// kernel that counts on them leaves them at zero (the last piece of a tile
// resets its counter), so no call clears them.
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

namespace {
constexpr int kMaxScratchDevices = 64;
struct FixedScratchSetup {
    std::mutex m;
    bool done = false;
    void *ptr = nullptr;
};
FixedScratchSetup g_fixed_setup[kMaxScratchDevices];
}  // namespace

cudaError_t fixed_scratch(FixedScratch *out, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    FixedScratchSetup &su = g_fixed_setup[dev];
    {
        std::lock_guard<std::mutex> lock(su.m);
        if (!su.done) {
            // set-up, once per device with the device current: the array's
            // device address, and zeroed counters before any kernel uses them
            cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
            if ((e = cudaStreamIsCapturing(stream, &capture)) != cudaSuccess) return e;
            if (capture != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
            void *ptr = nullptr;
            if ((e = cudaGetSymbolAddress(&ptr, g_fixed_scratch)) != cudaSuccess) return e;
            if ((e = cudaMemsetAsync(ptr, 0, kFixedCounterBytes, stream)) != cudaSuccess) return e;
            if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
            su.ptr = ptr;
            su.done = true;
        }
    }
    out->counters = static_cast<int *>(su.ptr);
    out->n_counters = kFixedCounterBytes / sizeof(int);
    out->part = static_cast<unsigned char *>(su.ptr) + kFixedCounterBytes;
    out->part_bytes = kFixedScratchBytes - kFixedCounterBytes;
    return cudaSuccess;
}

cudaError_t launch_scale_c(const Problem &p, cudaStream_t stream, const char **name) {
    const int64_t total = p.M * p.N;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    set_pdl_attribute(&attr[0]);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, scale_c_kernel, p);
    *name = "scale_c";
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace gemm
