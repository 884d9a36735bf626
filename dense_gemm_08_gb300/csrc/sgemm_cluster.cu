// sgemm_cluster.cu -- FP32 CUDA-core GEMM for small problems: the K range of
// every 64 x 64 tile is split over the CTAs of one thread-block cluster, and
// the partial tiles are added through distributed shared memory.
//
// A small problem (FP32 256^3 has sixteen 64 x 64 tiles) leaves most SMs
// idle unless K is split ("GEMM on NVIDIA GPUs", section 5, split-K for
// problems with few output tiles).  The CUDA-core kernel's split sends the
// pieces through global memory and lets the last one add them, which puts
// two more memory round trips on a critical path of a few microseconds.
// Here the CL pieces of a tile are the CL CTAs of one cluster (CL = 2, 4 or
// 8): each multiplies its K slice into a partial tile in its own shared
// memory; after a cluster barrier, CTA r adds rows [r 64/CL, (r+1) 64/CL) of
// all CL partials, read from the other CTAs' shared memory in rank order, and
// writes D = alpha * sum + beta * C.  The sum order is fixed, so results do
// not depend on timing.  No workspace, no counters, no second kernel.
//
// Per CTA: 256 threads; the K slice is walked in chunks of 32.  Every
// thread fetches 8 elements of op(A) and 8 of op(B) per chunk (coalesced
// along whichever dimension is contiguous, zero past the matrix and past the
// slice), the next chunk's while the current one is multiplied.  Shared
// memory holds op(A) as [m][k] and op(B) as [n][k], rows padded to 33 words
// so that both the transposing stores and the fragment reads avoid bank
// conflicts.  Thread (ty, tx) of a 16 x 16 grid owns rows ty + 16 i and
// columns tx + 16 j (i, j < 4) of the tile.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace gemm {
namespace {

constexpr int kTile = 64;    // tile rows and columns
constexpr int kChunk = 32;   // K per shared-memory chunk
constexpr int kThreads = 256;
constexpr int kPad = kChunk + 1;       // row stride of the staged operands (words)
constexpr int kMaxChunksPerSlice = 4;  // K slices of at most 128

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float of CTA `rank`'s shared memory at the address of `local` in this CTA.
__device__ __forceinline__ float load_peer(const float *local, uint32_t rank) {
    const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

struct ClusterArgs {
    const float *A, *B, *C;
    float *D;
    int64_t M, N, K, lda, ldb, ldc, ldd;
    float alpha, beta;
    int64_t tiles_n;
    int64_t ks;  // K per slice (a multiple of kChunk)
};

// Element e (0 .. 2047) of a 64 x 32 chunk, in the order that walks the
// contiguous dimension fastest: its (row, k) within the chunk.
template <bool KContig>
__device__ __forceinline__ void chunk_coords(int e, int &row, int &k) {
    if (KContig) {
        row = e >> 5;
        k = e & (kChunk - 1);
    } else {
        k = e >> 6;
        row = e & (kTile - 1);
    }
}

// op(A) rows m0.., op(B) columns n0..: 8 values each for this thread.
template <bool AK, bool BKM>
__device__ __forceinline__ void fetch_chunk(const ClusterArgs &a, int64_t m0, int64_t n0,
                                            int64_t k0, int64_t k_end, float (&ra)[8],
                                            float (&rb)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = threadIdx.x + kThreads * j;
        int r, k;
        chunk_coords<AK>(e, r, k);
        const int64_t gm = m0 + r, gka = k0 + k;
        ra[j] = (gm < a.M && gka < k_end)
                    ? __ldg(AK ? a.A + gm * a.lda + gka : a.A + gm + gka * a.lda)
                    : 0.f;
        chunk_coords<BKM>(e, r, k);
        const int64_t gn = n0 + r, gkb = k0 + k;
        rb[j] = (gn < a.N && gkb < k_end)
                    ? __ldg(BKM ? a.B + gn * a.ldb + gkb : a.B + gkb * a.ldb + gn)
                    : 0.f;
    }
}

template <bool AK, bool BKM>
__device__ __forceinline__ void stage_chunk(float *as, float *bs, const float (&ra)[8],
                                            const float (&rb)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = threadIdx.x + kThreads * j;
        int r, k;
        chunk_coords<AK>(e, r, k);
        as[r * kPad + k] = ra[j];
        chunk_coords<BKM>(e, r, k);
        bs[r * kPad + k] = rb[j];
    }
}

template <int CL, bool AK, bool BKM>
__global__ void __launch_bounds__(kThreads) sgemm_cluster_kernel(const ClusterArgs a) {
    // staged operands; after the K loop the same words hold the partial tile
    __shared__ __align__(16) float smem[2 * kTile * kPad];
    static_assert(kTile * kTile <= 2 * kTile * kPad, "the partial tile reuses the staging");
    float *as = smem, *bs = smem + kTile * kPad;

    pdl_wait();  // the previous kernel on the stream is done with its memory
    pdl_launch_dependents();
    const uint32_t rank = cluster_rank();
    const int64_t tile = blockIdx.x / CL;
    const int64_t m0 = (tile / a.tiles_n) * kTile, n0 = (tile % a.tiles_n) * kTile;
    const int64_t k_begin = static_cast<int64_t>(rank) * a.ks;
    const int64_t k_end = k_begin + a.ks < a.K ? k_begin + a.ks : a.K;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    float ra[8], rb[8];
    if (k_begin < k_end) fetch_chunk<AK, BKM>(a, m0, n0, k_begin, k_end, ra, rb);
    for (int64_t k0 = k_begin; k0 < k_end; k0 += kChunk) {
        __syncthreads();  // the previous chunk has been multiplied
        stage_chunk<AK, BKM>(as, bs, ra, rb);
        __syncthreads();
        if (k0 + kChunk < k_end) fetch_chunk<AK, BKM>(a, m0, n0, k0 + kChunk, k_end, ra, rb);
#pragma unroll 8
        for (int k = 0; k < kChunk; ++k) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = as[(ty + 16 * i) * kPad + k];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = bs[(tx + 16 * j) * kPad + k];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
    }

    // this CTA's partial tile, row-major 64 x 64
    __syncthreads();
    float *part = smem;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[(ty + 16 * i) * kTile + tx + 16 * j] = acc[i][j];
    cluster_barrier();  // every CTA's partial is in place

    // rows [rank R, rank R + R) of the tile: the CL partials added in rank order
    constexpr int R = kTile / CL;
    for (int idx = threadIdx.x; idx < R * kTile; idx += kThreads) {
        const int row = static_cast<int>(rank) * R + idx / kTile, col = idx % kTile;
        const int64_t gm = m0 + row, gn = n0 + col;
        if (gm >= a.M || gn >= a.N) continue;
        float s = 0.f;
#pragma unroll
        for (int src = 0; src < CL; ++src) s += load_peer(part + row * kTile + col, src);
        float o = a.alpha * s;
        if (a.beta != 0.f) o = fmaf(a.beta, a.C[gm * a.ldc + gn], o);
        a.D[gm * a.ldd + gn] = o;
    }
    cluster_barrier();  // no CTA leaves while another still reads its partial
}

template <int CL, bool AK, bool BKM>
cudaError_t launch_layout(const ClusterArgs &a, unsigned grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl_attribute(&attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, sgemm_cluster_kernel<CL, AK, BKM>, a);
}

// Whether the current device can hold at least one cluster of CL CTAs of
// this kernel at a time (asked once per device and cluster size).
template <int CL>
bool cluster_fits() {
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static bool fits[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::call_once(once[dev], [dev] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = CL;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        const cudaError_t e =
            cudaOccupancyMaxActiveClusters(&n, sgemm_cluster_kernel<CL, true, false>, &cfg);
        fits[dev] = e == cudaSuccess && n > 0;
        if (e != cudaSuccess) cudaGetLastError();  // a refused query is not a launch error
    });
    return fits[dev];
}

template <int CL>
cudaError_t launch_cl(const ClusterArgs &a, bool ak, bool bk, unsigned grid, cudaStream_t stream) {
    if (ak && bk) return launch_layout<CL, true, true>(a, grid, stream);
    if (ak) return launch_layout<CL, true, false>(a, grid, stream);
    if (bk) return launch_layout<CL, false, true>(a, grid, stream);
    return launch_layout<CL, false, false>(a, grid, stream);
}

}  // namespace

int sgemm_cluster_size(const Problem &p, int sms) {
    if (p.M < 1 || p.N < 1 || p.K < 1) return 0;
    const int64_t tiles = ((p.M + kTile - 1) / kTile) * ((p.N + kTile - 1) / kTile);
    // the most K pieces per tile with one CTA per SM, every piece at least
    // one chunk long and at most kMaxChunksPerSlice chunks, in clusters the
    // device can schedule
    for (int cl = 8; cl >= 2; cl /= 2) {
        if (tiles * cl > sms) continue;
        if (p.K < static_cast<int64_t>(cl) * kChunk) continue;
        if (p.K > static_cast<int64_t>(cl) * kChunk * kMaxChunksPerSlice) continue;
        const bool fits = cl == 8 ? cluster_fits<8>() : cl == 4 ? cluster_fits<4>() : cluster_fits<2>();
        if (!fits) continue;
        return cl;
    }
    return 0;
}

cudaError_t launch_sgemm_cluster(const Problem &p, int cl, cudaStream_t stream,
                                 const char **name) {
    if (cl != 2 && cl != 4 && cl != 8) return cudaErrorInvalidValue;
    ClusterArgs a;
    a.A = static_cast<const float *>(p.A);
    a.B = static_cast<const float *>(p.B);
    a.C = p.C;
    a.D = p.D;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.lda = p.lda;
    a.ldb = p.ldb;
    a.ldc = p.ldc;
    a.ldd = p.ldd;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.tiles_n = (p.N + kTile - 1) / kTile;
    const int64_t per = (p.K + cl - 1) / cl;
    a.ks = (per + kChunk - 1) / kChunk * kChunk;
    const int64_t grid = ((p.M + kTile - 1) / kTile) * a.tiles_n * cl;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    const unsigned g = static_cast<unsigned>(grid);
    cudaError_t e;
    if (cl == 8) {
        e = launch_cl<8>(a, p.a_kmajor, p.b_kmajor, g, stream);
        *name = "sgemm_cluster<f32,ks:8>";
    } else if (cl == 4) {
        e = launch_cl<4>(a, p.a_kmajor, p.b_kmajor, g, stream);
        *name = "sgemm_cluster<f32,ks:4>";
    } else {
        e = launch_cl<2>(a, p.a_kmajor, p.b_kmajor, g, stream);
        *name = "sgemm_cluster<f32,ks:2>";
    }
    return e;
}

}  // namespace gemm
