// gemm_tc.cu -- BF16- or FP16-input, FP32-accumulate GEMM on the sm_103a tensor cores.
//
// D = alpha * op(A) * op(B) + beta * C, D row-major FP32.
//
// Design (what the pages prescribe, rebuilt for tcgen05):
//   * Accumulators live in tensor memory (TMEM); A and B are read by the
//     tensor core straight from shared memory through matrix descriptors
//     ("GEMM on NVIDIA GPUs", section 4, "Tensor Core pipeline": on
//     Blackwell tcgen05.mma keeps the accumulator in TMEM and takes B from
//     shared memory).
//   * TMA fills a multi-stage ring of 128-byte-swizzled A/B tiles; full/empty
//     mbarriers hand each stage from the load warp to the MMA warp and back
//     ("Worklog: optimising GEMM on NVIDIA H100", kernel 7 TMA + barriers,
//     and the producer/consumer pipeline after kernel 8).
//   * Warp roles: warp 0 issues TMA (one lane), warp 1 owns TMEM and issues
//     tcgen05.mma (one lane), warps 2-5 run the epilogue.
//   * Persistent grid, static round-robin over output tiles in grouped order
//     along M so that tiles running together share A and B panels in L2
//     ("GEMM on NVIDIA GPUs", section 5 / grouped schedulers); every other
//     round walks K backwards, so a round starts on the K blocks the one
//     before it read last (still in L2).
//   * Two TMEM accumulators (2 x 256 columns): the epilogue of tile i runs
//     while the MMA warp accumulates tile i + 1.
//   * Epilogue: tcgen05.ld TMEM -> registers, D = alpha * acc + beta * C
//     (C read only when beta != 0), guarded stores; tiles past the matrix
//     edge are zero-filled by TMA on the way in and clipped on the way out.
//   * Every barrier wait is bounded; a wait that runs out records a timeout
//     in a device status word, the CTA drains what it has in flight, frees
//     TMEM and exits.
//
// Two variants (template parameter CG, the tcgen05 CTA group):
//   CG = 1: one CTA per tile of 128 x 256; each 128 x 256 x 16 MMA reads
//           4 KiB of A and 8 KiB of B from the CTA's shared memory.
//   CG = 2: a cluster of two CTAs on neighbouring SMs shares a 256 x 256
//           tile (tcgen05 cta_group::2).  Each CTA loads its own 128 rows of
//           A and its own 128 columns of B (no multicast); the MMA, issued
//           by the even CTA, reads both CTAs' shared memory and writes each
//           CTA's 128 rows of the accumulator into that CTA's TMEM.  Shared
//           memory traffic per MMA and L2 traffic for B halve, and a stage
//           shrinks to 32 KiB, so six stages fit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "epilogue.cuh"
#include "internal.h"

namespace gemm {
namespace {

constexpr int BK = 64;  // 64 BF16 = 128 bytes = one swizzle row
constexpr int UMMA_K = 16;
constexpr int BM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;  // tile width = MMA N
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;  // 512: all of TMEM
constexpr int kGroupM = 16;               // grouped raster width (tile rows)

// Depth of the CTA pair's operand ring (stages of 32 KiB per CTA).  With the
// epilogue's staging boxes (64 KiB) five stages fit; without them (the
// direct epilogue, below) seven.  A build may set fewer
// (-DGEMM_TC_PAIR_STAGES=S, 2 <= S <= 5; -DGEMM_TC_DIRECT_STAGES=S,
// 2 <= S <= 7) to measure throughput against depth.
#ifndef GEMM_TC_PAIR_STAGES
#define GEMM_TC_PAIR_STAGES 5
#endif
#ifndef GEMM_TC_DIRECT_STAGES
#define GEMM_TC_DIRECT_STAGES 7
#endif
// Debug build (-DGEMM_TC_DEBUG=1): every ring at its smallest depth (2
// stages, the fewest the MMA loop's two-stage rounds take) and a grid of one
// work item per CTA (or pair) instead of the persistent one, so that a wrong
// result can be told apart from a ring or phase mistake.  Same results
// contract; for checking, not for speed.
#ifndef GEMM_TC_DEBUG
#define GEMM_TC_DEBUG 0
#endif
constexpr bool kDebug = GEMM_TC_DEBUG != 0;
static_assert(GEMM_TC_PAIR_STAGES >= 2 && GEMM_TC_PAIR_STAGES <= 5,
              "the staged pair ring holds 2 to 5 stages");
static_assert(GEMM_TC_DIRECT_STAGES >= 2 && GEMM_TC_DIRECT_STAGES <= 7,
              "the direct pair ring holds 2 to 7 stages");

// DIRECT (CTA pairs only): the epilogue moves each accumulator row from
// registers straight to D with 32-byte stores (and reads C the same way), and
// a split tile's pieces travel the same way, so the kernel needs no staging
// boxes and the ring takes their shared memory.  For D (and C, when
// beta != 0) rows that start on 32 bytes.
template <int CG, bool DIRECT = false>
struct Cfg {
    static_assert(!DIRECT || CG == 2, "the direct epilogue is built for CTA pairs");
    static constexpr int TILE_M = BM * CG;  // tile rows covered by the CTA group
    static constexpr int B_ROWS = BN / CG;  // B columns (N) held by each CTA
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // (the debug build keeps the same shared-memory layout, using 2 stages)
    static constexpr int STAGES =
        CG == 1 ? 4 : (DIRECT ? GEMM_TC_DIRECT_STAGES : GEMM_TC_PAIR_STAGES);
    static constexpr int RING_STAGES = kDebug ? 2 : STAGES;  // stages the ring cycles through
    // single CTAs with a narrow B tile (N <= 128: 64 or 128 rows of B per
    // stage) cut the same ring into more, smaller stages, at most 8
    static constexpr int MAX_STAGES = CG == 1 ? 8 : STAGES;
    // epilogue warps: eight (two per TMEM lane quarter) for the staged CTA
    // pair, whose epilogue is its limit when K is short; four otherwise.
    // Each has two 32 x 32 FP32 boxes of 4 KiB (C for the next chunk
    // arrives in one while the other is in use).
    static constexpr int EPI_WARPS = (CG == 2 && !DIRECT) ? 8 : 4;
    static constexpr int BOXES = 2;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int STAGING_BYTES = DIRECT ? 0 : EPI_WARPS * BOXES * 32 * 32 * 4;
    // ring + staging + barriers + slack for aligning the ring to 1024 bytes
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 512;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
};

__device__ int g_tc_status;  // 0 = fine, 1 = a bounded wait ran out

// Single-CTA split-K: the K range of a 128 x 256 tile is split over the CTAs
// of one cluster, at most the largest portable cluster.
constexpr int kMaxClusterK = 8;

// Shared memory the owner of a split tile's chunks receives the other
// pieces' chunks in: per lane quarter, (ks - 1) slots of 4 KiB for each of
// its at most ceil(8 / ks) chunks; the largest over ks = 2..kMaxClusterK.
constexpr int split_slots_bytes(int ks) { return 4 * (ks - 1) * ((BN / 32 + ks - 1) / ks) * 4096; }
constexpr int max_split_slots_bytes(int ks = 2) {
    return ks > kMaxClusterK ? 0
                             : (split_slots_bytes(ks) > max_split_slots_bytes(ks + 1)
                                    ? split_slots_bytes(ks)
                                    : max_split_slots_bytes(ks + 1));
}
static_assert(max_split_slots_bytes() <= Cfg<1>::STAGES * Cfg<1>::STAGE_BYTES,
              "the single-CTA ring holds every split size's receive slots");

struct TcArgs {
    int64_t M, N, K;
    float alpha, beta;
    const float *C;
    int64_t ldc;
    float *D;
    int64_t ldd;
    int64_t tiles_m, tiles_n, num_kb;
    int a_kmajor, b_kmajor;
    // Split-K (fewer tiles than SMs): work item w is tile w / ks, K blocks
    // [num_kb * s / ks, num_kb * (s + 1) / ks) with s = w % ks (see
    // cluster_k).
    int ks;
    // CTA pairs, last partial round: tiles from tail_first on are split into
    // tail_ks K ranges, one work item each.  Each piece's epilogue warps
    // publish their 32-row slab of partial sums in ws and count themselves in
    // ws_count[((tile - tail_first) * 2 + rank) * 4 + warp]; the last piece
    // to arrive adds the slabs in K order and writes D (no piece waits for
    // another).
    int64_t tail_first;
    int tail_ks;
    // CG = 2, tail_split_n: the tail tiles are instead split along N into
    // tail_ks = 2 halves of BN / 2 columns, each over the whole K range (no
    // partial sums, no reduction; B comes through map_b_half).
    int tail_split_n;
    float *ws;
    int *ws_count;  // the stream's split counters: zero between calls
    // CG = 1 split-K: the ks pieces of a tile are the CTAs of one cluster
    // (cluster rank = piece), which add their partial sums through
    // distributed shared memory (no workspace)
    int cluster_k;
    // CG = 1: columns of B per tile (BN, or 64 / 128 when N fits: one tile
    // column, a narrower B box and N = bn1 MMAs) and the ring cut to match
    int bn1;
    int stages1;
    uint32_t stage_bytes1;
    // CG = 1: rows of A loaded per stage (BM, or 16 / 32 / 64 when M fits:
    // the rows past them in shared memory hold stale values, which reach
    // only accumulator rows past M -- rows of D that are never stored), and
    // likewise rows of a K-contiguous B (bn1, or 16 / 32 when N fits; the
    // stale rows reach only columns past N)
    int am1;
    int bk1;
    // CG = 1: bytes of A at the start of each stage, B after them (BM rows,
    // or am1 rows packed tight: the MMA's 128-row A operand then runs on
    // into B and the next stage, stale rows that reach only rows past M)
    uint32_t a_region1;
    int ab_format;  // operand format of A and B for kind::f16: 1 = BF16, 0 = FP16
    // fused epilogue: D = act(alpha * acc + beta * C + bias), FP32 or BF16
    const float *bias;
    int bias_per_row;
    int act;
    int d_bf16;
    int tma_c;  // C is read through TMA boxes (16-byte aligned base and pitch)
    int tma_d;  // D is written through TMA boxes
    uint64_t timeout_ns;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// 16 bytes into the shared memory of a CTA of the cluster (address from
// map_to_rank); a cluster barrier makes them visible to that CTA.
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

// Every thread of every CTA of the cluster; the warp converges first (the
// .aligned form wants all its lanes at the same instruction).
__device__ __forceinline__ void cluster_sync() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier of another CTA of the cluster (address from map_to_rank).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up
// (returns false) when the CTA's abort flag is raised or after timeout_ns.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             const volatile int *abort_flag,
                                             uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (*abort_flag) return false;
            if (global_timer() - start > timeout_ns) return false;
        }
    }
}

__device__ __forceinline__ void raise_abort(volatile int *abort_flag) {
    *abort_flag = 1;
    atomicExch(&g_tc_status, 1);
}

// 2-D tiled TMA load into this CTA's shared memory; completion is signalled
// on `bar`.  CG = 2: `bar` may live in the peer CTA (cluster address).
template <int CG>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                            int32_t c1, uint32_t bar) {
    if constexpr (CG == 1) {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
            : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
            : "memory");
    }
}

// 2-D tiled TMA store of a shared-memory box to global memory (bulk group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int32_t c0, int32_t c1,
                                             uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from shared to global memory (bulk group).
__device__ __forceinline__ void bulk_copy_to_global(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from global to this CTA's shared
// memory; completion is counted on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_copy_to_shared(uint32_t dst, const void *src, uint32_t bytes,
                                                    uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Wait until at most N bulk groups of this thread are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once all tcgen05 operations issued so far by this thread
// have completed.  CG = 2: on the barrier at the same offset in both CTAs.
template <int CG>
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    if constexpr (CG == 1) {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    } else {
        const uint16_t both = 0x3;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(bar),
            "h"(both)
            : "memory");
    }
}

// Arrive on this CTA's `bar` once all tcgen05 operations issued so far by
// this thread have completed (a kernel may use only one CTA-group size).
template <int CG>
__device__ __forceinline__ void tc_commit_local(uint32_t bar) {
    if constexpr (CG == 1) {
        tc_commit<1>(bar);
    } else {
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    }
}

template <int CG>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (CG == 1) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t slot) {
    if constexpr (CG == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
    if constexpr (CG == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base),
                     "r"(TMEM_COLS)
                     : "memory");
    } else {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// 32 lanes x 32 columns of 32-bit TMEM words: thread t of the warp gets its
// lane's 32 consecutive columns.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------- matrix descriptors
// tcgen05 shared-memory matrix descriptor (64 bits):
//   [0,14)  start address >> 4        [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4
//   [46,48) version = 1               [49,52) base offset (0: atoms 1024-aligned)
//   [52]    LBO mode = 0              [61,64) swizzle: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// K-major operand: rows of 64 BF16 (128 B), 8-row swizzle atoms of 1 KiB
// stacked along M/N (SBO = 1024).  The k-th 16-wide slice starts 32 B in.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
    return smem_desc(tile + kk * UMMA_K * 2, 16, 1024);
}

// MN-major operand: per 64-element MN block, 64 K-rows of 128 B (8 KiB);
// blocks stacked along MN (LBO = 8 KiB), 8-row groups along K (SBO = 1 KiB).
// The k-th 16-deep slice starts 16 rows = 2 KiB in.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
    return smem_desc(tile + kk * UMMA_K * 128, 64 * 128, 1024);
}

// Instruction descriptor, kind::f16: D FP32 (bits 4-5 = 1), A and B format
// (bits 7-9 and 10-12: 1 = BF16, 0 = FP16), A/B major-ness (bit 15 / 16:
// 0 = K-major, 1 = MN-major), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, int a_mn_major, int b_mn_major,
                                                  int ab_format) {
    return (1u << 4) | (static_cast<uint32_t>(ab_format) << 7) |
           (static_cast<uint32_t>(ab_format) << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
           (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// Work item w of the persistent loop: tile t, piece sp of nsp, K blocks
// [kb_begin, kb_end).  CG = 1: every tile is split into ks pieces (ks = 1:
// whole tiles).  CG = 2: whole tiles, then the split tail tiles.
struct WorkItem {
    int64_t t, kb_begin, kb_end;
    int sp, nsp;         // K piece sp of nsp (nsp = 1: the whole K range)
    int n_off, n_width;  // columns [n_off, n_off + n_width) of the tile (BN unless split along N)
};

// Work items and tiles number below 2^31 (the host checks), so the index
// arithmetic is unsigned 32-bit: a 64-bit division costs several times as
// much, and the first item's arithmetic lies on the kernel's start-up path.
template <int CG>
__device__ __forceinline__ WorkItem work_item(int64_t w, const TcArgs &a) {
    WorkItem it;
    const uint32_t w32 = static_cast<uint32_t>(w);
    if (CG == 1) {
        const uint32_t ks = static_cast<uint32_t>(a.ks);
        it.t = w32 / ks;
        it.sp = static_cast<int>(w32 % ks);
        it.nsp = a.ks;
    } else if (w < a.tail_first) {
        it.t = w;
        it.sp = 0;
        it.nsp = 1;
    } else {
        const uint32_t r = w32 - static_cast<uint32_t>(a.tail_first);
        const uint32_t tks = static_cast<uint32_t>(a.tail_ks);
        it.t = a.tail_first + r / tks;
        it.sp = static_cast<int>(r % tks);
        it.nsp = a.tail_ks;
    }
    it.n_off = 0;
    it.n_width = CG == 1 ? a.bn1 : BN;
    if (CG == 2 && a.tail_split_n && w >= a.tail_first) {
        // an N half of a tail tile, whole K
        it.n_off = it.sp * (BN / 2);
        it.n_width = BN / 2;
        it.sp = 0;
        it.nsp = 1;
    }
    // num_kb < 2^25 (K < 2^31), times a piece index below 8
    const uint32_t nkb = static_cast<uint32_t>(a.num_kb), nsp = static_cast<uint32_t>(it.nsp);
    it.kb_begin = nkb * static_cast<uint32_t>(it.sp) / nsp;
    it.kb_end = nkb * static_cast<uint32_t>(it.sp + 1) / nsp;
    return it;
}

template <int CG>
__device__ __forceinline__ int64_t work_items(const TcArgs &a) {
    const int64_t tiles = a.tiles_m * a.tiles_n;
    return CG == 1 ? tiles * a.ks : a.tail_first + (tiles - a.tail_first) * a.tail_ks;
}

__device__ __forceinline__ void tile_coords(int64_t t, const TcArgs &a, int64_t &tm,
                                            int64_t &tn) {
    const uint32_t t32 = static_cast<uint32_t>(t);
    const uint32_t width = kGroupM * static_cast<uint32_t>(a.tiles_n);
    const uint32_t group = t32 / width, in_group = t32 - group * width;
    const uint32_t first_m = group * kGroupM;
    const uint32_t rest = static_cast<uint32_t>(a.tiles_m) - first_m;
    const uint32_t gsz = rest < static_cast<uint32_t>(kGroupM) ? rest : kGroupM;
    const uint32_t q = in_group / gsz;
    tm = first_m + (in_group - q * gsz);
    tn = q;
}

// ---------------------------------------------------------- epilogue boxes
// Each epilogue warp owns two 32 x 32 FP32 boxes in shared memory, laid out
// with the 128-byte swizzle: element (r, c) sits at byte r * 128 +
// ((c / 4) ^ (r % 8)) * 16 + (c % 4) * 4.  Thread r reading or writing its own
// row as eight 16-byte pieces, and the warp reading or writing one row with
// one element per lane, are both free of bank conflicts; a TMA box with
// CU_TENSOR_MAP_SWIZZLE_128B uses the same layout.
__device__ __forceinline__ uint32_t box_offset(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((((c >> 2) ^ (r & 7))) << 4) + (c & 3) * 4);
}

// A split-K slot holds a 32 x 32 FP32 chunk with columns 4 * j4 .. 4 * j4 + 3
// of row r at byte j4 * 512 + r * 16: the warp's 16-byte store (or load) of
// one j4 covers 512 contiguous bytes, which the cluster's shared-memory
// network moves in a few wide transfers (a row-per-lane layout would make
// each lane's 16 bytes a transfer of its own).
__device__ __forceinline__ uint32_t slot_offset(int r, int j4) {
    return static_cast<uint32_t>(j4 * 512 + r * 16);
}

// Rows of the 32-row block at row0 that lie inside the matrix (0 to 32).
__device__ __forceinline__ int rows_inside(const TcArgs &a, int64_t row0) {
    const int64_t left = a.M - row0;
    return left <= 0 ? 0 : (left >= 32 ? 32 : static_cast<int>(left));
}

// Start copying C[row0 + rr, c0 + lane], rr < 32, into the box with 4-byte
// asynchronous copies (one coalesced row per instruction; elements outside
// the matrix are zero-filled) and commit them as one group of this thread.
// The row pointer advances by ldc and the box address is fixed per row, so
// a row costs a handful of instructions.
__device__ __forceinline__ void box_load_rows_async(uint8_t *box, const TcArgs &a, int64_t row0,
                                                    int64_t c0, int lane) {
    const int nrows = rows_inside(a, row0);
    const bool col_ok = c0 + lane < a.N;
    const float *src = a.C + (nrows > 0 ? row0 * a.ldc + c0 + lane : 0);
    const uint32_t dst = smem_addr(box) + static_cast<uint32_t>((lane & 3) * 4);
    const uint32_t quad = static_cast<uint32_t>(lane >> 2);
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
        const bool ok = col_ok && rr < nrows;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                         dst + static_cast<uint32_t>(rr * 128) + ((quad ^ (rr & 7)) << 4)),
                     "l"(ok ? src : a.C), "r"(ok ? 4 : 0)
                     : "memory");
        src += a.ldc;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's asynchronous-copy groups are pending.
template <int N>
__device__ __forceinline__ void async_copy_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The box into D[row0 + rr, c0 + lane], one coalesced row per step, clipped
// to the matrix.
__device__ __forceinline__ void box_store_rows(const uint8_t *box, const TcArgs &a, int64_t row0,
                                               int64_t c0, int lane) {
    const int nrows = rows_inside(a, row0);
    const bool col_ok = c0 + lane < a.N;
    // all 32 box reads first: a read placed after a store to D could not be
    // started before it (the compiler cannot tell the two pointers apart),
    // which would make every row wait out a shared-memory round trip
    float d[32];
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) d[rr] = *reinterpret_cast<const float *>(box + box_offset(rr, lane));
    float *dp = a.D + (nrows > 0 ? row0 * a.ldd + c0 + lane : 0);
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
        if (col_ok && rr < nrows) *dp = d[rr];
        dp += a.ldd;
    }
}

// BF16 box (32 rows of 64 bytes, unswizzled) into D[row0 + rr, c0 + lane],
// one coalesced row per step, clipped to the matrix.
__device__ __forceinline__ void box_store_rows_bf16(const uint8_t *box, const TcArgs &a,
                                                    int64_t row0, int64_t c0, int lane) {
    const int nrows = rows_inside(a, row0);
    const bool col_ok = c0 + lane < a.N;
    uint16_t d[32];  // all box reads before the first store, as in box_store_rows
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) d[rr] = *reinterpret_cast<const uint16_t *>(box + rr * 64 + lane * 2);
    uint16_t *dp = reinterpret_cast<uint16_t *>(a.D) + (nrows > 0 ? row0 * a.ldd + c0 + lane : 0);
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
        if (col_ok && rr < nrows) *dp = d[rr];
        dp += a.ldd;
    }
}

// 32 bytes (eight 32-bit words) to global memory in one store.
__device__ __forceinline__ void st_global_v8(void *p, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                             uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0),
                 "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}

// 32 bytes from global memory through L2 only (data other CTAs wrote).
__device__ __forceinline__ void ld_global_cg_v8(const float *p, float (&v)[8]) {
    asm volatile("ld.global.cg.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                   "=f"(v[6]), "=f"(v[7])
                 : "l"(p)
                 : "memory");
}

// Direct epilogue: one lane's 32 values C(row, c0 + j), j < 32, into c
// (32-byte loads through L2 when the 32 columns are inside the matrix,
// guarded scalar loads at its edge, zeros past it).  Each element of C is
// read by the thread that later writes the same element of D, before it
// does, so C may be D (in-place update).
__device__ __forceinline__ void load_c_row_direct(const TcArgs &a, int64_t row, int64_t c0,
                                                  float (&c)[32]) {
    if (row >= a.M) {
#pragma unroll
        for (int j = 0; j < 32; ++j) c[j] = 0.f;
        return;
    }
    const float *src = a.C + row * a.ldc + c0;
    if (c0 + 32 <= a.N) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float v[8];
            ld_global_cg_v8(src + q * 8, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) c[q * 8 + j] = v[j];
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) c[j] = c0 + j < a.N ? src[j] : 0.f;
    }
}

// Direct epilogue: bias, activation and the store of one lane's 32 values
// o[j] = D(row, c0 + j), from registers straight to D (32-byte stores when
// the 32 columns are inside the matrix, guarded scalar stores at its edge).
__device__ __forceinline__ void store_row_direct(float (&o)[32], const TcArgs &a, int64_t row,
                                                 int64_t c0) {
    if (a.bias != nullptr) {
        if (a.bias_per_row) {
            const float bv = row < a.M ? a.bias[row] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] += bv;
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] += c0 + j < a.N ? a.bias[c0 + j] : 0.f;
        }
    }
    if (a.act != kActNone) {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = apply_activation(o[j], a.act);
    }
    if (row >= a.M) return;
    const bool whole = c0 + 32 <= a.N;
    if (a.d_bf16) {
        uint16_t *d = reinterpret_cast<uint16_t *>(a.D) + row * a.ldd + c0;
        if (whole) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
                st_global_v8(d + q * 16, pack_bf16x2(o[q * 16 + 0], o[q * 16 + 1]),
                             pack_bf16x2(o[q * 16 + 2], o[q * 16 + 3]),
                             pack_bf16x2(o[q * 16 + 4], o[q * 16 + 5]),
                             pack_bf16x2(o[q * 16 + 6], o[q * 16 + 7]),
                             pack_bf16x2(o[q * 16 + 8], o[q * 16 + 9]),
                             pack_bf16x2(o[q * 16 + 10], o[q * 16 + 11]),
                             pack_bf16x2(o[q * 16 + 12], o[q * 16 + 13]),
                             pack_bf16x2(o[q * 16 + 14], o[q * 16 + 15]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < a.N) d[j] = to_bf16_bits(o[j]);
        }
    } else {
        float *d = a.D + row * a.ldd + c0;
        if (whole) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                st_global_v8(d + q * 8, __float_as_uint(o[q * 8 + 0]),
                             __float_as_uint(o[q * 8 + 1]), __float_as_uint(o[q * 8 + 2]),
                             __float_as_uint(o[q * 8 + 3]), __float_as_uint(o[q * 8 + 4]),
                             __float_as_uint(o[q * 8 + 5]), __float_as_uint(o[q * 8 + 6]),
                             __float_as_uint(o[q * 8 + 7]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < a.N) d[j] = o[j];
        }
    }
}

// Staged epilogue: bias, activation, the 32 values of this lane's row into
// the box (FP32 swizzled, or BF16 rows of 64 bytes), then the box to D (one
// TMA store, or coalesced row stores when D cannot be described to TMA).
__device__ __forceinline__ void emit_box_chunk(float (&o)[32], uint8_t *box, int64_t r0,
                                               int64_t c0, int lane, const TcArgs &args,
                                               const CUtensorMap *map_d) {
    if (args.bias != nullptr) {
        if (args.bias_per_row) {
            const int64_t r = r0 + lane;
            const float bv = r < args.M ? args.bias[r] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] += bv;
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] += c0 + j < args.N ? args.bias[c0 + j] : 0.f;
        }
    }
    if (args.act != kActNone) {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = apply_activation(o[j], args.act);
    }
    if (args.d_bf16) {
        // BF16 box: 32 rows of 64 bytes, unswizzled
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8)
            *reinterpret_cast<uint4 *>(box + lane * 64 + q8 * 16) =
                make_uint4(pack_bf16x2(o[q8 * 8 + 0], o[q8 * 8 + 1]),
                           pack_bf16x2(o[q8 * 8 + 2], o[q8 * 8 + 3]),
                           pack_bf16x2(o[q8 * 8 + 4], o[q8 * 8 + 5]),
                           pack_bf16x2(o[q8 * 8 + 6], o[q8 * 8 + 7]));
    } else {
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4)
            *reinterpret_cast<float4 *>(box + box_offset(lane, j4 * 4)) =
                make_float4(o[j4 * 4 + 0], o[j4 * 4 + 1], o[j4 * 4 + 2], o[j4 * 4 + 3]);
    }
    if (args.tma_d) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0)
            tma_store_2d(map_d, static_cast<int32_t>(c0), static_cast<int32_t>(r0),
                         smem_addr(box));
    } else {
        __syncwarp();
        if (args.d_bf16)
            box_store_rows_bf16(box, args, r0, c0, lane);
        else
            box_store_rows(box, args, r0, c0, lane);
        __syncwarp();
    }
}

// ------------------------------------------------------------------- kernel
template <int CG, bool DIRECT = false>
__global__ void __launch_bounds__(Cfg<CG, DIRECT>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_b_half,
                        const __grid_constant__ CUtensorMap map_c,
                        const __grid_constant__ CUtensorMap map_d, const TcArgs args) {
    using C = Cfg<CG, DIRECT>;
    extern __shared__ uint8_t smem_raw[];
    // the ring must be 1024-byte aligned for the 128-byte swizzle atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint8_t *staging = smem + C::STAGES * C::STAGE_BYTES;  // 1024-aligned epilogue boxes
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + C::STAGING_BYTES);
    uint64_t *full = bars;                       // [MAX_STAGES]  TMA -> MMA (leader counts both CTAs)
    uint64_t *empty = bars + C::MAX_STAGES;      // [MAX_STAGES]  MMA -> TMA
    uint64_t *tfull = bars + 2 * C::MAX_STAGES;  // [2]           MMA -> epilogue
    uint64_t *tempty = tfull + ACC_BUFS;     // [2]       epilogue -> MMA (leader counts both)
    uint64_t *drain = tempty + ACC_BUFS;     // [1]       MMA teardown
    uint64_t *cbar = drain + 1;              // [16]      C box loaded (epilogue warp x box)
    uint64_t *pbar = cbar + 16;              // [8]       split-K pieces loaded (epilogue warp)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(pbar + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = CG == 1 ? 0u : cluster_rank();  // position in the CTA pair
    const bool leader = rank == 0;
    const int64_t group_id = blockIdx.x / CG;  // tile-group (pair) index
    const int64_t num_groups = gridDim.x / CG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::MAX_STAGES; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(smem_addr(&tfull[b]), 1);
            // one arrival per epilogue warp of the group
            mbar_init(smem_addr(&tempty[b]), C::EPI_WARPS * CG);
        }
        mbar_init(smem_addr(drain), 1);
        for (int i = 0; i < 16; ++i) mbar_init(smem_addr(&cbar[i]), 1);
        for (int i = 0; i < 8; ++i) mbar_init(smem_addr(&pbar[i]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b))
                     : "memory");
        if (args.tail_split_n && args.b_kmajor)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b_half))
                         : "memory");
        if (args.tma_c)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_c))
                         : "memory");
        if (args.tma_d)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_d))
                         : "memory");
    }
    if (warp == 1) tmem_alloc<CG>(smem_addr(tmem_slot));
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();  // peer barriers initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // on-chip set-up done: wait for the previous kernel on the stream before
    // any global memory access, and let the next launch be scheduled
    pdl_wait();
    pdl_launch_dependents();

    const int64_t n_items = work_items<CG>(args);
    const uint32_t ring_base = smem_addr(ring);
    // ring stages (compile-time for CTA pairs)
    const int stages = CG == 1 ? args.stages1 : C::RING_STAGES;
    const uint32_t stage_bytes = CG == 1 ? args.stage_bytes1 : C::STAGE_BYTES;
    const uint32_t a_region = CG == 1 ? args.a_region1 : C::A_BYTES;  // B starts here in a stage
    bool aborted = false;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            int64_t li = 0;
            for (int64_t w = group_id; w < n_items && ok; w += num_groups, ++li) {
                const WorkItem it = work_item<CG>(w, args);
                int64_t tm, tn;
                tile_coords(it.t, args, tm, tn);
                const int32_t m0 = static_cast<int32_t>(tm * C::TILE_M + rank * BM);
                const int b_rows = it.n_width / CG;  // columns of B this CTA loads
                const int32_t n0 = static_cast<int32_t>(tn * BN + it.n_off + rank * b_rows);
                const int a_rows = CG == 1 ? args.am1 : BM;  // rows of A this stage loads
                const int b_load = (CG == 1 && args.b_kmajor) ? args.bk1 : b_rows;  // and of B
                const uint32_t stage_tx = CG * (a_rows * BK * 2 + b_load * BK * 2);
                // Serpentine K order: every other work item walks its K blocks
                // backwards, so the blocks a round of tiles reads last are the
                // ones the next round (the same tile rows, under the grouped
                // raster) reads first, while they are still in L2.  The MMA
                // side takes the stages as they come (the sum's order changes,
                // not its terms).
                const bool reverse = (li & 1) != 0;
                // Single-CTA tiles with M <= 64 share A's K blocks, a few
                // lines each: each tile starts its K range at a different
                // block, so the CTAs do not all read the same lines at once.
                const int64_t nkb = it.kb_end - it.kb_begin;
                const int64_t rot = (CG == 1 && args.am1 < BM && nkb > 1) ? it.t % nkb : 0;
                for (int64_t i = 0; i < nkb; ++i) {
                    int64_t j = (reverse ? nkb - 1 - i : i) + rot;
                    if (j >= nkb) j -= nkb;
                    const int64_t kb = it.kb_begin + j;
                    if (!wait_bounded(smem_addr(&empty[stage]), phase ^ 1, abort_flag,
                                      args.timeout_ns)) {
                        raise_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_addr(&full[stage]);
                    // the leader's full barrier counts both CTAs' bytes
                    const uint32_t fb = CG == 1 ? fb_local : map_to_rank(fb_local, 0);
                    const uint32_t sa = ring_base + stage * stage_bytes;
                    const uint32_t sb = sa + a_region;
                    const int32_t k0 = static_cast<int32_t>(kb * BK);
                    if (leader) mbar_arrive_expect_tx(fb_local, stage_tx);
                    if (args.a_kmajor) {
                        tma_load_2d<CG>(sa, &map_a, k0, m0, fb);
                    } else {
                        for (int i = 0; i < a_rows / 64; ++i)
                            tma_load_2d<CG>(sa + i * 64 * 128, &map_a, m0 + 64 * i, k0, fb);
                    }
                    if (args.b_kmajor) {
                        // (single CTAs: map_b's box is bn1 rows, the item's width)
                        tma_load_2d<CG>(sb, (CG == 1 || b_rows == C::B_ROWS) ? &map_b : &map_b_half,
                                        k0, n0, fb);
                    } else {
                        for (int i = 0; i < b_rows / 64; ++i)
                            tma_load_2d<CG>(sb + i * 64 * 128, &map_b, n0 + 64 * i, k0, fb);
                    }
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // Let the copies still in flight land before the CTA can exit:
            // wait on the full barrier of each of the last issued stages.
            // CG = 2: the leader's full barriers also count the peer's bytes,
            // so the leader's drain covers both CTAs' copies.
            if (leader) {
                const int64_t outstanding = issued < stages ? issued : stages;
                int s = stage;
                uint32_t ph = phase;
                for (int64_t i = 0; i < outstanding; ++i) {
                    if (--s < 0) {
                        s = stages - 1;
                        ph ^= 1;
                    }
                    const volatile int never = 0;  // issued copies complete regardless of aborts
                    if (!wait_bounded(smem_addr(&full[s]), ph, &never, args.timeout_ns))
                        raise_abort(abort_flag);
                }
            }
            aborted = !ok;
        }
        __syncwarp();
        if (CG == 1 && args.cluster_k) {
            cluster_sync();  // the epilogue warps' (A): operand rings idle
            cluster_sync();  // their (C): pieces delivered
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {
            const uint32_t idesc_full =
                make_idesc(C::TILE_M, BN, !args.a_kmajor, !args.b_kmajor, args.ab_format);
            const uint32_t idesc_half =
                make_idesc(C::TILE_M, BN / 2, !args.a_kmajor, !args.b_kmajor, args.ab_format);
            const uint32_t idesc_n1 =  // single CTAs: N = bn1
                make_idesc(C::TILE_M, CG == 1 ? args.bn1 : BN, !args.a_kmajor, !args.b_kmajor,
                           args.ab_format);
            int stage = 0;
            uint32_t phase = 0;
            int64_t li = 0;
            bool ok = true;
            // The tensor pipe idles while this thread runs anything between
            // two stages' MMAs, so the loop keeps that short: barrier
            // addresses and stage-0 descriptors are fixed here (stage s adds
            // s x the stage size, K slice kk adds kk x the step, in 16-byte
            // units), and it waits for two stages at a time, then issues
            // their 8 MMAs back to back.
            const uint32_t full0 = smem_addr(&full[0]), empty0 = smem_addr(&empty[0]);
            const uint64_t a_desc0 = args.a_kmajor ? desc_kmajor(ring_base, 0) : desc_mnmajor(ring_base, 0);
            const uint64_t b_desc0 = args.b_kmajor ? desc_kmajor(ring_base + a_region, 0)
                                                   : desc_mnmajor(ring_base + a_region, 0);
            const uint64_t a_step = args.a_kmajor ? (UMMA_K * 2) >> 4 : (UMMA_K * 128) >> 4;
            const uint64_t b_step = args.b_kmajor ? (UMMA_K * 2) >> 4 : (UMMA_K * 128) >> 4;
            for (int64_t w = group_id; w < n_items && ok; w += num_groups, ++li) {
                const WorkItem it = work_item<CG>(w, args);
                const int64_t kb_begin = it.kb_begin;
                const int64_t kb_end = it.kb_end;
                const int buf = static_cast<int>(li & 1);
                const uint32_t acc_phase = static_cast<uint32_t>((li >> 1) & 1);
                const uint32_t idesc =
                    CG == 1 ? idesc_n1 : (it.n_width == BN ? idesc_full : idesc_half);
                if (!wait_bounded(smem_addr(&tempty[buf]), acc_phase ^ 1, abort_flag,
                                  args.timeout_ns)) {
                    raise_abort(abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                static_assert(BK / UMMA_K == 4, "four MMAs per stage below");
                const int nkb = static_cast<int>(kb_end - kb_begin);
                for (int i = 0; i < nkb; i += 2) {
                    const bool two = i + 1 < nkb;
                    const int s0 = stage;
                    const uint32_t p0 = phase;
                    const int s1 = s0 + 1 == stages ? 0 : s0 + 1;
                    const uint32_t p1 = s1 == 0 ? p0 ^ 1u : p0;
                    const uint32_t fb0 = full0 + 8u * static_cast<uint32_t>(s0);
                    const uint32_t fb1 = full0 + 8u * static_cast<uint32_t>(s1);
                    if (!mbar_try_wait(fb0, p0) && !wait_bounded(fb0, p0, abort_flag, args.timeout_ns)) {
                        raise_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    if (two && !mbar_try_wait(fb1, p1) &&
                        !wait_bounded(fb1, p1, abort_flag, args.timeout_ns)) {
                        raise_abort(abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint64_t ad = a_desc0 + static_cast<uint64_t>(s0) * (stage_bytes >> 4);
                    uint64_t bd = b_desc0 + static_cast<uint64_t>(s0) * (stage_bytes >> 4);
                    tc_mma<CG>(d_tmem, ad, bd, idesc, i > 0 ? 1u : 0u);
                    tc_mma<CG>(d_tmem, ad + a_step, bd + b_step, idesc, 1u);
                    tc_mma<CG>(d_tmem, ad + 2 * a_step, bd + 2 * b_step, idesc, 1u);
                    tc_mma<CG>(d_tmem, ad + 3 * a_step, bd + 3 * b_step, idesc, 1u);
                    if (two) {
                        ad = a_desc0 + static_cast<uint64_t>(s1) * (stage_bytes >> 4);
                        bd = b_desc0 + static_cast<uint64_t>(s1) * (stage_bytes >> 4);
                        tc_mma<CG>(d_tmem, ad, bd, idesc, 1u);
                        tc_mma<CG>(d_tmem, ad + a_step, bd + b_step, idesc, 1u);
                        tc_mma<CG>(d_tmem, ad + 2 * a_step, bd + 2 * b_step, idesc, 1u);
                        tc_mma<CG>(d_tmem, ad + 3 * a_step, bd + 3 * b_step, idesc, 1u);
                    }
                    tc_commit<CG>(empty0 + 8u * static_cast<uint32_t>(s0));  // frees the stages (both CTAs)
                    if (two) tc_commit<CG>(empty0 + 8u * static_cast<uint32_t>(s1));
                    if (two) {
                        stage = s1 + 1 == stages ? 0 : s1 + 1;
                        phase = stage == 0 ? p1 ^ 1u : p1;
                    } else {
                        stage = s1;
                        phase = p1;
                    }
                }
                if (!ok) break;
                tc_commit<CG>(smem_addr(&tfull[buf]));  // accumulator ready for the epilogue(s)
            }
            // all MMAs issued here have finished once `drain` completes
            tc_commit_local<CG>(smem_addr(drain));
            const volatile int never = 0;
            if (!wait_bounded(smem_addr(drain), 0, &never, args.timeout_ns))
                raise_abort(abort_flag);
            aborted = !ok;
        }
        __syncwarp();
        if (CG == 1 && args.cluster_k) {
            cluster_sync();  // the epilogue warps' (A) and (C)
            cluster_sync();
        }
    } else if constexpr (DIRECT) {
        // ------------------------------------------ epilogue warps 2-5, direct
        // Per tile, the warp drains its 32 accumulator rows (TMEM lanes) in
        // 32-column chunks: tcgen05.ld -> alpha * acc + beta * C (bias,
        // activation) in registers -> each lane stores its row's 32 values
        // to D with 32-byte stores; each lane loads its row's C with 32-byte
        // loads, one chunk ahead.  A split tile's pieces
        // publish their raw sums the same way (one 32 x 32 block of rows per
        // warp and chunk) and the last piece adds them, in K order, straight
        // from global memory.
        const int quarter = warp % 4;  // TMEM lanes this warp may access
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const bool use_c = args.beta != 0.f;
        int64_t li = 0;
        for (int64_t w = group_id; w < n_items; w += num_groups, ++li) {
            const WorkItem it = work_item<CG>(w, args);
            const int64_t t = it.t;
            const int buf = static_cast<int>(li & 1);
            const uint32_t acc_phase = static_cast<uint32_t>((li >> 1) & 1);
            // lane 0 waits, the warp follows its verdict (keeps the warp converged)
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_addr(&tfull[buf]), acc_phase, abort_flag, args.timeout_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_abort(abort_flag);
                aborted = true;
                break;
            }
            tc_fence_after();
            int64_t tm, tn;
            tile_coords(t, args, tm, tn);
            const int64_t row0 = tm * C::TILE_M + rank * BM + quarter * 32;  // warp's first row
            const int64_t row = row0 + lane;                                 // this lane's row
            const int64_t col0 = tn * BN + it.n_off;
            int n_chunks = 0;  // chunks holding part of D (warp-uniform)
            if (row0 < args.M) {
                const int64_t rest = args.N - col0;
                n_chunks = rest >= it.n_width ? it.n_width / 32
                                              : static_cast<int>(rest > 0 ? (rest + 31) / 32 : 0);
            }
            const uint32_t t_acc = tmem_base + lane_off + static_cast<uint32_t>(buf * BN);
            auto release_acc = [&]() {
                // accumulator rows read: hand the buffer back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_addr(&tempty[buf]), 0));
            };
            if (it.nsp > 1 && n_chunks > 0) {
                // ---- a split tail tile: publish this piece's raw sums, count
                // the piece; the last piece to be counted adds all pieces in
                // K order and writes D (no piece waits for another)
                auto piece_row = [&](int piece, int chunk) -> float * {
                    const int64_t slot = ((t - args.tail_first) * it.nsp + piece) * 2 + rank;
                    return args.ws + ((slot * 4 + quarter) * 8 + chunk) * 1024 + lane * 32;
                };
                int *const counter = args.ws_count + ((t - args.tail_first) * 2 + rank) * 4 + quarter;
#pragma unroll 1
                for (int chunk = 0; chunk < n_chunks; ++chunk) {
                    uint32_t v[32];
                    __syncwarp();  // tcgen05.ld is warp-collective: converge first
                    tmem_load_32cols(t_acc + chunk * 32, v);
                    float *dst = piece_row(it.sp, chunk);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_global_v8(dst + q * 8, v[q * 8 + 0], v[q * 8 + 1], v[q * 8 + 2],
                                     v[q * 8 + 3], v[q * 8 + 4], v[q * 8 + 5], v[q * 8 + 6],
                                     v[q * 8 + 7]);
                }
                release_acc();
                __threadfence();  // each lane's sums are visible device-wide before the count
                __syncwarp();
                int reduce = 0;
                if (lane == 0) {
                    const int before = atomicAdd(counter, 1);
                    reduce = before == it.nsp - 1;
                    if (reduce) *counter = 0;  // all pieces counted: ready for the next call
                }
                __syncwarp();
                reduce = __shfl_sync(0xffffffffu, reduce, 0);
                if (!reduce) continue;
                __threadfence();  // the other pieces' sums (read through L2) after the count
#pragma unroll 1
                for (int chunk = 0; chunk < n_chunks; ++chunk) {
                    float o[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0.f;
                    for (int s2 = 0; s2 < it.nsp; ++s2) {  // K order
                        const float *src = piece_row(s2, chunk);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float pv[8];
                            ld_global_cg_v8(src + q * 8, pv);
#pragma unroll
                            for (int j = 0; j < 8; ++j) o[q * 8 + j] += pv[j];
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= args.alpha;
                    if (use_c) {
                        float c[32];
                        load_c_row_direct(args, row, col0 + chunk * 32, c);
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = fmaf(args.beta, c[j], o[j]);
                    }
                    store_row_direct(o, args, row, col0 + chunk * 32);
                }
                continue;
            }
            float c_next[32];  // C of the next chunk, loaded one chunk ahead
            if (use_c && n_chunks > 0) load_c_row_direct(args, row, col0, c_next);
#pragma unroll 1
            for (int chunk = 0; chunk < n_chunks; ++chunk) {
                float c[32];
                if (use_c) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) c[j] = c_next[j];
                    if (chunk + 1 < n_chunks)
                        load_c_row_direct(args, row, col0 + (chunk + 1) * 32, c_next);
                }
                uint32_t v[32];
                __syncwarp();  // tcgen05.ld is warp-collective: converge first
                tmem_load_32cols(t_acc + chunk * 32, v);
                if (chunk == n_chunks - 1) release_acc();
                float o[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = args.alpha * __uint_as_float(v[j]);
                if (use_c) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = fmaf(args.beta, c[j], o[j]);
                }
                store_row_direct(o, args, row, col0 + chunk * 32);
            }
            if (n_chunks == 0) release_acc();
        }
        __syncwarp();
    } else if constexpr (C::EPI_WARPS == 8) {
        // -------------------------------------- epilogue warps 2-9, staged, wide
        // Two warps per TMEM lane quarter (warp % 4), two boxes each: warp
        // e = warp - 2 drains the chunks of parity e / 4 of its quarter's 32
        // accumulator rows, so two chunks of a quarter are in flight at once.
        // Per chunk: C into a box (TMA, or coalesced row loads), started
        // while the previous chunk is processed -> tcgen05.ld -> D = alpha *
        // acc + beta * C in registers -> the box -> one TMA store (or
        // coalesced row stores when D's pitch cannot be described to TMA).
        const int e = warp - 2;
        const int quarter = warp % 4;  // TMEM lanes this warp may access
        const int half = e / 4;        // this warp's chunks: half, half + 2, ...
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const bool use_c = args.beta != 0.f;
        const bool tma_c = use_c && args.tma_c;
        uint8_t *const boxes = staging + e * 2 * 4096;  // this warp's two boxes
        uint8_t *box = boxes;                            // the box in use
        const uint32_t cb0 = smem_addr(&cbar[e * 2]);
        const uint32_t pb = smem_addr(&pbar[e]);
        uint32_t cphase = 0;  // bit b: parity of box b's next C arrival
        uint32_t pphase = 0;  // parity of the next split-K piece batch
        bool stop = false;
        auto emit_chunk = [&](float (&o)[32], int64_t r0, int64_t c0) {
            emit_box_chunk(o, box, r0, c0, lane, args, &map_d);
        };
        // at most the `pending` most recent TMA stores of D (one per chunk,
        // issued in chunk order) may still be reading their boxes
        auto box_free = [&](int pending) {
            if (lane == 0) {
                if (pending) bulk_wait_read<1>();
                else bulk_wait_read<0>();
            }
            __syncwarp();
        };
        auto load_c = [&](int b, int64_t c0, int64_t r0) {  // box b is free
            if (tma_c) {
                if (lane == 0) {
                    const uint32_t cb = cb0 + 8 * b;
                    mbar_arrive_expect_tx(cb, 32 * 32 * 4);
                    tma_load_2d<CG>(smem_addr(boxes + b * 4096), &map_c, static_cast<int32_t>(c0),
                                    static_cast<int32_t>(r0), map_to_rank(cb, rank));
                }
            } else {
                box_load_rows_async(boxes + b * 4096, args, r0, c0, lane);
            }
        };
        // C of box b has landed (`later`: one more load was started after it)
        auto wait_c = [&](int b, bool later) -> bool {
            if (tma_c) {
                int landed = 1;
                if (lane == 0)
                    landed = wait_bounded(cb0 + 8 * b, (cphase >> b) & 1u, abort_flag,
                                          args.timeout_ns);
                landed = __shfl_sync(0xffffffffu, landed, 0);
                cphase ^= 1u << b;
                return landed != 0;
            }
            if (later) async_copy_wait<1>();
            else async_copy_wait<0>();
            __syncwarp();
            return true;
        };
        auto add_c = [&](float (&o)[32]) {
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const float4 c = *reinterpret_cast<const float4 *>(box + box_offset(lane, j4 * 4));
                o[j4 * 4 + 0] = fmaf(args.beta, c.x, o[j4 * 4 + 0]);
                o[j4 * 4 + 1] = fmaf(args.beta, c.y, o[j4 * 4 + 1]);
                o[j4 * 4 + 2] = fmaf(args.beta, c.z, o[j4 * 4 + 2]);
                o[j4 * 4 + 3] = fmaf(args.beta, c.w, o[j4 * 4 + 3]);
            }
            __syncwarp();  // every lane has read its C before the box is overwritten
        };
        int64_t li = 0;
        for (int64_t w = group_id; w < n_items && !stop; w += num_groups, ++li) {
            const WorkItem it = work_item<CG>(w, args);
            const int64_t t = it.t;
            const int sp = it.sp;
            const int buf = static_cast<int>(li & 1);
            const uint32_t acc_phase = static_cast<uint32_t>((li >> 1) & 1);
            // lane 0 waits, the warp follows its verdict (keeps the warp converged)
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_addr(&tfull[buf]), acc_phase, abort_flag, args.timeout_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_abort(abort_flag);
                aborted = true;
                break;
            }
            tc_fence_after();
            int64_t tm, tn;
            tile_coords(t, args, tm, tn);
            const int64_t row0 = tm * C::TILE_M + rank * BM + quarter * 32;  // warp's first row
            const int64_t col0 = tn * BN + it.n_off;
            int n_chunks = 0;  // chunks holding part of D (warp-uniform)
            if (row0 < args.M) {
                const int64_t rest = args.N - col0;
                n_chunks = rest >= it.n_width ? it.n_width / 32
                                              : static_cast<int>(rest > 0 ? (rest + 31) / 32 : 0);
            }
            // this warp's last chunk (-1: it has none)
            const int my_last = n_chunks > half ? half + ((n_chunks - 1 - half) / 2) * 2 : -1;
            const uint32_t t_acc = tmem_base + lane_off + static_cast<uint32_t>(buf * BN);
            auto release_acc = [&]() {
                // accumulator rows read: hand the buffer back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_addr(&tempty[buf]), 0));
            };
            if (it.nsp > 1 && n_chunks > 0) {
                // ---- a split tail tile: publish this warp's chunks of the
                // piece's raw sums, count the piece per warp; the last piece
                // to be counted adds the pieces in K order and writes D (no
                // piece waits for another)
                auto piece_box = [&](int piece, int chunk) -> float * {
                    const int64_t slot = ((t - args.tail_first) * it.nsp + piece) * 2 + rank;
                    return args.ws + ((slot * 4 + quarter) * 8 + chunk) * 1024;
                };
                int *const counter = args.ws_count + ((t - args.tail_first) * 2 + rank) * 8 + e;
#pragma unroll 1
                for (int chunk = half; chunk < n_chunks; chunk += 2) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_load_32cols(t_acc + chunk * 32, v);
                    box_free(0);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4)
                        *reinterpret_cast<uint4 *>(box + box_offset(lane, j4 * 4)) =
                            make_uint4(v[j4 * 4 + 0], v[j4 * 4 + 1], v[j4 * 4 + 2], v[j4 * 4 + 3]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) bulk_copy_to_global(piece_box(sp, chunk), smem_addr(box), 4096);
                }
                release_acc();
                if (my_last < 0) continue;  // no piece of this tile has chunks for this warp
                int reduce = 0;
                if (lane == 0) {
                    bulk_wait_all();  // the partial sums are in global memory
                    __threadfence();
                    const int before = atomicAdd(counter, 1);
                    reduce = before == it.nsp - 1;
                    if (reduce) {
                        *counter = 0;  // all pieces counted: ready for the next call
                        __threadfence();
                    }
                }
                reduce = __shfl_sync(0xffffffffu, reduce, 0);
                if (!reduce) continue;
                // the operand ring is idle: a split piece is its CTA's last work item
                uint8_t *pieces = ring + e * (C::STAGES * C::STAGE_BYTES / 8);
#pragma unroll 1
                for (int chunk = half; chunk < n_chunks && !stop; chunk += 2) {
                    const int64_t c0 = col0 + chunk * 32;
                    box_free(0);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(pb, static_cast<uint32_t>(it.nsp) * 4096);
                        for (int s2 = 0; s2 < it.nsp; ++s2)
                            bulk_copy_to_shared(smem_addr(pieces + s2 * 4096), piece_box(s2, chunk),
                                                4096, pb);
                    }
                    if (use_c) load_c(0, c0, row0);
                    int got = 1;
                    if (lane == 0) got = wait_bounded(pb, pphase, abort_flag, args.timeout_ns);
                    got = __shfl_sync(0xffffffffu, got, 0);
                    pphase ^= 1u;
                    if (!got) {
                        if (lane == 0) raise_abort(abort_flag);
                        aborted = stop = true;
                        break;
                    }
                    // sum of the K pieces in K order (the same order on every run)
                    float o[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0.f;
                    for (int s2 = 0; s2 < it.nsp; ++s2) {
                        const uint8_t *part = pieces + s2 * 4096;
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 pv =
                                *reinterpret_cast<const float4 *>(part + box_offset(lane, j4 * 4));
                            o[j4 * 4 + 0] += pv.x;
                            o[j4 * 4 + 1] += pv.y;
                            o[j4 * 4 + 2] += pv.z;
                            o[j4 * 4 + 3] += pv.w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= args.alpha;
                    if (use_c) {
                        if (!wait_c(0, false)) {
                            if (lane == 0) raise_abort(abort_flag);
                            aborted = stop = true;
                            break;
                        }
                        add_c(o);
                    }
                    __syncwarp();  // every lane has read the pieces
                    emit_chunk(o, row0, c0);
                }
                continue;
            }
            // chunk k of this warp (chunk half + 2k) uses box k & 1; C of the
            // next chunk is started before this one is processed
            if (my_last >= 0) {
                box_free(0);  // every store of the previous tile has read its box
                if (use_c) load_c(0, col0 + half * 32, row0);
            }
#pragma unroll 1
            for (int chunk = half, k = 0; chunk < n_chunks; chunk += 2, ++k) {
                const int64_t c0 = col0 + chunk * 32;
                const int b = k & 1;
                box = boxes + b * 4096;
                const bool next = chunk + 2 < n_chunks;
                if (use_c && next) {
                    box_free(0);  // the store of chunk k - 1 has read box b ^ 1
                    load_c(b ^ 1, c0 + 64, row0);
                } else if (!use_c && k >= 2) {
                    box_free(1);  // the store of chunk k - 2 has read box b
                }
                uint32_t v[32];
                __syncwarp();  // tcgen05.ld is warp-collective: converge first
                tmem_load_32cols(t_acc + chunk * 32, v);
                if (chunk == my_last) release_acc();
                float o[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = args.alpha * __uint_as_float(v[j]);
                if (use_c) {
                    if (!wait_c(b, next)) {
                        if (lane == 0) raise_abort(abort_flag);
                        aborted = stop = true;
                        break;
                    }
                    add_c(o);
                }
                emit_chunk(o, row0, c0);
            }
            box = boxes;
            if (my_last < 0) release_acc();
        }
        if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
        __syncwarp();
    } else {
        // ------------------------------------------------- epilogue warps 2-5
        // Per tile, the warp drains its 32 accumulator rows (TMEM lanes) in
        // 32-column chunks: tcgen05.ld -> D = alpha * acc + beta * C in
        // registers -> a swizzled 32 x 32 box in shared memory -> one TMA
        // store (or, when D's pitch cannot be described to TMA, coalesced
        // row stores).  C arrives in the same box, by TMA one chunk ahead
        // (or by coalesced row loads), and each thread reads its row from it.
        const int quarter = warp % 4;  // TMEM lanes this warp may access
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const bool use_c = args.beta != 0.f;
        const bool tma_c = use_c && args.tma_c;
        uint8_t *boxes = staging + quarter * 2 * 4096;  // this warp's two boxes
        const uint32_t cbar0 = smem_addr(&cbar[quarter * 2]);
        uint32_t nb = 0;      // boxes used so far (box nb & 1 is next)
        uint32_t cphase = 0;  // bit b: parity of box b's next C arrival
        bool stop = false;
        int cluster_bars = 0;  // cluster barriers passed (split pieces pass two)
        auto issue_c = [&](int b, int64_t c0, int64_t r0) {
            // lane 0 only; box b is free (no store still reading it)
            const uint32_t bar = cbar0 + 8 * b;
            mbar_arrive_expect_tx(bar, 32 * 32 * 4);
            tma_load_2d<CG>(smem_addr(boxes + b * 4096), &map_c, static_cast<int32_t>(c0),
                            static_cast<int32_t>(r0), CG == 1 ? bar : map_to_rank(bar, rank));
        };
        // bias, activation, the box, then the box to D (TMA store or rows)
        auto emit_chunk = [&](float (&o)[32], uint8_t *box, int64_t r0, int64_t c0) {
            emit_box_chunk(o, box, r0, c0, lane, args, &map_d);
        };
        int64_t li = 0;
        for (int64_t w = group_id; w < n_items && !stop; w += num_groups, ++li) {
            const WorkItem it = work_item<CG>(w, args);
            const int64_t t = it.t;
            const int sp = it.sp;
            const int buf = static_cast<int>(li & 1);
            const uint32_t acc_phase = static_cast<uint32_t>((li >> 1) & 1);
            // lane 0 waits, the warp follows its verdict (keeps the warp converged)
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(smem_addr(&tfull[buf]), acc_phase, abort_flag, args.timeout_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_abort(abort_flag);
                aborted = true;
                break;
            }
            tc_fence_after();
            int64_t tm, tn;
            tile_coords(t, args, tm, tn);
            const int64_t row0 = tm * C::TILE_M + rank * BM + quarter * 32;  // warp's first row
            const int64_t col0 = tn * BN + it.n_off;
            int n_chunks = 0;  // chunks holding part of D (warp-uniform)
            if (row0 < args.M) {
                const int64_t rest = args.N - col0;
                n_chunks = rest >= it.n_width ? it.n_width / 32
                                              : static_cast<int>(rest > 0 ? (rest + 31) / 32 : 0);
            }
            const uint32_t t_acc = tmem_base + lane_off + static_cast<uint32_t>(buf * BN);
            auto release_acc = [&]() {
                // accumulator rows read: hand the buffer back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t te = smem_addr(&tempty[buf]);
                    if (CG == 1)
                        mbar_arrive(te);
                    else
                        mbar_arrive_cluster(map_to_rank(te, 0));
                }
            };
            if (it.nsp > 1) {
                // ---- a split tile (single CTAs): the ks pieces of the tile
                // are the CTAs of one thread-block cluster, piece = cluster
                // rank = K range.  Chunk c (32 columns) belongs to rank c % ks.
                // A) cluster barrier: every piece's MMAs are done, so every
                //    CTA's operand ring is idle (a piece is its CTA's only
                //    work item);
                // B) each piece stores the chunks it does not own, from TMEM,
                //    into their owner's ring, one slot per (owned chunk,
                //    sender) (plain remote stores: nothing waits on them one
                //    by one);
                // C) cluster barrier: every slot is written and visible, and
                //    no CTA touches another's shared memory after it;
                // D) the owner adds the ks pieces in rank (K) order -- its own
                //    straight from TMEM -- so the sum does not depend on
                //    timing, and runs the epilogue.
                const int ks = it.nsp;
                const int own_max = (BN / 32 + ks - 1) / ks;  // owned chunks per rank, at most
                auto slot = [&](int j, int s2) -> uint32_t {  // owned chunk j, sender s2
                    const int idx = s2 < sp ? s2 : s2 - 1;
                    return ring_base +
                           static_cast<uint32_t>(((quarter * own_max + j) * (ks - 1) + idx) * 4096);
                };
                cluster_sync();  // (A)
                ++cluster_bars;
                // rows past M are never stored to D: they are not sent (and
                // their slots are read but unused)
                const bool row_ok = row0 + lane < args.M;
#pragma unroll 1
                for (int chunk = 0; chunk < n_chunks; ++chunk) {
                    const int owner = chunk % ks;
                    if (owner == sp) continue;
                    uint32_t v[32];
                    __syncwarp();  // tcgen05.ld is warp-collective: converge first
                    tmem_load_32cols(t_acc + chunk * 32, v);
                    // the owner's slot for this chunk and this sender
                    const int idx = sp < owner ? sp : sp - 1;
                    const uint32_t dst_local = ring_base + static_cast<uint32_t>(
                        ((quarter * own_max + chunk / ks) * (ks - 1) + idx) * 4096);
                    const uint32_t dst = map_to_rank(dst_local, static_cast<uint32_t>(owner));
                    if (row_ok) {
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4)
                            st_cluster_v4(dst + slot_offset(lane, j4), v[j4 * 4 + 0],
                                          v[j4 * 4 + 1], v[j4 * 4 + 2], v[j4 * 4 + 3]);
                    }
                }
                cluster_sync();  // (C)
                ++cluster_bars;
#pragma unroll 1
                for (int chunk = sp; chunk < n_chunks && !stop; chunk += ks) {
                    const int b = nb & 1;
                    uint8_t *box = boxes + b * 4096;
                    const int64_t c0 = col0 + chunk * 32;
                    if (use_c) {
                        if (lane == 0) bulk_wait_read<0>();  // no store still reads this box
                        __syncwarp();
                        if (tma_c) {
                            if (lane == 0) issue_c(b, c0, row0);
                        } else {
                            box_load_rows_async(box, args, row0, c0, lane);
                        }
                    }
                    uint32_t v[32];
                    __syncwarp();
                    tmem_load_32cols(t_acc + chunk * 32, v);
                    // the ks pieces in rank order (the same order on every run)
                    float o[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0.f;
                    for (int s2 = 0; s2 < ks; ++s2) {
                        if (s2 == sp) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) o[j] += __uint_as_float(v[j]);
                            continue;
                        }
                        const uint8_t *src = ring + (slot(chunk / ks, s2) - ring_base);
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 pv =
                                *reinterpret_cast<const float4 *>(src + slot_offset(lane, j4));
                            o[j4 * 4 + 0] += pv.x;
                            o[j4 * 4 + 1] += pv.y;
                            o[j4 * 4 + 2] += pv.z;
                            o[j4 * 4 + 3] += pv.w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= args.alpha;
                    if (use_c) {
                        if (tma_c) {
                            int landed = 1;
                            if (lane == 0)
                                landed = wait_bounded(cbar0 + 8 * b, (cphase >> b) & 1u,
                                                      abort_flag, args.timeout_ns);
                            landed = __shfl_sync(0xffffffffu, landed, 0);
                            cphase ^= 1u << b;
                            if (!landed) {
                                if (lane == 0) raise_abort(abort_flag);
                                aborted = stop = true;
                                break;
                            }
                        } else {
                            async_copy_wait<0>();
                            __syncwarp();
                        }
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 c =
                                *reinterpret_cast<const float4 *>(box + box_offset(lane, j4 * 4));
                            o[j4 * 4 + 0] = fmaf(args.beta, c.x, o[j4 * 4 + 0]);
                            o[j4 * 4 + 1] = fmaf(args.beta, c.y, o[j4 * 4 + 1]);
                            o[j4 * 4 + 2] = fmaf(args.beta, c.z, o[j4 * 4 + 2]);
                            o[j4 * 4 + 3] = fmaf(args.beta, c.w, o[j4 * 4 + 3]);
                        }
                    } else {
                        if (lane == 0) bulk_wait_read<1>();  // the store that used this box has read it
                    }
                    __syncwarp();  // every lane has read C before the box is overwritten
                    emit_chunk(o, box, row0, c0);
                    ++nb;
                }
                release_acc();
                continue;
            }
            if (use_c && n_chunks > 0) {
                if (lane == 0) bulk_wait_read<0>();  // the box is not read by an earlier store
                __syncwarp();
                if (tma_c) {
                    if (lane == 0) issue_c(nb & 1, col0, row0);
                } else {
                    box_load_rows_async(boxes + (nb & 1) * 4096, args, row0, col0, lane);
                }
            }
#pragma unroll 1
            for (int chunk = 0; chunk < n_chunks; ++chunk) {
                const int b = nb & 1;
                uint8_t *box = boxes + b * 4096;
                const int64_t c0 = col0 + chunk * 32;
                const bool more = chunk + 1 < n_chunks;
                if (use_c && more) {
                    // C of the next chunk into the other box, one chunk ahead
                    if (lane == 0) bulk_wait_read<0>();  // the other box's store has read it
                    __syncwarp();
                    if (tma_c) {
                        if (lane == 0) issue_c(b ^ 1, c0 + 32, row0);
                    } else {
                        box_load_rows_async(boxes + (b ^ 1) * 4096, args, row0, c0 + 32, lane);
                    }
                }
                uint32_t v[32];
                __syncwarp();  // tcgen05.ld is warp-collective: converge first
                tmem_load_32cols(t_acc + chunk * 32, v);
                if (chunk == n_chunks - 1) release_acc();
                float o[32];
                {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = args.alpha * __uint_as_float(v[j]);
                }
                if (use_c) {
                    if (tma_c) {
                        int landed = 1;
                        if (lane == 0)
                            landed = wait_bounded(cbar0 + 8 * b, (cphase >> b) & 1u, abort_flag,
                                                  args.timeout_ns);
                        landed = __shfl_sync(0xffffffffu, landed, 0);
                        cphase ^= 1u << b;
                        if (!landed) {
                            if (lane == 0) raise_abort(abort_flag);
                            aborted = stop = true;
                            break;
                        }
                    } else {
                        // this chunk's copies done (the next chunk's may still run)
                        if (more)
                            async_copy_wait<1>();
                        else
                            async_copy_wait<0>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 c = *reinterpret_cast<const float4 *>(box + box_offset(lane, j4 * 4));
                        o[j4 * 4 + 0] = fmaf(args.beta, c.x, o[j4 * 4 + 0]);
                        o[j4 * 4 + 1] = fmaf(args.beta, c.y, o[j4 * 4 + 1]);
                        o[j4 * 4 + 2] = fmaf(args.beta, c.z, o[j4 * 4 + 2]);
                        o[j4 * 4 + 3] = fmaf(args.beta, c.w, o[j4 * 4 + 3]);
                    }
                    __syncwarp();  // every lane has its C before the box is overwritten
                } else {
                    if (lane == 0) bulk_wait_read<1>();  // the store that used this box has read it
                    __syncwarp();
                }
                emit_chunk(o, box, row0, c0);
                ++nb;
            }
            if (n_chunks == 0) release_acc();
        }
        // every thread of a split cluster passes both cluster barriers, on
        // every path (the other CTAs wait there)
        if (args.cluster_k)
            for (; cluster_bars < 2; ++cluster_bars) cluster_sync();
        if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
        __syncwarp();
    }

    if (aborted) {
        // give copies issued by a peer that gave up a short time to land
        const uint64_t t0 = global_timer();
        while (global_timer() - t0 < 2000000ull) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();  // the pair's MMAs and remote arrivals are done
    tc_fence_after();
    if (warp == 1) tmem_dealloc<CG>(tmem_base);
}

// ------------------------------------------------------- bounded-wait probe
// One thread waits, with the kernels' bounded wait, on an mbarrier that
// nothing arrives on; after timeout_ns it gives up and sets the device status
// word exactly as a GEMM whose wait ran out would.  Nothing else is in flight.
__global__ void wait_probe_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_addr(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const volatile int never = 0;
    if (!wait_bounded(smem_addr(&bar), 0, &never, timeout_ns)) atomicExch(&g_tc_status, 1);
}

// -------------------------------------------------------- tensor-pipe probe
// The tensor pipe with no memory traffic: each CTA (pair) writes one A tile
// (128 x 64) and one B tile (B_ROWS x 64) of BF16 values into shared memory
// once, then one lane issues n_mma back-to-back TILE_M x 256 x 16 MMAs into
// one TMEM accumulator, cycling over the tiles' four 16-deep slices (the
// MMA stream of the GEMM's mainloop with the loads taken away).
constexpr int PROBE_THREADS = 128;

template <int CG>
__global__ void __launch_bounds__(PROBE_THREADS, 1)
    tc_probe_kernel(int64_t n_mma, uint64_t timeout_ns) {
    using C = Cfg<CG>;
    constexpr int kTileBytes = (BM + C::B_ROWS) * BK * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *done = reinterpret_cast<uint64_t *>(smem + kTileBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    const int warp = threadIdx.x / 32;
    const uint32_t rank = CG == 1 ? 0u : cluster_rank();

    // operands: BF16 values +-[0.5, 1) with fractions and signs from a
    // multiplicative hash of the word index, so the multipliers see data
    // that changes from element to element
    uint32_t *words = reinterpret_cast<uint32_t *>(smem);
    for (int i = threadIdx.x; i < kTileBytes / 4; i += PROBE_THREADS) {
        const uint32_t h = (static_cast<uint32_t>(i) + 0x9E3779B9u * (blockIdx.x + 1u)) * 0x85EBCA6Bu;
        const uint32_t lo = 0x3F00u | ((h >> 9) & 0x7Fu) | (((h >> 16) & 1u) << 15);
        const uint32_t hi = 0x3F00u | ((h >> 17) & 0x7Fu) | (((h >> 24) & 1u) << 15);
        words[i] = lo | (hi << 16);
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(done), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // operands -> tensor pipe
    if (warp == 0) tmem_alloc<CG>(smem_addr(tmem_slot));
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();  // both CTAs' operands and barriers are ready
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (threadIdx.x == 0 && rank == 0) {
        const uint32_t idesc = make_idesc(C::TILE_M, BN, 0, 0, 1);
        const uint32_t sa = smem_addr(smem), sb = sa + BM * BK * 2;
        for (int64_t i = 0; i < n_mma; ++i) {
            const int kk = static_cast<int>(i & (BK / UMMA_K - 1));
            tc_mma<CG>(tmem_base, desc_kmajor(sa, kk), desc_kmajor(sb, kk), idesc,
                       i > 0 ? 1u : 0u);
        }
        tc_commit<CG>(smem_addr(done));  // CG = 2: arrives on both CTAs' `done`
    }
    if (threadIdx.x == 0) {
        const volatile int never = 0;
        if (!wait_bounded(smem_addr(done), 0, &never, timeout_ns)) atomicExch(&g_tc_status, 1);
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();
    tc_fence_after();
    if (warp == 0) tmem_dealloc<CG>(tmem_base);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 2-D 16-bit tensor map: inner dimension `inner` (contiguous), outer `outer`,
// row pitch ld elements, box = box_inner x box_outer, 128-byte swizzle,
// out-of-bounds elements read as zero.
bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, int64_t inner,
               int64_t outer, int64_t ld, uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D FP32 row-major M x N map with 32 x 32 boxes and the 128-byte swizzle
// (the epilogue's box layout).
bool encode_box32_f32(CUtensorMap *map, const void *base, int64_t M, int64_t N, int64_t ld) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;


struct DeviceInfo {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 1;
    int pairs = 0;         // CTA pairs that can be resident at once (0: pair variant not used)
    int pairs_direct = 0;  // the same for the direct-epilogue pair variant
    // clusters of k single CTAs that can be resident at once, k = 2..8
    // (-1: not asked yet); asked under `mu`
    int clusters[kMaxClusterK + 1] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
    std::mutex mu;
};
DeviceInfo g_dev[kMaxDevices];

bool aligned(const void *ptr, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) % bytes) == 0;
}

// A launch of `grid` CTAs in clusters of cg (cg = 1: no cluster), allowed to
// start early (programmatic dependent launch, see pdl_wait).  attr must hold
// two entries: [0] the dependent-launch attribute, [1] the cluster shape.
cudaLaunchConfig_t launch_config(int grid, int cg, int threads, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    set_pdl_attribute(&attr[cfg.numAttrs++]);
    if (cg > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(cg);
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    return cfg;
}

// Per device, once: opt in to the large shared-memory carve-out and find how
// many CTA pairs can be resident at once.
DeviceInfo *device_info(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceInfo *d = &g_dev[dev];
    std::call_once(d->once, [d, dev] {
        int n = 0;
        d->err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (d->err != cudaSuccess) return;
        d->sms = n > 0 ? n : 1;
        d->err = cudaFuncSetAttribute(gemm_tc_kernel<1>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<1>::SMEM_BYTES);
        if (d->err != cudaSuccess) return;
        d->err = cudaFuncSetAttribute(gemm_tc_kernel<2, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<2, false>::SMEM_BYTES);
        if (d->err != cudaSuccess) return;
        d->err = cudaFuncSetAttribute(gemm_tc_kernel<2, true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg<2, true>::SMEM_BYTES);
        if (d->err != cudaSuccess) return;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = launch_config(2 * (d->sms / 2), 2, Cfg<2, false>::THREADS,
                                               Cfg<2, false>::SMEM_BYTES, 0, attr);
        cfg.attrs = attr + 1;  // the occupancy query takes the cluster shape only
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_kernel<2, false>, &cfg) !=
            cudaSuccess) {
            clusters = 0;
            (void)cudaGetLastError();  // clear it: the pair variant is then not used
        }
        d->pairs = clusters;
        cfg = launch_config(2 * (d->sms / 2), 2, Cfg<2, true>::THREADS, Cfg<2, true>::SMEM_BYTES,
                            0, attr);
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_kernel<2, true>, &cfg) !=
            cudaSuccess) {
            clusters = 0;
            (void)cudaGetLastError();  // clear it: the direct variant is then not used
        }
        d->pairs_direct = clusters;
    });
    return d;
}

// How many clusters of k single-CTA tensor-core kernels (each holding most of
// an SM's shared memory) the device can hold at once; asked once per k.  A
// cluster's CTAs must share a GPC, so this is below SMs / k when k does not
// divide a GPC's SM count.
int resident_clusters(DeviceInfo *d, int k) {
    std::lock_guard<std::mutex> lock(d->mu);
    if (d->clusters[k] < 0) {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg =
            launch_config(k * (d->sms / k), k, Cfg<1>::THREADS, Cfg<1>::SMEM_BYTES, 0, attr);
        cfg.attrs = attr + 1;  // the occupancy query takes the cluster shape only
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<1, false>, &cfg) != cudaSuccess) {
            n = 0;
            (void)cudaGetLastError();
        }
        d->clusters[k] = n;
    }
    return d->clusters[k];
}

template <int CG, bool DIRECT = false>
cudaError_t launch_variant(const Problem &p, const TcArgs &a0, int grid, cudaStream_t stream) {
    using C = Cfg<CG, DIRECT>;
    CUtensorMap map_a, map_b;
    const CUtensorMapDataType dt =
        a0.ab_format == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    bool ok;
    if (p.a_kmajor)  // A(i, k) at A[i * lda + k]: inner K, outer M; box 64 K x 128 rows
        // (single CTAs: am1 rows)
        ok = encode_2d(&map_a, dt, p.A, p.K, p.M, p.lda, BK,
                       CG == 1 ? static_cast<uint32_t>(a0.am1) : BM);
    else  // A(i, k) at A[i + k * lda]: inner M, outer K; boxes of 64 M x 64 K
        ok = encode_2d(&map_a, dt, p.A, p.M, p.K, p.lda, 64, BK);
    if (!ok) return cudaErrorInvalidValue;
    if (p.b_kmajor)  // B(k, j) at B[k + j * ldb]: inner K, outer N; box 64 K x B_ROWS
        // (single CTAs: bn1 rows)
        ok = encode_2d(&map_b, dt, p.B, p.K, p.N, p.ldb, BK,
                       CG == 1 ? static_cast<uint32_t>(a0.bk1) : C::B_ROWS);
    else  // B(k, j) at B[k * ldb + j]: inner N, outer K; boxes of 64 N x 64 K
        ok = encode_2d(&map_b, dt, p.B, p.N, p.K, p.ldb, 64, BK);
    if (!ok) return cudaErrorInvalidValue;
    // tail tiles split along N: a K-major B box of half the rows (an
    // MN-major B takes one 64-column box of map_b instead of two)
    CUtensorMap map_b_half = map_b;
    if (a0.tail_split_n && p.b_kmajor &&
        !encode_2d(&map_b_half, dt, p.B, p.K, p.N, p.ldb, BK, C::B_ROWS / 2))
        return cudaErrorInvalidValue;
    // C and D: FP32 row-major M x N; 32 x 32 boxes with the 128-byte swizzle
    CUtensorMap map_c, map_d;
    TcArgs a = a0;
    if (a.tma_c && !encode_box32_f32(&map_c, p.C, p.M, p.N, p.ldc)) a.tma_c = 0;
    if (a.tma_d) {
        bool ok_d;
        if (a.d_bf16) {
            // BF16 D: 32 x 32 boxes of 64-byte rows, unswizzled
            cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M)};
            cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ldd) * 2};
            cuuint32_t box[2] = {32, 32};
            cuuint32_t estr[2] = {1, 1};
            ok_d = g_encode(&map_d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.D, dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
                   CUDA_SUCCESS;
        } else {
            ok_d = encode_box32_f32(&map_d, p.D, p.M, p.N, p.ldd);
        }
        if (!ok_d) a.tma_d = 0;
    }
    if (!a.tma_c) map_c = map_a;  // unused placeholders
    if (!a.tma_d) map_d = map_a;
    a.tiles_m = (p.M + C::TILE_M - 1) / C::TILE_M;
    a.tiles_n = (p.N + BN - 1) / BN;
    cudaLaunchAttribute attr[2];
    // CTA pairs: clusters of 2; split single CTAs: clusters of ks
    const int cluster = CG == 2 ? 2 : (a.cluster_k ? a.ks : 1);
    cudaLaunchConfig_t cfg = launch_config(grid, cluster, C::THREADS, C::SMEM_BYTES, stream, attr);
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<CG, DIRECT>, map_a, map_b, map_b_half, map_c,
                              map_d, a);
}

}  // namespace

bool tc_eligible(const Problem &p) {
    // TMA: global base 16-byte aligned, row pitch a multiple of 16 bytes,
    // extents below 2^31 (coordinates are signed 32-bit).
    return aligned(p.A, 16) && aligned(p.B, 16) && (p.lda % 8 == 0) && (p.ldb % 8 == 0) &&
           p.M < (int64_t(1) << 31) && p.N < (int64_t(1) << 31) && p.K < (int64_t(1) << 31);
}

cudaError_t launch_tc(const Problem &p, InType in, cudaStream_t stream, const char **name) {
    if (in != InType::BF16 && in != InType::F16) return cudaErrorInvalidValue;
    const bool bf16 = in == InType::BF16;
    if (!tc_eligible(p)) return cudaErrorNotSupported;
    if (!load_encoder()) return cudaErrorSymbolNotFound;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DeviceInfo *d = device_info(dev);
    if (d == nullptr) return cudaErrorInvalidDevice;
    if (d->err != cudaSuccess) return d->err;

    TcArgs a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.C = p.C;
    a.ldc = p.ldc;
    a.D = p.D;
    a.ldd = p.ldd;
    a.num_kb = (p.K + BK - 1) / BK;
    a.a_kmajor = p.a_kmajor ? 1 : 0;
    a.b_kmajor = p.b_kmajor ? 1 : 0;
    // TMA needs a 16-byte aligned base and a pitch of whole 16 bytes, and its
    // stores clip at the matrix edge only in whole 16-byte pieces: C and D go
    // through TMA boxes only when a row of N elements is whole 16-byte pieces
    // (otherwise the coalesced row path runs).
    a.tma_c = (p.beta != 0.f && aligned(p.C, 16) && p.ldc % 4 == 0 && p.N % 4 == 0) ? 1 : 0;
    a.bias = p.bias;
    a.bias_per_row = p.bias_per_row ? 1 : 0;
    a.act = p.act;
    a.d_bf16 = p.d_bf16 ? 1 : 0;
    // D rows start on 16 bytes and hold whole 16-byte pieces: ldd and N
    // multiples of 4 (FP32) or 8 (BF16)
    const int64_t d_vec = p.d_bf16 ? 8 : 4;
    a.tma_d = (aligned(p.D, 16) && p.ldd % d_vec == 0 && p.N % d_vec == 0) ? 1 : 0;
    a.timeout_ns = 1000ull * 1000ull * 1000ull;  // 1 s per wait
    a.ks = 1;
    a.tail_first = 0;
    a.tail_ks = 1;
    a.tail_split_n = 0;
    a.ws = nullptr;
    a.ws_count = nullptr;
    a.cluster_k = 0;
    a.bn1 = BN;
    a.am1 = BM;
    a.bk1 = BN;
    a.a_region1 = Cfg<1>::A_BYTES;
    a.stages1 = Cfg<1>::STAGES;
    a.stage_bytes1 = Cfg<1>::STAGE_BYTES;
    a.ab_format = bf16 ? 1 : 0;

    // CTA pairs when there are at least as many 256 x 256 tiles as resident
    // pairs (large problems); single CTAs on 128 x 256 tiles otherwise.
    const int64_t pair_tiles = ((p.M + 255) / 256) * ((p.N + BN - 1) / BN);
    // The kernel's work-item arithmetic is 32-bit: at most 2^28 tiles of
    // 128 x 256 (a D of 2^43 elements, beyond any device's memory), times at
    // most 8 pieces each.
    if (((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN) > (int64_t(1) << 28))
        return cudaErrorInvalidValue;
    // D rows (and C rows, when beta != 0) that start on 32 bytes: the direct
    // epilogue (C and D through registers, no staging boxes), whose ring is
    // one stage deeper
    const int64_t d_per_32b = p.d_bf16 ? 16 : 8;
    const bool c_rows_32b = p.beta == 0.f || (aligned(p.C, 32) && p.ldc % 8 == 0);
    const bool direct = c_rows_32b && aligned(p.D, 32) && p.ldd % d_per_32b == 0 &&
                        d->pairs_direct > 0;
    const int pairs = direct ? d->pairs_direct : d->pairs;
    if (pairs > 0 && pair_tiles >= pairs) {
        *name = direct ? (bf16 ? "gemm_bf16_tc<pair,direct>" : "gemm_f16_tc<pair,direct>")
                       : (bf16 ? "gemm_bf16_tc<pair>" : "gemm_f16_tc<pair>");
        // The tiles of the last, partial round would leave pairs idle: when
        // they fill at most half of the pairs, split each so that round ends
        // sooner -- into its two N halves (whole K, no partial sums) when
        // they fill more than a quarter of the pairs and K is at most
        // kSplitNMaxKb blocks, else into tail_ks K ranges (2 to 4, at least
        // 4 K blocks each) whose partial sums the last piece adds.  (Timed on
        // GB300: at 4096^3 the N halves end the round 6 % sooner; at 8192^3
        // the two ways take the same time -- N = 128 MMAs move 1.5 x the
        // operand bytes per FLOP, and the K split's reduction is short
        // beside a half tile of 64 K blocks.)
        constexpr int64_t kSplitNMaxKb = 96;
        const int64_t groups = pairs;
        const int64_t tail = pair_tiles % groups;
        int64_t tail_ks = 1;
        if (tail > 0 && 2 * tail <= groups && 4 * tail > groups && a.num_kb <= kSplitNMaxKb) {
            tail_ks = 2;
            a.tail_split_n = 1;
        } else if (tail > 0 && 2 * tail <= groups) {
            tail_ks = groups / tail;
            if (tail_ks > 4) tail_ks = 4;
            if (tail_ks > a.num_kb / 4) tail_ks = a.num_kb / 4;
            if (tail_ks < 2) tail_ks = 1;
        }
        a.tail_first = tail_ks > 1 ? pair_tiles - tail : pair_tiles;
        a.tail_ks = static_cast<int>(tail_ks);
        void *ws = nullptr;
        SplitSync sync;  // the stream's split counters, held until the launch is enqueued
        if (a.tail_split_n) {
            *name = direct ? (bf16 ? "gemm_bf16_tc<pair,direct,split-n-tail>"
                                   : "gemm_f16_tc<pair,direct,split-n-tail>")
                           : (bf16 ? "gemm_bf16_tc<pair,split-n-tail>"
                                   : "gemm_f16_tc<pair,split-n-tail>");
        } else if (tail_ks > 1) {
            *name = direct ? (bf16 ? "gemm_bf16_tc<pair,direct,split-tail>"
                                   : "gemm_f16_tc<pair,direct,split-tail>")
                           : (bf16 ? "gemm_bf16_tc<pair,split-tail>" : "gemm_f16_tc<pair,split-tail>");
            // counters: per tail tile 2 CTAs x the epilogue warps (the
            // stream's, zero)
            const int epi_warps = direct ? Cfg<2, true>::EPI_WARPS : Cfg<2, false>::EPI_WARPS;
            e = sync.acquire(stream, static_cast<size_t>(tail) * 2 * epi_warps);
            if (e != cudaSuccess) return e;
            a.ws_count = sync.counters;
            // per tail tile and piece: 2 CTAs x 4 warps x 8 boxes of 4 KiB
            const size_t part_bytes = static_cast<size_t>(tail) * tail_ks * 2 * 4 * 8 * 4096;
            e = workspace_alloc(part_bytes, stream, &ws);
            if (e != cudaSuccess) return e;
            a.ws = static_cast<float *>(ws);
        }
        // (debug: one work item per pair)
        const int64_t pair_items = a.tail_first + (pair_tiles - a.tail_first) * a.tail_ks;
        const int grid2 = static_cast<int>(kDebug ? 2 * pair_items : 2 * pairs);
        e = direct ? launch_variant<2, true>(p, a, grid2, stream)
                   : launch_variant<2, false>(p, a, grid2, stream);
        if (ws != nullptr) {
            const cudaError_t ef = workspace_free(ws, stream);
            if (e == cudaSuccess) e = ef;
        }
        const cudaError_t er = sync.release();
        if (e == cudaSuccess) e = er;
    } else {
        const int64_t tiles = ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
        // Fewer tiles than SMs: split each tile's K range over the ks CTAs
        // of a cluster ("GEMM on NVIDIA GPUs", section 5, split-K for short
        // M / N), at most kMaxClusterK (the portable cluster size) and at
        // least 4 K blocks per piece; the pieces add their partial sums
        // through distributed shared memory, so no workspace is taken.  The
        // largest such ks whose clusters (one per tile) are all resident at
        // once: a second wave of clusters would double the time.
        int64_t ks = 1;
        if (tiles < d->sms) {
            ks = d->sms / tiles;
            if (ks > a.num_kb / 4) ks = a.num_kb / 4;
            if (ks > kMaxClusterK) ks = kMaxClusterK;
            while (ks >= 2 && resident_clusters(d, static_cast<int>(ks)) < tiles) --ks;
            if (ks < 2) ks = 1;
        }
        if (ks > 1) {
            static const char *const kNames[2][kMaxClusterK + 1] = {
                {"", "", "gemm_f16_tc<splitk,x2>", "gemm_f16_tc<splitk,x3>", "gemm_f16_tc<splitk,x4>",
                 "gemm_f16_tc<splitk,x5>", "gemm_f16_tc<splitk,x6>", "gemm_f16_tc<splitk,x7>",
                 "gemm_f16_tc<splitk,x8>"},
                {"", "", "gemm_bf16_tc<splitk,x2>", "gemm_bf16_tc<splitk,x3>",
                 "gemm_bf16_tc<splitk,x4>", "gemm_bf16_tc<splitk,x5>", "gemm_bf16_tc<splitk,x6>",
                 "gemm_bf16_tc<splitk,x7>", "gemm_bf16_tc<splitk,x8>"}};
            a.ks = static_cast<int>(ks);
            a.cluster_k = 1;
            *name = kNames[bf16 ? 1 : 0][ks];  // xN: the K range split over N CTAs
        } else {
            *name = bf16 ? "gemm_bf16_tc" : "gemm_f16_tc";
        }
        // N <= 128: one tile column with a 64- or 128-row B box and N = 64
        // or 128 MMAs, so a stage carries less of B's zero fill past N and
        // the ring holds 8 or 6 stages instead of 4 -- more of A in flight
        // when A is the stream (16384 x 64 x 8192)
        // M <= 64: load only the rows of A that hold data (at least 16 for a
        // K-major A, 64 -- one box -- for an M-major one); TMA then moves
        // fewer zero-filled rows per stage
        if (p.M <= 64) a.am1 = p.a_kmajor ? (p.M <= 16 ? 16 : (p.M <= 32 ? 32 : 64)) : 64;
        if (p.N <= BN / 2) {
            a.bn1 = p.N <= BN / 4 ? BN / 4 : BN / 2;
            a.bk1 = p.N <= 16 ? 16 : (p.N <= 32 ? 32 : a.bn1);
        }
        // stages packed tight: A's loaded rows, then the bn1 rows of B the
        // MMAs read; as many as the ring holds, at most MAX_STAGES
        a.a_region1 = static_cast<uint32_t>(a.am1 * BK * 2);
        a.stage_bytes1 = a.a_region1 + static_cast<uint32_t>(a.bn1 * BK * 2);
        const int fit = static_cast<int>(Cfg<1>::STAGES * Cfg<1>::STAGE_BYTES / a.stage_bytes1);
        a.stages1 = fit < Cfg<1>::MAX_STAGES ? fit : Cfg<1>::MAX_STAGES;
        if (kDebug) a.stages1 = 2;
        const int64_t items = tiles * ks;
        // (debug: one item per CTA; items < 2^31 by the tile bound above)
        const int grid = static_cast<int>(kDebug || items < d->sms ? items : d->sms);
        e = launch_variant<1>(p, a, grid, stream);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_tc_probe(int cta_group, int64_t n_mma, cudaStream_t stream, double *flops) {
    if ((cta_group != 1 && cta_group != 2) || n_mma < 1) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DeviceInfo *d = device_info(dev);
    if (d == nullptr) return cudaErrorInvalidDevice;
    if (d->err != cudaSuccess) return d->err;
    // one CTA per SM: the shared memory of the GEMM kernel keeps a second
    // CTA (and its TMEM allocation) off the SM
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    std::call_once(once[dev], [dev] {
        attr_err[dev] = cudaFuncSetAttribute(tc_probe_kernel<1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<1>::SMEM_BYTES);
        if (attr_err[dev] == cudaSuccess)
            attr_err[dev] = cudaFuncSetAttribute(tc_probe_kernel<2>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Cfg<2>::SMEM_BYTES);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    const int groups = cta_group == 1 ? d->sms : d->pairs;
    if (groups < 1) return cudaErrorNotSupported;
    // 1 s per wait, and at least 4x the time the MMAs take at 2 PFLOP/s
    const double mma_flops = 2.0 * BM * cta_group * BN * UMMA_K;
    const double est_ns = static_cast<double>(n_mma) * mma_flops * groups / 2.0e6;
    const uint64_t timeout_ns = static_cast<uint64_t>(est_ns * 4 > 1e9 ? est_ns * 4 : 1e9);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    cfg.gridDim = dim3(static_cast<unsigned>(groups * cta_group), 1, 1);
    cfg.blockDim = dim3(PROBE_THREADS, 1, 1);
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 0;
    if (cta_group == 2) {
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.numAttrs = 1;
        cfg.dynamicSmemBytes = Cfg<2>::SMEM_BYTES;
        e = cudaLaunchKernelEx(&cfg, tc_probe_kernel<2>, n_mma, timeout_ns);
    } else {
        cfg.dynamicSmemBytes = Cfg<1>::SMEM_BYTES;
        e = cudaLaunchKernelEx(&cfg, tc_probe_kernel<1>, n_mma, timeout_ns);
    }
    if (e != cudaSuccess) return e;
    *flops = mma_flops * static_cast<double>(n_mma) * groups;
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(uint64_t timeout_ns, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns);
    return cudaGetLastError();
}

cudaError_t tc_read_and_clear_status(cudaStream_t stream, int *status) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_tc_status, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                    stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e;
}

}  // namespace gemm
