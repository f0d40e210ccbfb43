// Fused matmul + all-gather for sm_103a (iris PR #626, "Summary" and
// "Benchmark": the matmul's epilogue all-gathers each output tile, with the
// heap-base translation hoisted above the K loop).
//
// C_r = A_r @ B for every source r of the launch.  Persistent CTAs, one per
// SM.  Three kernels, chosen by the caller's tile and path:
//   * mag2w (128 x 512 CTA tile): CTA pairs (clusters of 2) on 256 x 512
//     tiles, two tcgen05.mma.cta_group::2 per K step sharing the A stage; a
//     last wave at most half full runs as 256 x 256 half tiles (wide::Unit);
//     see the "wide pair tiles" section below for how it differs from mag2;
//   * mag2 (128 x 256 CTA tile): CTA pairs on 256 x 256 tiles;
//   * mag1 (128 x 256 CTA tile, one CTA): 128 x 256 tiles.
// Tiles are taken in column groups, so that a wave of tiles reads few
// distinct slices of A and B (see tile_coord).  Per CTA of mag1 / mag2:
//   * warp 0 (producer): TMA tensor loads of A (128 x 64, K-major) and of the
//     CTA's columns of B (64-deep, N-major, 64-column boxes; one 3-d box per
//     stage when N is a multiple of 64) into a ring of 128B-swizzled stages
//     (6 on 2 SMs, 4 on 1 SM); a pair's loads complete on the leader's
//     mbarriers;
//   * warp 1 (MMA): allocates 512 TMEM columns (two fp32 accumulators) and,
//     in the leader, issues tcgen05.mma kind::f16 (M=256 or 128, N=256,
//     K=16) from one thread; tcgen05.commit frees ring stages (in both CTAs
//     of a pair) and hands finished accumulators to the epilogue;
//   * warps 2-5 (epilogue): tcgen05.ld of their 32 TMEM lanes (= tile rows),
//     round to f16/bf16 and write each value once into shared memory as
//     32-row x 64-column boxes in the 128-byte swizzled layout, then one TMA
//     tensor store (cp.async.bulk.tensor shared->global) per box and
//     destination: the local copy first, then the peers in rotated order,
//     one destination per time slot spread over most of a tile period (store
//     pacing: the CTAs' epilogues would otherwise coincide and flood DRAM
//     with writes while the next tile's operands load).
//     The accumulator is released right after it has been read, so the next
//     tile's MMAs overlap this tile's stores.
// Each destination's tensor map is built on the host from the heap-bases
// table once per launch (the per-peer translation hoisted out of every loop);
// the map views that member's output as {N, M, W} so that a box is clipped at
// the end of its own row block.
//
// Every mbarrier wait is bounded (wall-clock limit from the launch); a wait
// that gives up stores GG_ERR_TIMEOUT in the status word, raises a CTA-wide
// abort flag, and every role then drains what it has in flight (loads, MMAs,
// stores) before the TMEM is freed and the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gg_internal.h"
#include "ptx.cuh"

namespace gg {
namespace {

constexpr int BM = 128, BN = 256, UK = 16;
constexpr int kMaxStages = 8;
// B stages load as one 3-d box (when N is a multiple of 64) instead of one
// 2-d box per 64 columns: one TMA instruction fewer per stage (measured
// +0-2.5%).
constexpr bool kBBoxes3d = true;
// Bytes of B one column group of the tile order may span (see tile_coord):
// 256-column / 512-column pair tiles (measured best at N=3584, K=8192:
// groups of 7 narrow tiles, one group of 7 wide ones).
constexpr int64_t kBGroupBytes = 32ll << 20;
constexpr int64_t kBGroupBytesWide = 64ll << 20;
constexpr int kKAtom = 64;                      // K elements of one 128-byte swizzle row
constexpr int kAAtom = BM * kKAtom * 2;         // 16 KB: 128 rows x 64 K, K-major
constexpr int kThreads = 192;                   // 6 warps
constexpr int kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 1000000000ull;

constexpr int kBox = 32 * 64 * 2;               // 4 KB: one epilogue store box, 32 rows x 64 cols
// Store pacing: the W copies of a tile go out in slots spread over this share
// of the previous tile's period (see the epilogue), and a period is capped at
// kPaceMaxPeriodNs so that a stalled tile cannot stretch the next one's waits.
constexpr uint64_t kPacePct = 70;
constexpr uint64_t kPaceMaxPeriodNs = 2000000ull;

// Geometry of the 1-SM (CG = 1) and 2-SM (CG = 2) variants.  With CG = 2 a
// CTA pair computes a 256 x 256 tile: each CTA holds its 128 rows of A and
// one 128-column half of B; the leader CTA's single thread issues
// tcgen05.mma.cta_group::2 over both CTAs' shared memory and TMEM.
template <int CG>
struct Geo {
    // K depth of one ring stage: 64 (one swizzle atom of A) or 128 (two)
    static constexpr int kBK = CG == 1 ? 64 : 64;
    static constexpr int kStages = CG == 1 ? 4 : 6;
    static constexpr int kAStage = BM * kBK * 2;       // A: kBK/64 atoms of 128 rows
    static constexpr int kBBox = kBK * 64 * 2;         // B box: kBK K-rows x 64 N-columns
    static constexpr int kBCols = BN / CG;             // B columns one CTA holds
    static constexpr int kBStage = kBK * kBCols * 2;   // kBCols/64 boxes
    static constexpr int kTileM = BM * CG;            // rows of one (pair) tile
    // The epilogue stages each warp's 32 rows in column passes of kEpiCols,
    // as kEpiCols/64 swizzled boxes.
    static constexpr int kEpiCols = CG == 1 ? 64 : 128;
    static constexpr int kEpiBoxes = kEpiCols / 64;
    static constexpr int kEpiWarp = kEpiBoxes * kBox;  // one epilogue warp's staging
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kAStage;
    static constexpr int kOffEpi = kOffB + kStages * kBStage;
    static constexpr int kOffShared = kOffEpi + 4 * kEpiWarp;
};

struct FusedShared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

template <int CG>
constexpr int smem_bytes()
{
    return Geo<CG>::kOffShared + (int)sizeof(FusedShared) + 1024;  // + alignment slack
}
static_assert(Geo<1>::kStages <= kMaxStages && Geo<2>::kStages <= kMaxStages, "ring barriers");
static_assert(smem_bytes<1>() <= 232448 && smem_bytes<2>() <= 232448,
              "at most 227 KB of dynamic shared memory per CTA");

// ---- tcgen05 / TMA / cluster wrappers --------------------------------------------
template <int CG>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar, uint64_t policy)
{
    if constexpr (CG == 1)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
            "cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
            : "memory");
    else  // the barrier may sit in the peer CTA of the pair
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
            "bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
            : "memory");
}

template <int CG>
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy)
{
    if constexpr (CG == 1)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
            "cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
            "bytes.L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
            : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// shared -> global tensor store of one box; completion by bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], "
        "[%1], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t ncluster_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (any CTA of the cluster).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
                 : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t slot)
{
    if constexpr (CG == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t tmem)
{
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 version (1)
//   bits 49-51 base offset (0: atoms are 1024-byte aligned)
//   bits 61-63 layout (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B f16 (0) or bf16 (1),
// A K-major, B N-major, N = 256, M = 128 * CG.
__host__ __device__ constexpr uint32_t instr_desc(int bf16, int cg)
{
    return (1u << 4)                           // D format: f32
           | ((uint32_t)bf16 << 7)             // A format
           | ((uint32_t)bf16 << 10)            // B format
           | (0u << 15)                        // A major: K
           | (1u << 16)                        // B major: MN
           | ((uint32_t)(BN >> 3) << 17)       // N >> 3
           | ((uint32_t)((BM * cg) >> 4) << 24); // M >> 4
}

template <int CG>
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate)
{
    if constexpr (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive on `bar` once the issuing thread's earlier MMAs are done; with CG = 2
// the arrival goes to the barrier at that offset in both CTAs of the pair.
template <int CG>
__device__ __forceinline__ void mma_commit_all(uint32_t bar)
{
    if constexpr (CG == 1)
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
            "[%0], %1;" ::"r"(bar),
            "h"((uint16_t)0x3)
            : "memory");
}

// Arrive on `bar` in the issuing CTA only.
template <int CG>
__device__ __forceinline__ void mma_commit_local(uint32_t bar)
{
    if constexpr (CG == 1)
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Wait for this thread's tcgen05.ld to complete.  The loaded registers are
// passed through as in/out operands so no use of them can be scheduled
// before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Orders later uses of r after the preceding volatile asm (a tcgen05 wait).
__device__ __forceinline__ void reg_order(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi, int bf16)
{
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Bounded wait that also gives up as soon as another role raised the abort flag.
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile int *abort_flag)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity))
                return true;
        if (*abort_flag || ptx::globaltimer() - t0 > limit_ns)
            return false;
    }
}

__device__ __forceinline__ void sleep_ns(uint64_t ns)
{
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < ns)
        __nanosleep(1000);
}

struct TileCoord {
    int g;        // group index of the source
    int h;        // heap index of the source
    int tm, tn;
};

// Tile order: the tile columns are split into groups of a.tn_group; group by
// group, every (source, tile row) runs over the group's columns.  A wave of
// concurrent tiles (one per CTA pair) then covers about (pairs / group)
// tile rows and the group's columns, whose slices of A and B it reads from
// DRAM once and shares through L2.  A is read once per group; the group's
// slice of B, hinted evict_last, is nevertheless re-read about once per wave
// on GB300 (measured with ncu), and groups of 7 at N=3584 read the least.
__device__ __forceinline__ TileCoord tile_coord(const FusedArgs &a, int64_t t, int tiles_m,
                                                int tiles_n)
{
    TileCoord c;
    const int gw = a.tn_group;
    const int64_t rows = (int64_t)a.n_src * tiles_m;  // (source, tile row) pairs
    const int j = (int)(t / (rows * gw));              // column group
    const int64_t r = t - (int64_t)j * rows * gw;
    const int width = tiles_n - j * gw < gw ? tiles_n - j * gw : gw;
    const int64_t sr = r / width;
    const int s = (int)(sr / tiles_m);
    c.g = a.src_first + s;
    c.h = a.rank_start + c.g * a.rank_stride;
    c.tm = (int)(sr - (int64_t)s * tiles_m);
    c.tn = j * gw + (int)(r - sr * width);
    return c;
}

template <int CG>
__device__ __forceinline__ void mag_body(const CUtensorMap &map_a, const CUtensorMap &map_b,
                                         const OutMaps &out, const FusedArgs &a)
{
    using G = Geo<CG>;
    trace_mark(a.trace, 0);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned for the 128B swizzle
    uint8_t *smem = smem_raw + (base - raw);
    FusedShared &sh = *reinterpret_cast<FusedShared *>(smem + G::kOffShared);
    volatile int *abort_flag = &sh.abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // position in the CTA pair
    const bool leader = rank == 0;
    const int64_t unit = CG == 2 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
    const int64_t nunits = CG == 2 ? (int64_t)ncluster_x() : (int64_t)gridDim.x;
    const int tiles_m = (int)((a.M + G::kTileM - 1) / G::kTileM);
    const int tiles_n = (int)((a.N + BN - 1) / BN);
    const int64_t total = (int64_t)a.n_src * tiles_m * tiles_n;
    const int num_kb = (int)((a.K + G::kBK - 1) / G::kBK);

    // ---- prologue: barriers, TMEM, destination bases (loaded once) ----------
    if (threadIdx.x == 0) {
        for (int s = 0; s < G::kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sh.full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sh.tmem_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.tmem_empty[s]), 4 * CG);
        }
        ptx::mbar_init(ptx::smem_addr(&sh.mma_done), 1);
        sh.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        tmem_alloc<CG>(ptx::smem_addr(&sh.tmem_base));
        tc_fence_before();
    }
    if (threadIdx.x < (unsigned)a.W)
        prefetch_tensormap(&out.map[threadIdx.x]);  // the member output maps, once
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ===================== producer =====================================
        const uint64_t pol_a = ptx::policy_evict_normal();  // A tile: read by tiles_n CTAs
        const uint64_t pol_b = ptx::policy_evict_last();    // B: read by every tile row
        constexpr uint32_t kTx = CG * (G::kAStage + G::kBStage);  // bytes of one stage, both CTAs
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        for (int64_t t = unit; t < total && ok; t += nunits) {
            const TileCoord c = tile_coord(a, t, tiles_m, tiles_n);
            const int h_coord = a.a_abs ? 0 : c.h;
            const int row0 = c.tm * G::kTileM + (int)rank * BM;
            const int col0 = c.tn * BN + (int)rank * G::kBCols;
            for (int kq = 0; kq < num_kb; ++kq) {  // the K block this stage carries
                const bool got = role_wait(ptx::smem_addr(&sh.empty[stage]), phase ^ 1u,
                                           a.wait_limit_ns, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const bool stall = a.inject_stall && unit == 0 && issued == 0;
                if (lane == 0 && !stall) {  // test hook: the first stage is never armed
                    const uint32_t local_full = ptx::smem_addr(&sh.full[stage]);
                    // every CTA's loads complete on the leader's barrier of this stage
                    const uint32_t bar = CG == 2 ? map_to_rank(local_full, 0) : local_full;
                    if (leader)
                        ptx::mbar_arrive_expect_tx(local_full, kTx);
                    const uint32_t sa = base + G::kOffA + stage * G::kAStage;
                    const uint32_t sb = base + G::kOffB + stage * G::kBStage;
#pragma unroll
                    for (int ka = 0; ka < G::kBK / kKAtom; ++ka)
                        tma_load_3d<CG>(sa + ka * kAAtom, &map_a, kq * G::kBK + ka * kKAtom, row0,
                                        h_coord, bar, pol_a);
                    if (a.b_boxes3d) {
                        // B viewed as {64 columns, K, N/64 chunks}: the kBCols/64
                        // boxes of the stage in one copy (same shared layout)
                        tma_load_3d<CG>(sb, &map_b, 0, kq * G::kBK, col0 / 64, bar, pol_b);
                    } else {
#pragma unroll
                        for (int j = 0; j < G::kBCols / 64; ++j)
                            tma_load_2d<CG>(sb + j * G::kBBox, &map_b, col0 + j * 64, kq * G::kBK,
                                            bar, pol_b);
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == G::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        // drain: every load this warp issued has landed before the CTA may exit
        if (leader) {
            const int64_t pending = issued < G::kStages ? issued : G::kStages;
            for (int64_t q = 0; q < pending; ++q) {
                const int64_t idx = issued - 1 - q;  // the q-th most recent k-block
                const int s = (int)(idx % G::kStages);
                const uint32_t ph = (uint32_t)((idx / G::kStages) & 1);
                ptx::mbar_wait(ptx::smem_addr(&sh.full[s]), ph, kDrainLimitNs);
            }
        } else if (!ok && issued > 0) {
            // the peer's loads complete on the leader's barriers, which it cannot
            // wait on: give copies already in flight time to land
            sleep_ns(200000);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer (leader CTA) ======================
        const uint32_t idesc = instr_desc(a.is_bf16, CG);
        int stage = 0;
        uint32_t phase = 0;
        int64_t lt = 0;  // local tile count
        bool issued_any = false;
        bool ok = true;
        for (int64_t t = unit; leader && t < total && ok; t += nunits, ++lt) {
            const int acc = (int)(lt & 1);
            const uint32_t acc_phase = (uint32_t)((lt >> 1) & 1);
            const bool free_acc = role_wait(ptx::smem_addr(&sh.tmem_empty[acc]), acc_phase ^ 1u,
                                            a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, free_acc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
            for (int kb = 0; kb < num_kb; ++kb) {
                const bool got = role_wait(ptx::smem_addr(&sh.full[stage]), phase, a.wait_limit_ns,
                                           abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = base + G::kOffA + stage * G::kAStage;
                    const uint32_t sb = base + G::kOffB + stage * G::kBStage;
#pragma unroll
                    for (int k = 0; k < G::kBK / UK; ++k) {
                        // A: K-major, atom k/4, +32 bytes per 16-element K step inside the
                        // 128-byte row; SBO = 8 rows x 128 B
                        const uint32_t a_at =
                            sa + (uint32_t)((k / (kKAtom / UK)) * kAAtom + (k % (kKAtom / UK)) * UK * 2);
                        const uint64_t ad = smem_desc(a_at, 16, 1024);
                        // B: N-major, +16 K-rows x 128 B per K step; LBO = next 64-column
                        // box, SBO = 8 K-rows x 128 B
                        const uint64_t bd = smem_desc(sb + k * (UK * 128), G::kBBox, 1024);
                        mma_f16<CG>(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit_all<CG>(ptx::smem_addr(&sh.empty[stage]));
                }
                __syncwarp();
                issued_any = true;
                if (++stage == G::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit_all<CG>(ptx::smem_addr(&sh.tmem_full[acc]));
            __syncwarp();
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        // drain: all MMAs of this thread have completed before TMEM is freed
        if (issued_any) {
            if (lane == 0)
                mma_commit_local<CG>(ptx::smem_addr(&sh.mma_done));
            __syncwarp();
            ptx::mbar_wait(ptx::smem_addr(&sh.mma_done), 0, kDrainLimitNs);
        }
    } else {
        // ===================== epilogue (warps 2-5) =========================
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t warp_stage = base + G::kOffEpi + (uint32_t)(q * G::kEpiWarp);
        const uint32_t my_row = warp_stage + (uint32_t)lane * 128u;  // row `lane` of box 0
        const uint32_t swz = (uint32_t)(lane & 7);                  // 128-byte swizzle phase
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const uint64_t pol_c = ptx::policy_evict_first();  // output: written once, never read
        constexpr int kOps = G::kEpiBoxes;                   // stores per destination per pass
        constexpr int kPasses = BN / G::kEpiCols;
        int64_t lt = 0;
        bool ok = true;
        // Store pacing.  Every CTA runs its K loop in step with the others, so
        // their epilogues would all fire at once and put a whole wave of W-fold
        // output writes on DRAM in a burst that starves the operand loads.
        // Instead a tile's W x kPasses store groups leave in evenly spaced
        // slots across kPacePct of the previous tile's period (the first
        // tile's period counts from the kernel's start), overlapping the next
        // tile's mainloop; a CTA's last tile, with no mainloop behind it, is
        // not paced.
        uint64_t prev_ready = ptx::globaltimer();
        for (int64_t t = unit; t < total; t += nunits, ++lt) {
            const TileCoord c = tile_coord(a, t, tiles_m, tiles_n);
            const int acc = (int)(lt & 1);
            const uint32_t acc_phase = (uint32_t)((lt >> 1) & 1);
            const bool got = role_wait(ptx::smem_addr(&sh.tmem_full[acc]), acc_phase,
                                       a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint64_t t_ready = ptx::globaltimer();
            uint64_t period = t_ready - prev_ready;
            period = period > kPaceMaxPeriodNs ? kPaceMaxPeriodNs : period;
            prev_ready = t_ready;
            // time between two store groups of this tile (0: no pacing)
            const uint64_t slot =
                t + nunits < total ? period * kPacePct / 100u / (uint64_t)(kPasses * a.W) : 0;
            tc_fence_after();
            const uint32_t t_addr = tmem + lane_addr + (uint32_t)(acc * BN);
            // first row of this warp's boxes, within the source's row block
            const int row0 = c.tm * G::kTileM + (int)rank * BM + q * 32;
#pragma unroll 1
            for (int pass = 0; pass < BN; pass += G::kEpiCols) {
                // the staging boxes are free once this warp's previous stores read them
                ptx::bulk_wait_read<0>();
                __syncwarp();
#pragma unroll 1
                for (int b = 0; b < G::kEpiBoxes; ++b) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(t_addr + (uint32_t)(pass + b * 64), v0);
                    tmem_ld_32x32b_x32(t_addr + (uint32_t)(pass + b * 64 + 32), v1);
                    tmem_wait_ld(v0);
                    reg_order(v1);
                    // 16-byte chunk k of the row holds columns 8k..8k+7 and sits at
                    // chunk position k ^ (row mod 8) (the 128-byte swizzle)
                    const uint32_t rowp = my_row + (uint32_t)(b * kBox);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_shared_v4(rowp + ((((uint32_t)k) ^ swz) << 4),
                                     pack2(v0[8 * k], v0[8 * k + 1], a.is_bf16),
                                     pack2(v0[8 * k + 2], v0[8 * k + 3], a.is_bf16),
                                     pack2(v0[8 * k + 4], v0[8 * k + 5], a.is_bf16),
                                     pack2(v0[8 * k + 6], v0[8 * k + 7], a.is_bf16));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_shared_v4(rowp + ((((uint32_t)(k + 4)) ^ swz) << 4),
                                     pack2(v1[8 * k], v1[8 * k + 1], a.is_bf16),
                                     pack2(v1[8 * k + 2], v1[8 * k + 3], a.is_bf16),
                                     pack2(v1[8 * k + 4], v1[8 * k + 5], a.is_bf16),
                                     pack2(v1[8 * k + 6], v1[8 * k + 7], a.is_bf16));
                }
                if (pass + G::kEpiCols >= BN) {
                    // accumulator fully read: hand it back to the (leader's) MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t e = ptx::smem_addr(&sh.tmem_empty[acc]);
                        if constexpr (CG == 2)
                            mbar_arrive_cluster(map_to_rank(e, 0));
                        else
                            ptx::mbar_arrive(e);
                    }
                }
                // staged boxes -> every destination, local first, peers rotated
                const int col0 = c.tn * BN + pass;
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (row0 < a.M && slot != 0) {
                    // one destination per slot: lane b stores box b
                    const uint64_t first = (uint64_t)(pass / G::kEpiCols) * (uint64_t)a.W;
                    for (int j = 0; j < a.W; ++j) {
                        const uint64_t due = t_ready + slot * (first + (uint64_t)j);
                        while (ptx::globaltimer() < due && !*abort_flag)
                            __nanosleep(256);
                        const int col = col0 + lane * 64;
                        if (lane < kOps && col < a.N) {
                            int i = c.g + j;
                            if (i >= a.W)
                                i -= a.W;
                            tma_store_3d(&out.map[i], warp_stage + (uint32_t)(lane * kBox), col,
                                         row0, c.g, pol_c);
                        }
                    }
                } else if (row0 < a.M) {
                    for (int op = lane; op < a.W * kOps; op += 32) {
                        const int j = op / kOps;
                        const int b = op - j * kOps;
                        const int col = col0 + b * 64;
                        if (col >= a.N)
                            continue;
                        int i = c.g + j;
                        if (i >= a.W)
                            i -= a.W;
                        tma_store_3d(&out.map[i], warp_stage + (uint32_t)(b * kBox), col, row0, c.g,
                                     pol_c);
                    }
                }
                ptx::bulk_commit();
            }
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        ptx::bulk_wait_all();
    }

    // ---- teardown ---------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2)
        cluster_sync();  // the leader's MMAs into the peer's TMEM and smem are done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem);
    }
    trace_mark(a.trace, 1);
}

__global__ void __launch_bounds__(kThreads, 1)
    mag1_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ OutMaps out, const FusedArgs a)
{
    mag_body<1>(map_a, map_b, out, a);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mag2_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ OutMaps out, const FusedArgs a)
{
    mag_body<2>(map_a, map_b, out, a);
}

// ---- wide pair tiles: 256 x 512 per CTA pair ------------------------------------
// The same pipeline with two N=256 MMAs per K step, side by side, sharing the
// A stage: a stage (A 16 KB + this CTA's 256 columns of B, 32 KB) feeds twice
// the tensor work of a 256 x 256 stage, so the 4-stage ring holds about a
// third more tensor time in flight.  The accumulator takes all 512 TMEM
// columns; eight epilogue warps (two per TMEM lane quarter, 256 columns each)
// copy it into registers as packed f16/bf16 right after the tile's last MMA
// and release it, then store from registers through one staged box per warp.
namespace wide {
constexpr int kStages = 4;
constexpr int kBK = 64;                          // one 128-byte swizzle atom of A
constexpr int kAStage = BM * kBK * 2;            // 16 KB
constexpr int kBBox = kBK * 64 * 2;              // 8 KB: 64 K-rows x 64 columns
constexpr int kBHalf = 2 * kBBox;                // this CTA's 128 columns of one N half
constexpr int kBStage = 2 * kBHalf;              // both N halves: 32 KB
constexpr int kTileM = 2 * BM;                   // 256 rows per pair tile
constexpr int kTileN = 2 * BN;                   // 512 columns per pair tile
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;    // producer, MMA, 8 epilogue warps
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAStage;
constexpr int kOffEpi = kOffB + kStages * kBStage;
constexpr int kOffShared = kOffEpi + kEpiWarps * kBox;
constexpr int kSmemBytes = kOffShared + (int)sizeof(FusedShared) + 1024;
static_assert(kSmemBytes <= 232448, "at most 227 KB of dynamic shared memory per CTA");
static_assert(kStages <= kMaxStages, "ring barriers");

// Work units.  A pair tile is one unit, except in a last wave that is at
// most half full (total mod pairs <= pairs / 2): its tiles are split into
// their two N halves (256 x 256 each, one MMA per K step), so that twice as
// many pairs share the tail and the kernel ends half a tile earlier.  Units
// [0, full) are whole tiles; unit full + 2j + h is half h of tile full + j.
struct Unit {
    int64_t t;   // pair tile
    int h0, nh;  // N halves computed: [h0, h0 + nh)
};

__device__ __forceinline__ Unit unit_of(int64_t u, int64_t full)
{
    Unit w;
    if (u < full) {
        w.t = u;
        w.h0 = 0;
        w.nh = 2;
    } else {
        const int64_t v = u - full;
        w.t = full + v / 2;
        w.h0 = (int)(v & 1);
        w.nh = 1;
    }
    return w;
}
}  // namespace wide

__device__ __forceinline__ void magw_body(const CUtensorMap &map_a, const CUtensorMap &map_b,
                                          const OutMaps &out, const FusedArgs &a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned for the 128B swizzle
    uint8_t *smem = smem_raw + (base - raw);
    FusedShared &sh = *reinterpret_cast<FusedShared *>(smem + wide::kOffShared);
    volatile int *abort_flag = &sh.abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t unit = (int64_t)cluster_id_x();
    const int64_t nunits = (int64_t)ncluster_x();
    const int tiles_m = (int)((a.M + wide::kTileM - 1) / wide::kTileM);
    const int tiles_n = (int)((a.N + wide::kTileN - 1) / wide::kTileN);
    const int64_t total = (int64_t)a.n_src * tiles_m * tiles_n;
    const int64_t rem = total % nunits;
    const int64_t full = rem != 0 && 2 * rem <= nunits ? total - rem : total;
    const int64_t units = total + (total - full);  // a split tile is two units
    const int num_kb = (int)((a.K + wide::kBK - 1) / wide::kBK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < wide::kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sh.full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sh.tmem_full[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&sh.tmem_empty[0]), 2 * wide::kEpiWarps);
        ptx::mbar_init(ptx::smem_addr(&sh.mma_done), 1);
        sh.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_a);
        prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        tmem_alloc<2>(ptx::smem_addr(&sh.tmem_base));
        tc_fence_before();
    }
    if (threadIdx.x < (unsigned)a.W)
        prefetch_tensormap(&out.map[threadIdx.x]);
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ===================== producer =====================================
        trace_mark(a.trace, 0);
        const uint64_t pol_a = ptx::policy_evict_normal();
        const uint64_t pol_b = ptx::policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        for (int64_t u = unit; u < units && ok; u += nunits) {
            const wide::Unit w = wide::unit_of(u, full);
            const TileCoord c = tile_coord(a, w.t, tiles_m, tiles_n);
            // bytes of one stage, both CTAs: A and the unit's halves of B
            const uint32_t tx = 2u * (uint32_t)(wide::kAStage + w.nh * wide::kBHalf);
            const int h_coord = a.a_abs ? 0 : c.h;
            const int row0 = c.tm * wide::kTileM + (int)rank * BM;
            const int colh0 = c.tn * wide::kTileN + (int)rank * (BN / 2);  // N half 0
            for (int kq = 0; kq < num_kb; ++kq) {
                const bool got = role_wait(ptx::smem_addr(&sh.empty[stage]), phase ^ 1u,
                                           a.wait_limit_ns, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const bool stall = a.inject_stall && unit == 0 && issued == 0;
                if (lane == 0 && !stall) {  // test hook: the first stage is never armed
                    const uint32_t local_full = ptx::smem_addr(&sh.full[stage]);
                    const uint32_t bar = map_to_rank(local_full, 0);
                    if (leader)
                        ptx::mbar_arrive_expect_tx(local_full, tx);
                    const uint32_t sa = base + wide::kOffA + stage * wide::kAStage;
                    const uint32_t sb = base + wide::kOffB + stage * wide::kBStage;
                    tma_load_3d<2>(sa, &map_a, kq * wide::kBK, row0, h_coord, bar, pol_a);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh >= w.nh)
                            break;
                        const int h = w.h0 + hh;
                        const int col0 = colh0 + h * BN;
                        if (a.b_boxes3d) {
                            tma_load_3d<2>(sb + h * wide::kBHalf, &map_b, 0, kq * wide::kBK,
                                           col0 / 64, bar, pol_b);
                        } else {
#pragma unroll
                            for (int j = 0; j < 2; ++j)
                                tma_load_2d<2>(sb + h * wide::kBHalf + j * wide::kBBox, &map_b,
                                               col0 + j * 64, kq * wide::kBK, bar, pol_b);
                        }
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == wide::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        if (leader) {
            const int64_t pending = issued < wide::kStages ? issued : wide::kStages;
            for (int64_t q = 0; q < pending; ++q) {
                const int64_t idx = issued - 1 - q;
                const int s = (int)(idx % wide::kStages);
                const uint32_t ph = (uint32_t)((idx / wide::kStages) & 1);
                ptx::mbar_wait(ptx::smem_addr(&sh.full[s]), ph, kDrainLimitNs);
            }
        } else if (!ok && issued > 0) {
            sleep_ns(200000);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer (leader CTA) ======================
        const uint32_t idesc = instr_desc(a.is_bf16, 2);
        int stage = 0;
        uint32_t phase = 0;
        int64_t lt = 0;
        bool issued_any = false;
        bool ok = true;
        for (int64_t u = unit; leader && u < units && ok; u += nunits, ++lt) {
            const wide::Unit w = wide::unit_of(u, full);
            // the epilogue has copied the previous tile's accumulator out of TMEM
            const bool free_acc = role_wait(ptx::smem_addr(&sh.tmem_empty[0]),
                                            (uint32_t)(lt & 1) ^ 1u, a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, free_acc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kb = 0; kb < num_kb; ++kb) {
                const bool got = role_wait(ptx::smem_addr(&sh.full[stage]), phase, a.wait_limit_ns,
                                           abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = base + wide::kOffA + stage * wide::kAStage;
                    const uint32_t sb = base + wide::kOffB + stage * wide::kBStage;
#pragma unroll
                    for (int k = 0; k < wide::kBK / UK; ++k) {
                        const uint64_t ad = smem_desc(sa + (uint32_t)(k * UK * 2), 16, 1024);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            if (hh >= w.nh)
                                break;
                            const int h = w.h0 + hh;
                            const uint64_t bd = smem_desc(
                                sb + (uint32_t)(h * wide::kBHalf + k * (UK * 128)), wide::kBBox, 1024);
                            mma_f16<2>(tmem + (uint32_t)(h * BN), ad, bd, idesc,
                                       (kb | k) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit_all<2>(ptx::smem_addr(&sh.empty[stage]));
                }
                __syncwarp();
                issued_any = true;
                if (++stage == wide::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit_all<2>(ptx::smem_addr(&sh.tmem_full[0]));
            __syncwarp();
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        if (issued_any) {
            if (lane == 0)
                mma_commit_local<2>(ptx::smem_addr(&sh.mma_done));
            __syncwarp();
            ptx::mbar_wait(ptx::smem_addr(&sh.mma_done), 0, kDrainLimitNs);
        }
    } else {
        // ===================== epilogue (warps 2-9) =========================
        const int ew = warp - 2;                   // 0..7
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        const int half = ew >> 2;                  // columns [half*256, half*256 + 256)
        const uint32_t staging = base + wide::kOffEpi + (uint32_t)(ew * kBox);
        const uint32_t my_row = staging + (uint32_t)lane * 128u;  // row `lane` of the box
        const uint32_t swz = (uint32_t)(lane & 7);
        const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * BN);
        const uint64_t pol_c = ptx::policy_evict_first();
        constexpr int kBoxes = BN / 64;            // 4 boxes of 64 columns per warp and tile
        int64_t lt = 0;
        bool ok = true;
        uint64_t prev_ready = ptx::globaltimer();
        for (int64_t u = unit; u < units; u += nunits, ++lt) {
            const wide::Unit w = wide::unit_of(u, full);
            const TileCoord c = tile_coord(a, w.t, tiles_m, tiles_n);
            const bool got = role_wait(ptx::smem_addr(&sh.tmem_full[0]), (uint32_t)(lt & 1),
                                       a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (half < w.h0 || half >= w.h0 + w.nh) {
                // a half tile without this warp's columns: nothing to copy
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(map_to_rank(ptx::smem_addr(&sh.tmem_empty[0]), 0));
                continue;
            }
            const uint64_t t_ready = ptx::globaltimer();
            uint64_t period = t_ready - prev_ready;
            period = period > kPaceMaxPeriodNs ? kPaceMaxPeriodNs : period;
            prev_ready = t_ready;
            const uint64_t slot =
                u + nunits < units ? period * kPacePct / 100u / (uint64_t)(kBoxes * a.W) : 0;
            // the whole accumulator slice of this warp, as packed 16-bit pairs
            // (16 columns per load keeps it within the registers, no spills)
            uint32_t pk[kBoxes * 32];
#pragma unroll
            for (int ch = 0; ch < 4 * kBoxes; ++ch) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(t_lane + (uint32_t)(ch * 16), v);
                tmem_wait_ld16(v);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    pk[ch * 8 + i] = pack2(v[2 * i], v[2 * i + 1], a.is_bf16);
            }
            // accumulator copied out: hand TMEM back to the leader's MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(map_to_rank(ptx::smem_addr(&sh.tmem_empty[0]), 0));
            const int row0 = c.tm * wide::kTileM + (int)rank * BM + q * 32;
#pragma unroll
            for (int b = 0; b < kBoxes; ++b) {
                // the box is free once this warp's previous stores have read it
                ptx::bulk_wait_read<0>();
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k)  // 16-byte chunk k at position k ^ (row mod 8)
                    st_shared_v4(my_row + ((((uint32_t)k) ^ swz) << 4), pk[b * 32 + 4 * k],
                                 pk[b * 32 + 4 * k + 1], pk[b * 32 + 4 * k + 2],
                                 pk[b * 32 + 4 * k + 3]);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                const int col = c.tn * wide::kTileN + half * BN + b * 64;
                if (row0 < a.M && col < a.N) {
                    if (slot != 0) {
                        for (int j = 0; j < a.W; ++j) {
                            const uint64_t due = t_ready + slot * (uint64_t)(b * a.W + j);
                            while (ptx::globaltimer() < due && !*abort_flag)
                                __nanosleep(256);
                            if (lane == 0) {
                                int i = c.g + j;
                                if (i >= a.W)
                                    i -= a.W;
                                tma_store_3d(&out.map[i], staging, col, row0, c.g, pol_c);
                            }
                        }
                    } else {
                        for (int j = lane; j < a.W; j += 32) {
                            int i = c.g + j;
                            if (i >= a.W)
                                i -= a.W;
                            tma_store_3d(&out.map[i], staging, col, row0, c.g, pol_c);
                        }
                    }
                }
                ptx::bulk_commit();
            }
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        ptx::bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the leader's MMAs into the peer's TMEM and smem are done
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<2>(tmem);
    }
    trace_mark(a.trace, 1);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(wide::kThreads, 1)
    mag2w_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const __grid_constant__ OutMaps out, const FusedArgs a)
{
    magw_body(map_a, map_b, out, a);
}

}  // namespace

cudaError_t launch_matmul_all_gather(const FusedArgs &a, const OutMaps &out, int programs,
                                     int variant, cudaStream_t s, const char **why)
{
    if (!tensor_maps_available()) {
        *why = "cuTensorMapEncodeTiled is not available";
        return cudaErrorNotSupported;
    }
    const CUtensorMapDataType dt =
        a.is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap map_a, map_b;
    {
        // A as {K, M, heaps}: one partition per heap (group launch) or the one block
        const bool group = a.a_abs == nullptr;
        const void *ga = group ? reinterpret_cast<const void *>(a.heap_base + (uint64_t)a.a_off)
                               : a.a_abs;
        const uint64_t dims[3] = {(uint64_t)a.K, (uint64_t)a.M,
                                  (uint64_t)(group ? a.num_heaps : 1)};
        const uint64_t strides[2] = {(uint64_t)a.lda * 2,
                                     group ? a.part_bytes : (uint64_t)(a.M * a.lda * 2)};
        const uint32_t box[3] = {kKAtom, BM, 1};
        if (!encode_map(&map_a, dt, 3, ga, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
            *why = "encoding the tensor map of A";
            return cudaErrorInvalidValue;
        }
    }
    const bool two_sm = fused_variant(programs, variant) == 2;
    const bool wide_tiles = two_sm && a.wide;  // 256 x 512 pair tiles
    const int bk = two_sm ? Geo<2>::kBK : Geo<1>::kBK;  // K rows of one B box
    FusedArgs args = a;
    args.b_boxes3d = 0;
    {
        // column groups whose B slice (K x the tile's columns each) fits in
        // kBGroupBytes, as equal as possible
        const int64_t tile_n = wide_tiles ? wide::kTileN : BN;
        const int64_t tn = a.N > tile_n ? (a.N + tile_n - 1) / tile_n : 1;
        const int64_t per_col = a.K * tile_n * 2;
        int64_t w = (wide_tiles ? kBGroupBytesWide : kBGroupBytes) / (per_col > 0 ? per_col : 1);
        w = w < 1 ? 1 : (w > tn ? tn : w);
        const int64_t groups = (tn + w - 1) / w;
        args.tn_group = (int)((tn + groups - 1) / groups);
    }
    if (kBBoxes3d && a.N % 64 == 0) {
        // {64 columns, K, N/64 column chunks}: one copy per stage brings all the
        // CTA's 64-column boxes (only when N is whole chunks, so no box reads
        // past the end of a row of B)
        const uint64_t dims[3] = {64, (uint64_t)a.K, (uint64_t)(a.N / 64)};
        const uint64_t strides[2] = {(uint64_t)a.ldb * 2, 128};
        const uint32_t box[3] = {64, (uint32_t)bk,
                                 (uint32_t)(two_sm ? Geo<2>::kBCols / 64 : Geo<1>::kBCols / 64)};
        args.b_boxes3d =
            encode_map(&map_b, dt, 3, a.b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ? 1 : 0;
    }
    if (!args.b_boxes3d) {
        const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.K};
        const uint64_t strides[1] = {(uint64_t)a.ldb * 2};
        const uint32_t box[2] = {64, (uint32_t)bk};
        if (!encode_map(&map_b, dt, 2, a.b, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) {
            *why = "encoding the tensor map of B";
            return cudaErrorInvalidValue;
        }
    }
    const int64_t tiles_n = (a.N + BN - 1) / BN;
    cudaError_t e;
    if (wide_tiles) {
        const int64_t pairs = (int64_t)a.n_src * ((a.M + wide::kTileM - 1) / wide::kTileM) *
                              ((a.N + wide::kTileN - 1) / wide::kTileN);
        e = cudaFuncSetAttribute(mag2w_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 wide::kSmemBytes);
        if (e != cudaSuccess) {
            *why = "setting the shared-memory size of the fused kernel";
            return e;
        }
        static int resident_by_dev[64];
        static std::once_flag once_by_dev[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            dev = 0;
        std::call_once(once_by_dev[dev], [&] {
            int resident = 0;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(wide::kThreads, 1, 1);
            cfg.dynamicSmemBytes = wide::kSmemBytes;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&resident, mag2w_kernel, &cfg) != cudaSuccess)
                resident = 0;
            (void)cudaGetLastError();
            resident_by_dev[dev] = resident;
        });
        const int resident = resident_by_dev[dev];
        int64_t clusters = gg_min64(programs / 2, pairs);
        if (resident > 0)
            clusters = gg_min64(clusters, resident);
        mag2w_kernel<<<(int)(2 * clusters), wide::kThreads, wide::kSmemBytes, s>>>(map_a, map_b,
                                                                                 out, args);
    } else if (two_sm) {
        const int64_t pairs = (int64_t)a.n_src * ((a.M + 2 * BM - 1) / (2 * BM)) * tiles_n;
        e = cudaFuncSetAttribute(mag2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes<2>());
        if (e != cudaSuccess) {
            *why = "setting the shared-memory size of the fused kernel";
            return e;
        }
        // persistent pairs: never more clusters than can be resident at once
        // (queried once per device; later calls, e.g. under stream capture,
        // reuse the answer)
        static int resident_by_dev[64];
        static std::once_flag once_by_dev[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            dev = 0;
        std::call_once(once_by_dev[dev], [&] {
            int resident = 0;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = smem_bytes<2>();
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&resident, mag2_kernel, &cfg) != cudaSuccess)
                resident = 0;
            (void)cudaGetLastError();
            resident_by_dev[dev] = resident;
        });
        const int resident = resident_by_dev[dev];
        int64_t clusters = gg_min64(programs / 2, pairs);
        if (resident > 0)
            clusters = gg_min64(clusters, resident);
        mag2_kernel<<<(int)(2 * clusters), kThreads, smem_bytes<2>(), s>>>(map_a, map_b, out, args);
    } else {
        const int64_t tiles = (int64_t)a.n_src * ((a.M + BM - 1) / BM) * tiles_n;
        e = cudaFuncSetAttribute(mag1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes<1>());
        if (e != cudaSuccess) {
            *why = "setting the shared-memory size of the fused kernel";
            return e;
        }
        mag1_kernel<<<(int)gg_min64(programs, tiles), kThreads, smem_bytes<1>(), s>>>(map_a, map_b,
                                                                                    out, args);
    }
    return cudaGetLastError();
}

}  // namespace gg
