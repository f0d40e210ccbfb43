// Fused matmul + all-gather for sm_103a (iris PR #626, "Summary" and
// "Benchmark": the matmul's epilogue all-gathers each output tile, with the
// heap-base translation hoisted above the K loop).
//
// C_r = A_r @ B for every source r of the launch, each 128 x 256 output tile:
//   * warp 0 (producer): TMA tensor loads of A (128 x 64, K-major) and B
//     (64 x 256, N-major, as four 64-column boxes) into a 3-stage ring of
//     128B-swizzled shared memory, completion on mbarriers;
//   * warp 1 (MMA): allocates 512 TMEM columns (two 128 x 256 fp32
//     accumulators) and issues tcgen05.mma kind::f16 (M=128, N=256, K=16)
//     from one thread; tcgen05.commit frees ring stages and hands finished
//     accumulators to the epilogue;
//   * warps 2-5 (epilogue): tcgen05.ld of their 32 TMEM lanes (= tile rows),
//     round to f16/bf16, write each row once into a padded shared-memory
//     staging row, then one bulk copy (cp.async.bulk shared->global) per row
//     and destination: the local copy first, then the peers in rotated order.
//     The accumulator is released right after it has been read, so the next
//     tile's MMAs overlap this tile's stores.
// The W destination bases come from the heap-bases table, loaded once per CTA
// before any tile (the hoisted translation).
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

constexpr int BM = 128, BN = 256, BK = 64, UK = 16;
constexpr int kStages = 3;
constexpr int kAStage = BM * BK * 2;            // 16 KB
constexpr int kBBox = BK * 64 * 2;              // 8 KB: 64 K-rows x 64 N-columns
constexpr int kBStage = BK * BN * 2;            // 32 KB
constexpr int kEpiPitch = BN * 2 + 16;          // staged row pitch (bytes), bank-conflict free
constexpr int kEpiWarp = 32 * kEpiPitch;        // one epilogue warp's 32 rows
constexpr int kThreads = 192;                   // 6 warps
constexpr int kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 1000000000ull;

struct FusedShared {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint64_t dst[kMaxWorld];
    uint32_t tmem_base;
    int abort_flag;
};

constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAStage;
constexpr int kOffEpi = kOffB + kStages * kBStage;
constexpr int kOffShared = kOffEpi + 4 * kEpiWarp;
constexpr int kSmemBytes = kOffShared + (int)sizeof(FusedShared) + 1024;  // + alignment slack

// ---- tcgen05 / TMA wrappers ---------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::"
        "cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

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
// A K-major, B N-major, N = 256, M = 128.
__host__ __device__ constexpr uint32_t instr_desc(int bf16)
{
    return (1u << 4)                      // D format: f32
           | ((uint32_t)bf16 << 7)        // A format
           | ((uint32_t)bf16 << 10)       // B format
           | (0u << 15)                   // A major: K
           | (1u << 16)                   // B major: MN
           | ((uint32_t)(BN >> 3) << 17)  // N >> 3
           | ((uint32_t)(BM >> 4) << 24); // M >> 4
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

struct TileCoord {
    int g;        // group index of the source
    int h;        // heap index of the source
    int tm, tn;
};

__device__ __forceinline__ TileCoord tile_coord(const FusedArgs &a, int64_t t, int tiles_m,
                                                int tiles_n)
{
    TileCoord c;
    const int64_t per_src = (int64_t)tiles_m * tiles_n;
    const int s = (int)(t / per_src);
    const int64_t rem = t - (int64_t)s * per_src;
    c.g = a.src_first + s;
    c.h = a.rank_start + c.g * a.rank_stride;
    c.tm = (int)(rem / tiles_n);
    c.tn = (int)(rem - (int64_t)c.tm * tiles_n);
    return c;
}

__global__ void __launch_bounds__(kThreads, 1)
    mag_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const FusedArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned for the 128B swizzle
    uint8_t *smem = smem_raw + (base - raw);
    FusedShared &sh = *reinterpret_cast<FusedShared *>(smem + kOffShared);
    volatile int *abort_flag = &sh.abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (int)((a.M + BM - 1) / BM);
    const int tiles_n = (int)((a.N + BN - 1) / BN);
    const int64_t total = (int64_t)a.n_src * tiles_m * tiles_n;
    const int num_kb = (int)((a.K + BK - 1) / BK);

    // ---- prologue: barriers, TMEM, destination bases (loaded once) ----------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sh.full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sh.tmem_full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh.tmem_empty[s]), 4);
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
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         ptx::smem_addr(&sh.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    for (int i = threadIdx.x; i < a.W; i += blockDim.x)
        sh.dst[i] = a.bases[a.rank_start + i * a.rank_stride] + (uint64_t)a.out_off;
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ===================== producer =====================================
        const uint64_t pol_a = ptx::policy_evict_normal();  // A tile: read by tiles_n CTAs
        const uint64_t pol_b = ptx::policy_evict_last();    // B: read by every tile row
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileCoord c = tile_coord(a, t, tiles_m, tiles_n);
            const int h_coord = a.a_abs ? 0 : c.h;
            for (int kb = 0; kb < num_kb; ++kb) {
                const bool got = role_wait(ptx::smem_addr(&sh.empty[stage]), phase ^ 1u,
                                           a.wait_limit_ns, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const bool stall = a.inject_stall && blockIdx.x == 0 && issued == 0;
                if (lane == 0 && !stall) {  // test hook: the first stage is never armed
                    const uint32_t bar = ptx::smem_addr(&sh.full[stage]);
                    ptx::mbar_arrive_expect_tx(bar, kAStage + kBStage);
                    const uint32_t sa = base + kOffA + stage * kAStage;
                    const uint32_t sb = base + kOffB + stage * kBStage;
                    tma_load_3d(sa, &map_a, kb * BK, c.tm * BM, h_coord, bar, pol_a);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sb + j * kBBox, &map_b, c.tn * BN + j * 64, kb * BK, bar, pol_b);
                }
                __syncwarp();
                ++issued;
                if (++stage == kStages) {
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
        const int64_t pending = issued < kStages ? issued : kStages;
        for (int64_t q = 0; q < pending; ++q) {
            // the q-th most recent k-block issued
            const int64_t idx = issued - 1 - q;
            const int s = (int)(idx % kStages);
            const uint32_t ph = (uint32_t)((idx / kStages) & 1);
            ptx::mbar_wait(ptx::smem_addr(&sh.full[s]), ph, kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ===================== MMA issuer ===================================
        const uint32_t idesc = instr_desc(a.is_bf16);
        int stage = 0;
        uint32_t phase = 0;
        int64_t lt = 0;  // local tile count
        bool issued_any = false;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x, ++lt) {
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
                    const uint32_t sa = base + kOffA + stage * kAStage;
                    const uint32_t sb = base + kOffB + stage * kBStage;
#pragma unroll
                    for (int k = 0; k < BK / UK; ++k) {
                        // A: K-major, +32 bytes per 16-element K step; SBO = 8 rows x 128 B
                        const uint64_t ad = smem_desc(sa + k * (UK * 2), 16, 1024);
                        // B: N-major, +16 K-rows x 128 B per K step; LBO = next 64-column
                        // box, SBO = 8 K-rows x 128 B
                        const uint64_t bd = smem_desc(sb + k * (UK * 128), kBBox, 1024);
                        mma_f16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(ptx::smem_addr(&sh.empty[stage]));
                }
                __syncwarp();
                issued_any = true;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                break;
            if (lane == 0)
                mma_commit(ptx::smem_addr(&sh.tmem_full[acc]));
            __syncwarp();
        }
        if (!ok) {
            *abort_flag = 1;
            report_status(a.status, kStatusTimeout);
        }
        // drain: all MMAs of this thread have completed before TMEM is freed
        if (issued_any) {
            if (lane == 0)
                mma_commit(ptx::smem_addr(&sh.mma_done));
            __syncwarp();
            ptx::mbar_wait(ptx::smem_addr(&sh.mma_done), 0, kDrainLimitNs);
        }
    } else {
        // ===================== epilogue (warps 2-5) =========================
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t stage_row = base + kOffEpi + (uint32_t)(q * kEpiWarp + lane * kEpiPitch);
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        const int64_t ld_out_b = a.ld_out * 2;
        const uint64_t pol_c = ptx::policy_evict_first();  // output: written once, never read
        int64_t lt = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
            const TileCoord c = tile_coord(a, t, tiles_m, tiles_n);
            const int acc = (int)(lt & 1);
            const uint32_t acc_phase = (uint32_t)((lt >> 1) & 1);
            const bool got = role_wait(ptx::smem_addr(&sh.tmem_full[acc]), acc_phase,
                                       a.wait_limit_ns, abort_flag);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // this warp's staging rows are free once its previous stores have read them
            ptx::bulk_wait_read<0>();
            __syncwarp();
            const uint32_t t_addr = tmem + lane_addr + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int cb = 0; cb < BN; cb += 64) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(t_addr + (uint32_t)cb, v0);
                tmem_ld_32x32b_x32(t_addr + (uint32_t)(cb + 32), v1);
                tmem_wait_ld(v0);
                reg_order(v1);
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    st_shared_v4(stage_row + (uint32_t)(cb * 2 + j * 2), pack2(v0[j], v0[j + 1], a.is_bf16),
                                 pack2(v0[j + 2], v0[j + 3], a.is_bf16),
                                 pack2(v0[j + 4], v0[j + 5], a.is_bf16),
                                 pack2(v0[j + 6], v0[j + 7], a.is_bf16));
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    st_shared_v4(stage_row + (uint32_t)((cb + 32) * 2 + j * 2),
                                 pack2(v1[j], v1[j + 1], a.is_bf16),
                                 pack2(v1[j + 2], v1[j + 3], a.is_bf16),
                                 pack2(v1[j + 4], v1[j + 5], a.is_bf16),
                                 pack2(v1[j + 6], v1[j + 7], a.is_bf16));
            }
            // accumulator fully read: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(ptx::smem_addr(&sh.tmem_empty[acc]));
            // staged rows -> every destination, local first, peers rotated
            ptx::fence_proxy_async_smem();
            __syncwarp();
            const int64_t row = (int64_t)c.tm * BM + q * 32 + lane;
            const int64_t col0 = (int64_t)c.tn * BN;
            if (row < a.M) {
                const uint32_t rb = (uint32_t)(gg_min64(BN, a.N - col0) * 2);
                const int64_t off = ((int64_t)c.g * a.M + row) * ld_out_b + col0 * 2;
                for (int j = 0; j < a.W; ++j) {
                    int i = c.g + j;
                    if (i >= a.W)
                        i -= a.W;
                    ptx::bulk_s2g_hint(reinterpret_cast<uint8_t *>(sh.dst[i]) + off, stage_row, rb,
                                       pol_c);
                }
            }
            ptx::bulk_commit();
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
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---- host: tensor maps and launch ------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

cudaError_t launch_matmul_all_gather(const FusedArgs &a, int programs, cudaStream_t s,
                                     const char **why)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        *why = "cuTensorMapEncodeTiled is not available";
        return cudaErrorNotSupported;
    }
    const CUtensorMapDataType dt =
        a.is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap map_a, map_b;
    {
        // A as {K, M, heaps}: one partition per heap (group launch) or the one block
        const bool group = a.a_abs == nullptr;
        void *ga = group ? reinterpret_cast<void *>(a.heap_base + (uint64_t)a.a_off)
                         : const_cast<void *>(a.a_abs);
        const cuuint64_t dims[3] = {(cuuint64_t)a.K, (cuuint64_t)a.M,
                                    (cuuint64_t)(group ? a.num_heaps : 1)};
        const cuuint64_t strides[2] = {(cuuint64_t)a.lda * 2,
                                       group ? (cuuint64_t)a.part_bytes
                                             : (cuuint64_t)(a.M * a.lda * 2)};
        const cuuint32_t box[3] = {BK, BM, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&map_a, dt, 3, ga, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *why = "encoding the tensor map of A";
            return cudaErrorInvalidValue;
        }
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.K};
        const cuuint64_t strides[1] = {(cuuint64_t)a.ldb * 2};
        const cuuint32_t box[2] = {64, BK};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&map_b, dt, 2, const_cast<void *>(a.b), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS) {
            *why = "encoding the tensor map of B";
            return cudaErrorInvalidValue;
        }
    }
    cudaError_t e =
        cudaFuncSetAttribute(mag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) {
        *why = "setting the shared-memory size of the fused kernel";
        return e;
    }
    const int64_t tiles = (int64_t)a.n_src * ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    const int grid = (int)(programs < tiles ? programs : tiles);
    mag_kernel<<<grid, kThreads, kSmemBytes, s>>>(map_a, map_b, a);
    return cudaGetLastError();
}

}  // namespace gg
