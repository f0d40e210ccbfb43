// Persistent tiled all-gather over a symmetric heap (sm_103a).
//
// What it computes (iris #594 "Multi-GPU CI", iris PR #626 "Summary"):
// every source block (one group member's M x N input) is written into its row
// block of the gathered output of every group member.  How (iris PR #626
// "Summary" and "Triton CCL all-gather"; iris #591 Description §1):
//  * the heap-bases table is read once per program, before the tile loop, and
//    turned into one output base per member (the hoisted per-peer translation;
//    no base is reloaded inside the loop);
//  * each tile is read from HBM once and staged on chip;
//  * the staged tile is stored to the local copy first, then to the peers in
//    rotated order (i+1, i+2, ... mod W), with no fence or reload between
//    destinations.
//
// Three data paths with identical results:
//  * tma:    one TMA tensor load per tile into shared memory (mbarrier
//            completion) and one TMA tensor store per tile and destination,
//            through per-member tensor maps built on the host from the
//            heap-bases table once per launch (the translation hoisted out of
//            every loop; each map views a member's output as {N, M, W} so a
//            tile is clipped at the end of its row block).  Same pipeline as
//            the bulk path; on large launches the tiles are handed out in
//            runs claimed from a workspace counter (load balancing, see Feed).
//  * bulk:   tiles are staged in shared memory by the TMA engine
//            (cp.async.bulk, completion on an mbarrier) and stored with
//            cp.async.bulk shared->global, one copy per tile row and
//            destination.  Each warp of a program runs an independent
//            pipeline over a ring of stages (the warps per program follow the
//            budget, see kAgTargetPipes); a stage is refilled once the stores
//            that read it have finished reading shared memory.
//  * vector: 16/8/4/2-byte loads into registers, then one store per
//            destination; several tiles' loads are in flight per thread.
//
// The same kernels run the two neighbouring collectives of the pages:
//  * partitioned all-gather (iris PR #626, "Triton CCL all-gather":
//    persistent_all_gather_partitioned): programs are split across the
//    destinations; program p serves destination p mod W only, so each tile is
//    read once per destination (tensor-map and vector paths);
//  * all-to-all (iris #594 "Compiler inspection and grouping", iris #591
//    Work): member i's input holds W row blocks; block d goes to row block i
//    of member d's output, one store per tile (tensor-map and vector paths).
// and the destination grouping of iris #594 "Compiler inspection and
// grouping" / iris #591 Description §2: with dests_per_wait = G the stores of
// a tile go out G destinations at a time, each group waiting until the
// previous ones have read shared memory (bulk and tensor-map paths).
#include <cuda_runtime.h>

#include <atomic>

#include "gg_internal.h"
#include "ptx.cuh"

namespace gg {
namespace {

constexpr int kAgWarps = 8;           // most independent pipelines (warps) per program
// Pipelines the whole launch aims for: each program runs about
// kAgTargetPipes / programs of them (1..kAgWarps), so a small budget still
// keeps enough copies in flight and a large one does not oversubscribe.
constexpr int kAgTargetPipes = 512;
// The partitioned gather and the all-to-all store each tile once (not W
// times), so a pipeline moves W times fewer bytes per load: they aim higher.
constexpr int kAgTargetPipesSingle = 2048;
constexpr int kAgMaxStages = 16;      // ring stages per pipeline
constexpr int kAgSmemBudget = 192 * 1024;
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // waits for copies already in flight

struct Item {
    int g;          // group index of the source
    int d;          // group index of the destination block (all-to-all), else -1
    int64_t tm, tn; // tile coordinates
    int rows;       // valid rows of the tile
    uint32_t rb;    // valid bytes per tile row
};

struct AgShared {
    uint64_t full[kAgWarps][kAgMaxStages];  // one mbarrier per ring stage
    Item item[kAgWarps][kAgMaxStages];      // the tile a ring stage holds (decoded at issue)
    uint64_t dst[kMaxWorld];                // output base of member i
    uint64_t src[kMaxWorld];                // input base of member i
};

constexpr int kAgHeader = (int)((sizeof(AgShared) + 127) / 128 * 128);

// Checked build (compiled with GG_CHECKED=1 into libgemm_gather_checked.so):
// device-side checks of the heap-bases table, of every decoded work item and
// of every raw address the bulk and vector paths form.  A failed check skips
// the access and stores GG_ERR_NOT_IN_HEAP in the status word.  The release
// build compiles every check out (kChecked is a constant).
#ifndef GG_CHECKED
#define GG_CHECKED 0
#endif
constexpr bool kChecked = GG_CHECKED != 0;

// [p, p + n) lies inside [lo, lo + ext).
__device__ __forceinline__ bool inside(uint64_t lo, int64_t ext, uint64_t p, uint64_t n)
{
    return p >= lo && p - lo <= (uint64_t)ext && n <= (uint64_t)ext - (p - lo);
}

__device__ __noinline__ void bounds_fault(int *status)
{
    report_status(status, kStatusNotInHeap);
}

// The validated output (and heap input) extents at their offsets fit inside
// one partition.  Uniform over the launch: a kernel that finds otherwise
// returns before its first access.
__device__ __forceinline__ bool extents_ok(const GatherArgs &a)
{
    return a.out_ext_b > 0 && (uint64_t)a.out_off + (uint64_t)a.out_ext_b <= a.part_bytes &&
           a.in_ext_b > 0 &&
           (a.in_abs != nullptr || (uint64_t)a.in_off + (uint64_t)a.in_ext_b <= a.part_bytes);
}

// The items a vector-path program walks (the whole program is one pipeline):
// first, first + step, ... and, for the partitioned all-gather, the one
// destination it serves.  The ring kernels walk a Feed instead.
struct Walk {
    int64_t first, step, n;
    int dest;
};

__device__ __forceinline__ Walk make_walk(const GatherArgs &a, int warp, int npipe)
{
    int64_t prog = blockIdx.x, nprog = gridDim.x;
    int dest = -1;
    if (a.mode == kModePartitioned) {  // program p serves destination p mod W
        dest = (int)(blockIdx.x % (unsigned)a.W);
        prog = blockIdx.x / (unsigned)a.W;
        nprog = (gridDim.x - 1 - dest) / a.W + 1;
    }
    Walk w;
    w.first = prog + (int64_t)warp * nprog;
    w.step = nprog * npipe;
    w.n = w.first < a.total_items ? (a.total_items - 1 - w.first) / w.step + 1 : 0;
    w.dest = dest;
    return w;
}

// The items one ring pipeline (warp) loads, in order.  With P pipelines
// (of one destination for the partitioned all-gather), items are handed
// out in runs: run n covers items b, b + P, b + 2P, ... (`chunk` of them, up to
// the last item), where b = (n / P) * P * chunk + n % P.  Pipelines working
// side by side therefore touch neighbouring tiles, as with fixed shares.
//  * fixed shares (no counter): pipeline p takes run p, with no length limit:
//    items p, p + P, p + 2P, ...;
//  * claimed runs (counter): pipeline p takes run p (`chunk` items), then
//    claims run P + (counter++) each time its run is done.  Programs on SMs
//    that move data faster claim more runs, so all programs finish together
//    whatever share of the memory system their SMs get.  Lane 0 keeps two
//    claims in flight (q0, q1) so that a claim's latency hides behind the
//    items before it.
struct Feed {
    int64_t cur;                // next item of the current run
    int64_t left;               // items left in the current run
    int64_t pipes, total;
    unsigned long long *ctr;    // claimed runs: the counter; null: fixed shares
    unsigned long long q0, q1;  // lane 0: the two claims in flight
    int chunk;
    int phase;                  // which claim is the older one
    bool dry;                   // no item left
};

__device__ __forceinline__ Feed make_feed(const GatherArgs &a, int warp, int npipe, int lane,
                                          int *dest)
{
    int64_t prog = blockIdx.x, nprog = gridDim.x;
    int d = -1;
    unsigned long long *ctr = a.work;
    if (a.mode == kModePartitioned) {  // program p serves destination p mod W
        d = (int)(blockIdx.x % (unsigned)a.W);
        prog = blockIdx.x / (unsigned)a.W;
        nprog = (gridDim.x - 1 - d) / a.W + 1;
        ctr = nullptr;  // fixed shares (claims do not pay off here)
    }
    *dest = d;
    Feed f;
    f.pipes = nprog * npipe;
    f.cur = prog + (int64_t)warp * nprog;
    f.total = a.total_items;
    f.ctr = ctr;
    f.chunk = a.chunk;
    f.left = ctr ? a.chunk : a.total_items;
    f.phase = 0;
    f.dry = false;
    f.q0 = f.q1 = 0;
    if (ctr && lane == 0 && f.pipes * a.chunk < a.total_items) {
        f.q0 = atomicAdd(ctr, 1ull);
        f.q1 = atomicAdd(ctr, 1ull);
    }
    return f;
}

// Next item of the pipeline, or -1.  Warp-uniform: every lane calls it.
__device__ __forceinline__ int64_t feed_next(Feed &f, int lane)
{
    if (f.dry)
        return -1;
    if (f.left == 0 || f.cur >= f.total) {
        if (!f.ctr || f.pipes * f.chunk >= f.total) {
            f.dry = true;
            return -1;
        }
        // take the older claim, put a new one in its place (each branch
        // touches one claim register, so the newer claim is not waited for)
        unsigned long long c;
        if (f.phase == 0)
            c = __shfl_sync(0xffffffffu, f.q0, 0);
        else
            c = __shfl_sync(0xffffffffu, f.q1, 0);
        const int64_t n = f.pipes + (int64_t)c;
        const int64_t b = n / f.pipes * f.pipes * f.chunk + n % f.pipes;
        // b grows with n: once past the end, every later claim is too
        if (b >= f.total) {
            f.dry = true;
            return -1;
        }
        if (lane == 0) {
            if (f.phase == 0)
                f.q0 = atomicAdd(f.ctr, 1ull);
            else
                f.q1 = atomicAdd(f.ctr, 1ull);
        }
        f.phase ^= 1;
        f.cur = b;
        f.left = f.chunk;
    }
    const int64_t t = f.cur;
    f.cur += f.pipes;
    --f.left;
    return t;
}

// Item t: source-major; for the all-to-all each source's items run over its W
// destination blocks in rotated order (its own block first), then tiles.
__device__ __forceinline__ Item decode_item(const GatherArgs &a, int64_t t)
{
    Item it;
    const int64_t per_src = a.mode == kModeAllToAll ? a.tiles_per_src * a.W : a.tiles_per_src;
    const int64_t s = t / per_src;
    int64_t tile = t - s * per_src;
    it.g = a.src_first + (int)s;
    it.d = -1;
    if (a.mode == kModeAllToAll) {
        const int jr = (int)(tile / a.tiles_per_src);
        tile -= (int64_t)jr * a.tiles_per_src;
        int d = it.g + jr;
        if (d >= a.W)
            d -= a.W;
        it.d = d;
    }
    it.tm = tile / a.tiles_n;
    it.tn = tile - it.tm * a.tiles_n;
    const int64_t r0 = it.tm * a.bm;
    it.rows = (int)gg_min64(a.bm, a.M - r0);
    const int64_t c0 = it.tn * a.bn_b;
    it.rb = (uint32_t)gg_min64(a.bn_b, a.row_b - c0);
    if (kChecked && !(t >= 0 && t < a.total_items && it.g >= 0 && it.g < a.W && it.d >= -1 &&
                      it.d < a.W && it.tm >= 0 && r0 < a.M && it.tn >= 0 && c0 < a.row_b)) {
        bounds_fault(a.status);  // an item outside the tile grid: nothing of it is moved
        it.g = 0;
        it.d = it.d < 0 ? -1 : 0;
        it.tm = it.tn = 0;
        it.rows = 0;
        it.rb = 0;
    }
    return it;
}

__device__ __forceinline__ void tma_prefetch(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                             int c2, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
        "[%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_box4(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                              int c2, int c3, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
        "[%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_box(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                              int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// The same store with an L2 eviction-priority hint (gg_set_store_policy).
__device__ __forceinline__ void tma_store_box_hint(const CUtensorMap *map, uint32_t src, int c0,
                                                   int c1, int c2, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%2, %3, %4}], [%1], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

// Heap bases -> per-member input and output bases, once per program.
__device__ __forceinline__ void load_member_bases(const GatherArgs &a, uint64_t *dst,
                                                  uint64_t *src)
{
    for (int i = threadIdx.x; i < a.W; i += blockDim.x) {
        const int h = a.rank_start + i * a.rank_stride;
        uint64_t base = a.bases[h];
        if (kChecked && base != a.heap_lo + (uint64_t)h * a.part_bytes) {
            // the entry disagrees with the heap layout: reported, and not used
            bounds_fault(a.status);
            base = a.heap_lo + (uint64_t)h * a.part_bytes;
        }
        dst[i] = base + (uint64_t)a.out_off;
        src[i] = a.in_abs ? reinterpret_cast<uint64_t>(a.in_abs) : base + (uint64_t)a.in_off;
    }
}

// D: store groups a pipeline may leave reading shared memory before it
// refills the oldest stage; the loads run stages - D items ahead.
template <int D>
__global__ void __launch_bounds__(kAgWarps * 32, 1)
    ag_bulk_kernel(const GatherArgs a, int stages, int stage_bytes)
{
    const int npipe = blockDim.x >> 5;
    extern __shared__ __align__(1024) uint8_t smem[];
    AgShared &sh = *reinterpret_cast<AgShared *>(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    trace_mark(a.trace, 0);
    if (kChecked && !extents_ok(a)) {
        if (threadIdx.x == 0)
            bounds_fault(a.status);
        return;
    }

    load_member_bases(a, sh.dst, sh.src);
    if (threadIdx.x == 0) {
        for (int w = 0; w < npipe; ++w)
            for (int s = 0; s < stages; ++s)
                ptx::mbar_init(ptx::smem_addr(&sh.full[w][s]), 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();

    int dest;
    Feed feed = make_feed(a, warp, npipe, lane, &dest);
    const int lookahead = stages - D;  // loads in flight ahead of the stores

    const uint32_t ring = ptx::smem_addr(smem + kAgHeader) + (uint32_t)(warp * stages * stage_bytes);
    const uint32_t full0 = ptx::smem_addr(&sh.full[warp][0]);
    const uint32_t pitch = (uint32_t)a.bn_b;  // staged row pitch (multiple of 16)
    const uint64_t pol_st = a.store_hint ? ptx::policy_evict_first() : 0;
    const int grp = (a.dests_per_wait > 0 && a.dests_per_wait < a.W) ? a.dests_per_wait : a.W;

    // Takes the pipeline's next item (if any) and starts its load into ring
    // slot `issued`.
    int64_t issued = 0;
    auto issue_next = [&]() {
        const int64_t t = feed_next(feed, lane);
        if (t < 0)
            return;
        if (issued >= stages) {
            // the stage last held item issued - stages = (issued - lookahead) - D
            ptx::bulk_wait_read<D>();
            __syncwarp();
        }
        Item it = decode_item(a, t);
        const int st = (int)(issued % stages);
        const uint32_t bar = full0 + 8u * st;
        const uint32_t buf = ring + (uint32_t)st * stage_bytes;
        bool load_ok = true;
        if (kChecked) {
            // the item's rows of its source block, as the loads below address them
            const uint64_t first = sh.src[it.g] + (uint64_t)(it.tm * a.bm * a.ld_in_b + it.tn * a.bn_b);
            const uint64_t span = it.rows > 0 ? (uint64_t)(it.rows - 1) * a.ld_in_b + it.rb : 0;
            load_ok = it.rows > 0 && inside(sh.src[it.g], a.in_ext_b, first, span);
            // (rows == 0: an item outside the grid, already reported at decode)
            if (!load_ok) {
                if (lane == 0 && it.rows > 0)
                    bounds_fault(a.status);
                it.rows = 0;  // nothing loaded, nothing stored
            }
        }
        if (lane == 0)
            sh.item[warp][st] = it;
        const bool stall = a.inject_stall && issued == 0 && blockIdx.x == 0 && warp == 0;
        ++issued;
        if (stall)
            return;  // test hook: this stage's barrier phase never completes
        if (kChecked && !load_ok) {
            if (lane == 0)
                ptx::mbar_arrive(bar);  // completes the stage's phase with no bytes
            __syncwarp();
            return;
        }
        if (lane == 0)
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)it.rows * it.rb);
        __syncwarp();
        const uint8_t *src = reinterpret_cast<const uint8_t *>(sh.src[it.g]) +
                             it.tm * a.bm * a.ld_in_b + it.tn * a.bn_b;
        for (int r = lane; r < it.rows; r += 32)
            ptx::bulk_g2s(buf + (uint32_t)r * pitch, src + r * a.ld_in_b, it.rb, bar);
    };

    for (int q = 0; q < lookahead; ++q)
        issue_next();

    int64_t k = 0;
    bool ok = true;
    for (; k < issued; ++k) {
        const int st = (int)(k % stages);
        const uint32_t parity = (uint32_t)((k / stages) & 1);
        const bool mine = ptx::mbar_wait(full0 + 8u * st, parity, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, mine)) {
            ok = false;
            break;
        }
        const Item it = sh.item[warp][st];
        const uint32_t buf = ring + (uint32_t)st * stage_bytes;
        const int64_t row0 = (int64_t)it.g * a.M + it.tm * a.bm;
        const int64_t col0 = it.tn * a.bn_b;
        // destinations go out `grp` at a time (all at once unless grouped);
        // pair p of a group -> destination j0 + p / rows (j = 0 is the local
        // copy), row p % rows
        for (int j0 = 0; j0 < a.W; j0 += grp) {
            const int nj = a.W - j0 < grp ? a.W - j0 : grp;
            for (int p = lane; p < nj * it.rows; p += 32) {
                const int jj = p / it.rows;
                const int r = p - jj * it.rows;
                int i = it.g + j0 + jj;
                if (i >= a.W)
                    i -= a.W;
                uint8_t *dst =
                    reinterpret_cast<uint8_t *>(sh.dst[i]) + (row0 + r) * a.ld_out_b + col0;
                if (kChecked && !inside(sh.dst[i], a.out_ext_b, reinterpret_cast<uint64_t>(dst),
                                        it.rb)) {
                    bounds_fault(a.status);
                    continue;
                }
                if (a.store_hint)
                    ptx::bulk_s2g_hint(dst, buf + (uint32_t)r * pitch, it.rb, pol_st);
                else
                    ptx::bulk_s2g(dst, buf + (uint32_t)r * pitch, it.rb);
            }
            ptx::bulk_commit();
            if (j0 + grp < a.W) {  // the next group waits until this one has read its data
                ptx::bulk_wait_read<0>();
                __syncwarp();
            }
        }
        __syncwarp();  // every lane has read this stage's item
        issue_next();
    }

    if (!ok) {
        report_status(a.status, kStatusTimeout);
        // loads issued but not consumed: items k .. issued - 1
        for (int64_t q = k; q < issued; ++q) {
            const int st = (int)(q % stages);
            ptx::mbar_wait(full0 + 8u * st, (uint32_t)((q / stages) & 1), kDrainLimitNs);
        }
    }
    ptx::bulk_wait_all();
    trace_mark(a.trace, 1);
}

// Tensor-map path: same ring pipeline as ag_bulk_kernel; a tile is one box.
// in_map views the sources as {N, M, heaps} (all-to-all: {N, M, W, heaps}).
template <int D>
__global__ void __launch_bounds__(kAgWarps * 32, 1)
    ag_tma_kernel(const __grid_constant__ CUtensorMap in_map, const __grid_constant__ OutMaps out,
                  const GatherArgs a, int stages, int stage_bytes)
{
    const int npipe = blockDim.x >> 5;
    extern __shared__ __align__(1024) uint8_t smem[];
    AgShared &sh = *reinterpret_cast<AgShared *>(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    trace_mark(a.trace, 0);
    if (kChecked && !extents_ok(a)) {
        if (threadIdx.x == 0)
            bounds_fault(a.status);
        return;
    }

    if (threadIdx.x == 0) {
        for (int w = 0; w < npipe; ++w)
            for (int s = 0; s < stages; ++s)
                ptx::mbar_init(ptx::smem_addr(&sh.full[w][s]), 1);
        ptx::fence_barrier_init();
        tma_prefetch(&in_map);
    }
    if (threadIdx.x < (unsigned)a.W)
        tma_prefetch(&out.map[threadIdx.x]);
    if (kChecked)  // the maps come from the host's bases; the device table must agree
        load_member_bases(a, sh.dst, sh.src);
    __syncthreads();

    int dest;
    Feed feed = make_feed(a, warp, npipe, lane, &dest);
    const int lookahead = stages - D;
    const uint32_t ring = ptx::smem_addr(smem + kAgHeader) + (uint32_t)(warp * stages * stage_bytes);
    const uint32_t full0 = ptx::smem_addr(&sh.full[warp][0]);
    const uint32_t box_bytes = (uint32_t)(a.bm * a.bn_b);  // a full box, clipped parts zero-filled
    const uint64_t pol_st = a.store_hint ? ptx::policy_evict_first() : 0;
    const int bn = (int)(a.bn_b / a.es);
    const int grp = (a.dests_per_wait > 0 && a.dests_per_wait < a.W) ? a.dests_per_wait : a.W;

    int64_t issued = 0;
    auto issue_next = [&]() {
        const int64_t t = feed_next(feed, lane);
        if (t < 0)
            return;
        if (issued >= stages) {
            ptx::bulk_wait_read<D>();
            __syncwarp();
        }
        const int st = (int)(issued % stages);
        const bool stall = a.inject_stall && issued == 0 && blockIdx.x == 0 && warp == 0;
        ++issued;
        if (lane == 0) {
            const Item it = decode_item(a, t);
            sh.item[warp][st] = it;
            if (kChecked && !stall && it.rows == 0) {
                ptx::mbar_arrive(full0 + 8u * st);  // an item outside the grid: no load
            } else if (!stall) {  // test hook: a stalled stage's barrier phase never completes
                const uint32_t bar = full0 + 8u * st;
                ptx::mbar_arrive_expect_tx(bar, box_bytes);
                const int h = a.in_abs ? 0 : a.rank_start + it.g * a.rank_stride;
                const uint32_t dst = ring + (uint32_t)st * stage_bytes;
                if (a.mode == kModeAllToAll)
                    tma_load_box4(dst, &in_map, (int)it.tn * bn, (int)(it.tm * a.bm), it.d, h,
                                  bar);
                else
                    tma_load_box(dst, &in_map, (int)it.tn * bn, (int)(it.tm * a.bm), h, bar);
            }
        }
        __syncwarp();
    };

    for (int q = 0; q < lookahead; ++q)
        issue_next();

    int64_t k = 0;
    bool ok = true;
    for (; k < issued; ++k) {
        const int st = (int)(k % stages);
        const uint32_t parity = (uint32_t)((k / stages) & 1);
        const bool mine = ptx::mbar_wait(full0 + 8u * st, parity, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, mine)) {
            ok = false;
            break;
        }
        const Item it = sh.item[warp][st];
        const uint32_t buf = ring + (uint32_t)st * stage_bytes;
        const int c0 = (int)it.tn * bn, c1 = (int)(it.tm * a.bm);
        if (kChecked && it.rows == 0) {
            // an item outside the grid (reported at decode): no store
        } else if (a.mode == kModeGather) {
            // lane j stores to destination j of the group: the local copy first,
            // peers rotated; `grp` destinations per wait
            for (int j0 = 0; j0 < a.W; j0 += grp) {
                const int jend = j0 + grp < a.W ? j0 + grp : a.W;
                for (int j = j0 + lane; j < jend; j += 32) {
                    int i = it.g + j;
                    if (i >= a.W)
                        i -= a.W;
                    if (a.store_hint)
                        tma_store_box_hint(&out.map[i], buf, c0, c1, it.g, pol_st);
                    else
                        tma_store_box(&out.map[i], buf, c0, c1, it.g);
                }
                ptx::bulk_commit();
                if (jend < a.W) {
                    ptx::bulk_wait_read<0>();
                    __syncwarp();
                }
            }
        } else {
            // one destination: the program's own (partitioned) or the block's (all-to-all)
            if (lane == 0) {
                const CUtensorMap *m = &out.map[a.mode == kModePartitioned ? dest : it.d];
                if (a.store_hint)
                    tma_store_box_hint(m, buf, c0, c1, it.g, pol_st);
                else
                    tma_store_box(m, buf, c0, c1, it.g);
            }
            ptx::bulk_commit();
        }
        __syncwarp();
        issue_next();
    }

    if (!ok) {
        report_status(a.status, kStatusTimeout);
        for (int64_t q = k; q < issued; ++q) {
            const int st = (int)(q % stages);
            ptx::mbar_wait(full0 + 8u * st, (uint32_t)((q / stages) & 1), kDrainLimitNs);
        }
    }
    ptx::bulk_wait_all();
    trace_mark(a.trace, 1);
}

template <int VB>
struct VecType;
template <>
struct VecType<16> { using T = uint4; };
template <>
struct VecType<8> { using T = uint2; };
template <>
struct VecType<4> { using T = uint32_t; };
template <>
struct VecType<2> { using T = uint16_t; };

constexpr int kVecThreads = 512;
constexpr int kVecUnroll = 4;

template <int VB>
__global__ void __launch_bounds__(kVecThreads) ag_vec_kernel(const GatherArgs a)
{
    using V = typename VecType<VB>::T;
    __shared__ uint64_t dst[kMaxWorld];
    __shared__ uint64_t src[kMaxWorld];
    trace_mark(a.trace, 0);
    if (kChecked && !extents_ok(a)) {
        if (threadIdx.x == 0)
            bounds_fault(a.status);
        return;
    }
    load_member_bases(a, dst, src);
    __syncthreads();

    const int crow = (int)(a.bn_b / VB);           // vectors per full tile row
    const int tile_vecs = a.bm * crow;             // vectors per full tile
    const Walk walk = make_walk(a, 0, 1);          // the whole program walks one item list
    const int64_t stride = walk.step * kVecUnroll;

    for (int64_t base = walk.first; base < a.total_items; base += stride) {
        for (int c = threadIdx.x; c < tile_vecs; c += blockDim.x) {
            const int r = c / crow;
            const int cc = c - r * crow;
            V v[kVecUnroll];
            bool valid[kVecUnroll];
            Item it[kVecUnroll];
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                const int64_t t = base + (int64_t)u * walk.step;
                valid[u] = false;
                if (t < a.total_items) {
                    it[u] = decode_item(a, t);
                    valid[u] = r < it[u].rows && (uint32_t)cc * VB < it[u].rb;
                    if (valid[u]) {
                        // all-to-all: the source's block d starts at row d*M
                        const int64_t srow = (it[u].d >= 0 ? (int64_t)it[u].d * a.M : 0) +
                                             it[u].tm * a.bm + r;
                        const uint8_t *s = reinterpret_cast<const uint8_t *>(src[it[u].g]) +
                                           srow * a.ld_in_b + it[u].tn * a.bn_b + (int64_t)cc * VB;
                        if (kChecked && !inside(src[it[u].g], a.in_ext_b,
                                                reinterpret_cast<uint64_t>(s), VB)) {
                            bounds_fault(a.status);
                            valid[u] = false;
                            continue;
                        }
                        v[u] = *reinterpret_cast<const V *>(s);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                if (!valid[u])
                    continue;
                const int64_t off = ((int64_t)it[u].g * a.M + it[u].tm * a.bm + r) * a.ld_out_b +
                                    it[u].tn * a.bn_b + (int64_t)cc * VB;
                if (a.mode == kModeGather) {
                    for (int j = 0; j < a.W; ++j) {
                        int i = it[u].g + j;
                        if (i >= a.W)
                            i -= a.W;
                        if (kChecked && !inside(dst[i], a.out_ext_b, dst[i] + (uint64_t)off, VB)) {
                            bounds_fault(a.status);
                            continue;
                        }
                        *reinterpret_cast<V *>(reinterpret_cast<uint8_t *>(dst[i]) + off) = v[u];
                    }
                } else {
                    const int i = a.mode == kModePartitioned ? walk.dest : it[u].d;
                    if (kChecked && !inside(dst[i], a.out_ext_b, dst[i] + (uint64_t)off, VB)) {
                        bounds_fault(a.status);
                        continue;
                    }
                    *reinterpret_cast<V *>(reinterpret_cast<uint8_t *>(dst[i]) + off) = v[u];
                }
            }
        }
    }
    trace_mark(a.trace, 1);
}

}  // namespace

// Ring geometry for a tile of `stage_raw` bytes and `programs` programs:
// pipelines (warps) per program, stages per pipeline and read depth D.
// False if not even one pipeline of three stages fits.
bool ring_geometry(int64_t stage_raw, int programs, int target, int *npipe, int *stages,
                   int *depth, int *stage_bytes)
{
    const int64_t sb = (stage_raw + 1023) / 1024 * 1024;
    int want = (target + programs - 1) / programs;
    want = want < 1 ? 1 : (want > kAgWarps ? kAgWarps : want);
    for (int np = want; np >= 1; --np) {
        const int64_t st = gg_min64(kAgMaxStages, (kAgSmemBudget - kAgHeader) / (np * sb));
        if (st >= 3) {
            *npipe = np;
            *stages = (int)st;
            *depth = st >= 6 ? 4 : (st >= 4 ? 2 : 1);
            *stage_bytes = (int)sb;
            return true;
        }
    }
    return false;
}

// Claimed runs (GatherArgs::work) on the tensor-map path for the all-gather
// and the all-to-all: about 64 runs per pipeline, 2 to 8 items a run; the
// counter is zeroed on the launch's stream first (one memset of a few
// microseconds).  The counter is a heap workspace slot, or, for
// gg_all_gather_noalloc, the library's static scratch array (gg_api.cu),
// which every call on a device shares: that call relies on this memset to
// start each launch from zero.  Automatic choice: only launches that move at least
// kClaimAutoBytes over at least 3/4 of the SMs claim.  Below that every SM
// gets the bandwidth it asks for, and claims only add their per-run cost
// (measured on GB300: 5-7% slower at 16-64 programs, 8-16% faster at 128-148
// programs for the larger all-gathers); the bulk path and the partitioned
// all-gather lost 5-7% with claims even at 148 programs and keep fixed shares.
constexpr int64_t kClaimAutoBytes = 256ll << 20;

static cudaError_t prepare_claims(GatherArgs &a, int programs, int npipe, cudaStream_t s)
{
    if (!a.work || a.mode == kModePartitioned || a.claim_policy == kClaimNever) {
        a.work = nullptr;
        return cudaSuccess;
    }
    const int64_t pipes = (int64_t)programs * npipe;
    const int64_t stores = a.mode == kModeGather ? a.W : 1;  // per item loaded
    const int64_t bytes = a.total_items * a.bm * a.bn_b * (1 + stores);
    int64_t c = a.total_items / (pipes * 64);
    c = c < 2 ? 2 : (c > 8 ? 8 : c);
    bool claim = a.total_items >= 4 * pipes * c;
    if (claim && a.claim_policy == kClaimAuto) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        claim = bytes >= kClaimAutoBytes && 4 * (int64_t)programs >= 3 * (int64_t)sms;
    }
    if (!claim) {
        a.work = nullptr;
        return cudaSuccess;
    }
    a.chunk = (int)c;
    return cudaMemsetAsync(a.work, 0, sizeof(unsigned long long), s);
}

// The ring kernels may use up to kAgSmemBudget bytes of dynamic shared
// memory: the limit is raised once per device and kernel (a launch then asks
// for what it uses), not on every launch.
template <typename Kernel>
static cudaError_t allow_ring_smem(Kernel kernel, std::atomic<uint64_t> &done_mask)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
    if (bit && (done_mask.load(std::memory_order_relaxed) & bit))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAgSmemBudget);
    if (e == cudaSuccess && bit)
        done_mask.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

template <int D>
static cudaError_t launch_bulk_depth(const GatherArgs &a, int programs, int npipe, int stages,
                                     int stage_bytes, cudaStream_t s)
{
    static std::atomic<uint64_t> done{0};
    const int smem = kAgHeader + npipe * stages * stage_bytes;  // <= kAgSmemBudget
    cudaError_t e = allow_ring_smem(ag_bulk_kernel<D>, done);
    if (e != cudaSuccess)
        return e;
    ag_bulk_kernel<D><<<programs, npipe * 32, smem, s>>>(a, stages, stage_bytes);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_tma_depth(const CUtensorMap &in_map, const OutMaps &out,
                                    const GatherArgs &a, int programs, int npipe, int stages,
                                    int stage_bytes, cudaStream_t s)
{
    static std::atomic<uint64_t> done{0};
    const int smem = kAgHeader + npipe * stages * stage_bytes;  // <= kAgSmemBudget
    cudaError_t e = allow_ring_smem(ag_tma_kernel<D>, done);
    if (e != cudaSuccess)
        return e;
    ag_tma_kernel<D><<<programs, npipe * 32, smem, s>>>(in_map, out, a, stages, stage_bytes);
    return cudaGetLastError();
}

cudaError_t launch_gather_tma(const CUtensorMap &in_map, const OutMaps &out, const GatherArgs &args,
                              int programs, cudaStream_t s)
{
    GatherArgs a = args;
    int npipe, stages, depth, stage_bytes;
    const int target = a.mode == kModeGather ? kAgTargetPipes : kAgTargetPipesSingle;
    if (!ring_geometry((int64_t)a.bm * a.bn_b, programs, target, &npipe, &stages, &depth,
                       &stage_bytes))
        return cudaErrorInvalidValue;
    cudaError_t e = prepare_claims(a, programs, npipe, s);
    if (e != cudaSuccess)
        return e;
    switch (depth) {
    case 4: return launch_tma_depth<4>(in_map, out, a, programs, npipe, stages, stage_bytes, s);
    case 2: return launch_tma_depth<2>(in_map, out, a, programs, npipe, stages, stage_bytes, s);
    default: return launch_tma_depth<1>(in_map, out, a, programs, npipe, stages, stage_bytes, s);
    }
}

cudaError_t launch_gather_bulk(const GatherArgs &args, int programs, cudaStream_t s)
{
    GatherArgs a = args;
    int npipe, stages, depth, stage_bytes;
    if (!ring_geometry((int64_t)a.bm * a.bn_b, programs, kAgTargetPipes, &npipe, &stages, &depth,
                       &stage_bytes))
        return cudaErrorInvalidValue;  // tile too large (the host validates first)
    a.work = nullptr;  // fixed shares (claims do not pay off on this path)
    switch (depth) {
    case 4: return launch_bulk_depth<4>(a, programs, npipe, stages, stage_bytes, s);
    case 2: return launch_bulk_depth<2>(a, programs, npipe, stages, stage_bytes, s);
    default: return launch_bulk_depth<1>(a, programs, npipe, stages, stage_bytes, s);
    }
}

cudaError_t launch_gather_vec(const GatherArgs &a, int programs, int vec_bytes, cudaStream_t s)
{
    switch (vec_bytes) {
    case 16: ag_vec_kernel<16><<<programs, kVecThreads, 0, s>>>(a); break;
    case 8: ag_vec_kernel<8><<<programs, kVecThreads, 0, s>>>(a); break;
    case 4: ag_vec_kernel<4><<<programs, kVecThreads, 0, s>>>(a); break;
    case 2: ag_vec_kernel<2><<<programs, kVecThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gg
