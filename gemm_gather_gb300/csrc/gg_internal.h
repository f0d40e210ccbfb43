// Declarations shared by the library's translation units (host side).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gg {

constexpr int kMaxWorld = 64;
constexpr int kStatusTimeout = -6;    // GG_ERR_TIMEOUT
constexpr int kStatusNotInHeap = -3;  // GG_ERR_NOT_IN_HEAP (checked build)
// Trace records (gg_set_trace): one per kernel family, 4 words each.
constexpr int kTraceGather = 0, kTraceFused = 4, kTraceWords = 8;

// Collectives the gather kernels run.
constexpr int kModeGather = 0;       // every tile to every member
constexpr int kModePartitioned = 1;  // program p serves member p mod W only
constexpr int kModeAllToAll = 2;     // member i's block d to member d's block i

// One TMA tensor map per group member's gathered output (kernel parameter).
struct OutMaps {
    CUtensorMap map[kMaxWorld];
};

bool tensor_maps_available();
// A tiled tensor map of `rank` dimensions (dims in elements, strides in bytes
// for dimensions 1..rank-1, box in elements), no interleave, zero OOB fill.
bool encode_map(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                const uint64_t *dims, const uint64_t *strides_b, const uint32_t *box,
                CUtensorMapSwizzle swizzle);
// Output maps of W members: member d's output at member_out[d], viewed as
// {N, M, W} so that boxes clip at the end of each row block.
bool encode_out_maps(OutMaps *out, const uint64_t *member_out, int W, int64_t M, int64_t N,
                     int64_t ld_out_b, int es, uint32_t box_cols, uint32_t box_rows,
                     CUtensorMapDataType dt, CUtensorMapSwizzle swizzle);

// One launch of the tiled all-gather (or of its partitioned form, or of the
// all-to-all).  A "source" is a group member whose M x N block is gathered; a
// launch covers n_src consecutive group indices starting at src_first.  Work
// item t (0 <= t < n_src * tiles_per_src, times W for the all-to-all) is a
// tile of source src_first + t / (items per source).
struct GatherArgs {
    const uint64_t *bases;  // device heap-bases table, one entry per heap
    // The heap layout the table must describe: entry h == heap_lo + h * part_bytes.
    // Read only by the checked build, which also bounds every raw access by the
    // extents below.
    uint64_t heap_lo, part_bytes;
    int64_t in_ext_b;   // bytes one source's input spans ((rows - 1) * ld_in_b + row_b)
    int64_t out_ext_b;  // bytes one member's gathered output spans
    int W, rank_start, rank_stride;
    int n_src, src_first;
    const uint8_t *in_abs;  // non-null: the one source's block (any device memory)
    int64_t in_off;         // else: source block at this offset in the member's partition
    int64_t out_off;        // gathered output at this offset in every member's partition
    int64_t ld_in_b, ld_out_b;  // row pitches in bytes
    int64_t M;                  // rows per block
    int64_t row_b;              // bytes per row (N * element size)
    int bm;                     // tile rows
    int64_t bn_b;               // tile row bytes (block_n * element size)
    int64_t tiles_n, tiles_per_src, total_items;
    int es;                     // element size (bytes)
    int mode;                   // kModeGather / kModePartitioned / kModeAllToAll
    int dests_per_wait;         // destinations stored per wait (0: all at once)
    int *status;
    uint64_t wait_limit_ns;
    int inject_stall;  // test hook: program 0 never arms its first stage
    // Claimed-run counter (tensor-map path), set to zero before the launch
    // when runs are claimed; null: every pipeline walks a fixed share of the
    // items.
    unsigned long long *work;
    int chunk;         // items per claimed run
    int claim_policy;  // kClaimAuto / kClaimAlways / kClaimNever
    unsigned long long *trace;  // non-null: the launch's trace record (see trace_mark)
    int store_hint;             // kStorePlain / kStoreEvictFirst (tensor-map and bulk stores)
};

constexpr int kClaimAuto = 0, kClaimAlways = 1, kClaimNever = 2;
constexpr int kStorePlain = 0, kStoreEvictFirst = 1;
// Bytes of one workspace slot (a counter, padded to its own 128 bytes).
constexpr int kWorkSlotBytes = 128;

// Bulk path: 16-byte aligned addresses, pitches, bn_b and row_b.
cudaError_t launch_gather_bulk(const GatherArgs &a, int programs, cudaStream_t s);
// Tensor-map path: in_map views the source blocks as {N, M, heaps} (or the one
// block as {N, M, 1}); out holds one map per member; box = one tile.
cudaError_t launch_gather_tma(const CUtensorMap &in_map, const OutMaps &out, const GatherArgs &a,
                              int programs, cudaStream_t s);
// Vector path: vec_bytes in {16, 8, 4, 2} divides every address, pitch and row length.
cudaError_t launch_gather_vec(const GatherArgs &a, int programs, int vec_bytes, cudaStream_t s);

// One launch of the fused matmul + all-gather (see mag_kernel.cu).  The
// outputs are reached through per-member tensor maps (OutMaps).
struct FusedArgs {
    int W, rank_start, rank_stride;
    int n_src, src_first;
    const void *a_abs;     // non-null: the one source's A (any device memory)
    int64_t a_off;         // else: A at this offset in each member's partition
    const void *b;         // K x N, shared
    int64_t lda, ldb;      // elements
    int64_t out_off;       // gathered output offset in every member's partition
    int64_t ld_out;        // elements
    int64_t M, N, K;
    int is_bf16;
    // for the A tensor map over all partitions (group launches)
    uint64_t heap_base;    // device address of partition 0
    uint64_t part_bytes;
    int num_heaps;
    int *status;
    uint64_t wait_limit_ns;
    int inject_stall;  // test hook: CTA 0 never arms its first ring stage
    int b_boxes3d;     // set by the launcher: B stages load as one 3-d box
    int wide;          // 128 x 512 CTA tiles (256 x 512 per pair): two MMAs per A stage
    int tn_group;      // set by the launcher: tile columns per group of the tile order
    unsigned long long *trace;  // non-null: the launch's trace record (see trace_mark)
};

// Fused kernel variants: 1 = 1-SM (one CTA per 128 x 256 tile), 2 = CTA
// pairs (256 x 256 pair tiles, or 256 x 512 with FusedArgs::wide); 0 =
// automatic.  The variant a launch runs for `requested`:
inline int fused_variant(int programs, int requested)
{
    return requested == 1 || programs < 2 ? 1 : 2;
}

// variant: 0 = automatic, 1 / 2 as fused_variant
cudaError_t launch_matmul_all_gather(const FusedArgs &a, const OutMaps &out, int programs,
                                     int variant, cudaStream_t s, const char **why);

// The fused call with K == 0: every product is the zero matrix, so the rows of
// sources [src_first, src_first + n_src) in every member's gathered output
// are filled with zeros (fill_kernel.cu).  Row pitch and row length are whole
// 16-byte units and the outputs 16-byte aligned.
struct ZeroArgs {
    uint64_t out[kMaxWorld];  // gathered output of member d (host-side bases + offset)
    int W;
    int src_first, n_src;
    int64_t M;                // rows per source block
    int64_t ld_out_b, row_b;  // row pitch and row length in bytes
};
cudaError_t launch_zero_rows(const ZeroArgs &z, int programs, cudaStream_t s);

}  // namespace gg
