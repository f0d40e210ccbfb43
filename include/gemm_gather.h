/*
 * gemm_gather — tiled all-gather over a symmetric heap, alone and fused into
 * the epilogue of a matmul, for one NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  All device memory is owned by the
 * caller; the library never allocates device memory, and its only device
 * state is three small static objects per device: the 256-byte counter array
 * of gg_all_gather_noalloc, the int status word of launches given no status
 * word (gg_device_status) and 64 bytes of trace records (gg_set_trace).  The
 * same calls also come in a checked build (gg_checked_build) with
 * device-side bounds checks in the gather kernels.  Every call that launches work is
 * asynchronous on the caller's stream.  Errors found on the host are
 * returned before anything is launched; gg_last_error() then describes
 * them.  No call aborts the process.
 *
 * Logical ranks.  On one GPU the W ranks of a group are logical: H equal
 * partitions ("heaps") of one device allocation, reached through a table of
 * heap base addresses, the way the ROCm/iris pages validate their kernels on
 * a single GPU (iris #594, "Local validation": independent allocations stand
 * for ranks).  A symmetric buffer sits at the same byte offset in every
 * partition (iris PR #626, "Summary": peer address = local address +
 * (peer base - local base)).
 *
 * Group (iris #591 "Gluon all-gather reloads peer heap bases inside the tile
 * loop", Description §1): member i of a group is heap
 * rank_start + i * rank_stride, for i in [0, world_size).  Heaps outside the
 * group are never touched.
 *
 * Gather (iris #594, "Multi-GPU CI": same result as
 * torch.distributed.all_gather_into_tensor): the gathered output of every
 * member d is world_size*M x N; row block i (rows i*M .. i*M+M-1) is member
 * i's M x N input.  Elements are copied bit for bit.  Columns N..ld_out-1 of
 * the output (padding) are never written.
 */
#ifndef GEMM_GATHER_H
#define GEMM_GATHER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *gg_stream_t;

typedef enum {
    GG_OK = 0,
    GG_ERR_INVALID_ARG = -1,  /* bad size, rank, group, pitch or overlap     */
    GG_ERR_ALIGNMENT = -2,    /* pointer/pitch alignment a path requires     */
    GG_ERR_NOT_IN_HEAP = -3,  /* a symmetric buffer does not fit a partition;
                                 checked build: a device access out of bounds */
    GG_ERR_UNSUPPORTED = -4,  /* valid request the library does not implement */
    GG_ERR_CUDA = -5,         /* a CUDA runtime call failed                  */
    GG_ERR_TIMEOUT = -6       /* device: a bounded wait gave up (status word)*/
} gg_status;

typedef enum { GG_F16 = 0, GG_BF16 = 1, GG_F32 = 2 } gg_dtype;

/* Tile shape.  Always explicit: the library has no default tile and never
 * replaces the one it is given (iris #594, "Reviewer performance evaluation":
 * a launcher that remapped an explicit 32x64 tile to 8x256 made 32x64
 * impossible to run).  A shape a kernel cannot run returns
 * GG_ERR_UNSUPPORTED. */
typedef struct { int block_m, block_n; } gg_tile;

/* Process group over heap indices (see above). */
typedef struct { int rank_start, rank_stride, world_size; } gg_group;

typedef struct gg_heap gg_heap; /* opaque host handle */

/* Largest world_size a call accepts, and largest number of heaps. */
#define GG_MAX_WORLD 64
#define GG_MAX_HEAPS 1024

/* Supported fused (matmul_all_gather) tiles: the output tile of one CTA,
 * {GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N} or {GG_FUSED_BLOCK_M,
 * GG_FUSED_BLOCK_N_WIDE}. */
#define GG_FUSED_BLOCK_M 128
#define GG_FUSED_BLOCK_N 256
#define GG_FUSED_BLOCK_N_WIDE 512

/* ---------------------------------------------------------------------------
 * gg_heap_create — describe a symmetric heap of `num_heaps` partitions of
 * `bytes_per_rank` bytes each, laid out back to back from `dev_base`
 * (device memory, caller-owned, at least num_heaps*bytes_per_rank bytes), and
 * write the heap-bases table: entry h = dev_base + h*bytes_per_rank, as
 * uint64, into `dev_bases_table` (device memory, caller-owned, num_heaps
 * entries).  The table write is a copy enqueued on `stream`; it is ordered
 * before any later gather or fused call on that stream.  (iris PR #626
 * "Summary" and iris #591 Description §1: heap_bases.)
 * Requirements: dev_base 256-byte aligned; bytes_per_rank a positive multiple
 * of 256; 1 <= num_heaps <= GG_MAX_HEAPS.  On success *out is a new handle
 * (host memory only), released by gg_heap_destroy.
 * ------------------------------------------------------------------------- */
gg_status gg_heap_create(void *dev_base, size_t bytes_per_rank, int num_heaps,
                         uint64_t *dev_bases_table, gg_stream_t stream, gg_heap **out);

/* gg_heap_wrap — the same handle as gg_heap_create, without writing the
 * device table: for callers that write or share the table themselves (its
 * contents must then equal gg_heap_bases before the first launch).  Touches
 * no device state, so it also serves host-only validation with the
 * *_check entry points below. */
gg_status gg_heap_wrap(void *dev_base, size_t bytes_per_rank, int num_heaps,
                       uint64_t *dev_bases_table, gg_heap **out);

/* Copy the heap-bases table (host copy kept by the handle) into host_out[0..n). */
gg_status gg_heap_bases(const gg_heap *heap, uint64_t *host_out, int n);

/* Number of partitions and partition size of a heap. */
gg_status gg_heap_info(const gg_heap *heap, int *num_heaps, size_t *bytes_per_rank);

/* Release the host handle (device memory stays the caller's). NULL is a no-op. */
gg_status gg_heap_destroy(gg_heap *heap);

/* ---------------------------------------------------------------------------
 * gg_heap_set_workspace — give the all-gather and all-to-all launches on
 * `heap` a workspace of `bytes` bytes of device memory (caller-owned,
 * 256-byte aligned, a positive multiple of GG_WORKSPACE_SLOT_BYTES, at most
 * 2^20 slots) for load balancing; NULL with bytes == 0 removes it.  The pages
 * have no counterpart: their programs each walk a fixed share of the tiles.
 *
 * With a workspace, a tensor-map-path launch that the claim policy (below)
 * selects hands tiles out in short runs claimed from a counter, instead of a
 * fixed share per program: programs on SMs that get more memory bandwidth
 * claim more runs, so all of them finish together.  Results are identical.
 * Such a launch takes the next slot of the workspace (round robin) and zeroes
 * its counter on its own stream before the kernel (one memset).  Launches on
 * one heap that may run at the same time (different streams, not ordered)
 * must number at most bytes / GG_WORKSPACE_SLOT_BYTES: two running launches
 * that share a slot may skip or repeat tiles (no access outside their
 * buffers and no hang, but wrong results).  This call touches no device
 * memory; the workspace must stay allocated while launches use it.
 * ------------------------------------------------------------------------- */
#define GG_WORKSPACE_SLOT_BYTES 128
gg_status gg_heap_set_workspace(gg_heap *heap, void *dev_work, size_t bytes);

/* Which launches claim runs (given a workspace):
 *   GG_CLAIM_AUTO (default): tensor-map all-gathers and all-to-alls that move
 *     at least 256 MiB of tile bytes (read plus written) with comm_programs at
 *     least 3/4 of the device's SMs, where the SMs compete for bandwidth;
 *   GG_CLAIM_ALWAYS: every tensor-map all-gather and all-to-all with at least
 *     a few runs per pipeline;
 *   GG_CLAIM_NEVER: fixed shares only.
 * The bulk and vector paths and the partitioned all-gather always keep fixed
 * shares.  Applies to launches made after the call, from any thread;
 * GG_ERR_INVALID_ARG for another value. */
#define GG_CLAIM_AUTO 0
#define GG_CLAIM_ALWAYS 1
#define GG_CLAIM_NEVER 2
gg_status gg_set_claim_policy(int policy);
int gg_get_claim_policy(void);

/* ---------------------------------------------------------------------------
 * gg_set_store_policy — an L2 eviction-priority hint on the stores of the
 * all-gather family (the pages' store-policy knob: the Gluon all-gather's
 * local copy stores with a write-through cache policy, iris #594 "PR
 * description").  GG_STORE_EVICT_FIRST (the default): every TMA tensor
 * store (tensor-map path) and bulk store (bulk path) carries an L2
 * evict_first hint, so the gathered output, written once and not read again
 * by the launch, is the first to leave L2 (measured on GB300: 0.25% faster
 * than plain stores at W=8 16384x8192 f32 and 4096x4096 f16).
 * GG_STORE_PLAIN: no hint.  The vector path stores without a hint.  Results
 * are identical either way.
 * Process-wide (all devices and threads), read when a call is validated.
 * Anything else returns GG_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
#define GG_STORE_PLAIN 0
#define GG_STORE_EVICT_FIRST 1
gg_status gg_set_store_policy(int policy);
int gg_get_store_policy(void);

/* ---------------------------------------------------------------------------
 * gg_all_gather — the persistent tiled all-gather (iris PR #626, "Triton CCL
 * all-gather"; iris #594, "PR description"; iris #591, Description §1).
 *
 * rank >= 0: heap `rank` (a member of `group`, group index i) contributes:
 *   `input` (any device pointer, M x N, row pitch ld_in elements) is written
 *   into row block i of the output of every member, itself first.
 * rank == -1: every member contributes in one launch; `input` must then be a
 *   symmetric heap buffer (the byte offset of `input` within its partition is
 *   used in every member's partition).
 * `output` is a symmetric heap buffer: a pointer into any partition; its byte
 *   offset within that partition locates the world_size*M x N output (row
 *   pitch ld_out elements) in every member's partition.  The whole output
 *   must fit inside a partition (else GG_ERR_NOT_IN_HEAP) and must not
 *   overlap the input (else GG_ERR_INVALID_ARG).
 * tile: block_m rows x block_n columns of one work item; each work item is
 *   read once and stored to every member, the local copy first and the peers
 *   in rotated order (i+1, i+2, ... mod world_size; iris PR #626, "Summary").
 *   block_m in [1, 256], block_n >= 1, block_m*block_n*elem_size <= 32768.
 * comm_programs: number of persistent programs (CTAs) of the launch, 1..65535;
 *   for rank == -1 they share all world_size x tiles work items.
 * dev_status: device int, or NULL; if a bounded wait inside the kernel gives
 *   up (the kernel then stops early and part of the output may be left
 *   unwritten), GG_ERR_TIMEOUT is stored there (first error wins; the caller
 *   zeroes it).  With NULL it is stored in the library's status word of the
 *   device instead (gg_device_status), so no early stop goes unreported.
 *   The checked build (gg_checked_build) also stores GG_ERR_NOT_IN_HEAP there
 *   when a device-side bounds check skips an access.
 *   M == 0 or N == 0 launches nothing and returns GG_OK.
 * Any alignment is accepted: 16-byte aligned pointers and pitches take the
 *   tensor-map or bulk-copy path, others a narrower vector path.  Results
 *   are identical.
 * ------------------------------------------------------------------------- */
gg_status gg_all_gather(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                        void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                        gg_tile tile, int comm_programs, gg_group group, int *dev_status,
                        gg_stream_t stream);

/* ---------------------------------------------------------------------------
 * gg_all_gather_noalloc — gg_all_gather for callers that cannot allocate
 * device memory.  The pages have no counterpart (they allocate freely).
 *
 * Who needs it: code that may not call cudaMalloc, or any allocator, once it
 * is running -- a plugin inside a framework that owns all device memory, a
 * real-time loop where an allocation's implicit device synchronization is not
 * allowed, a process whose memory budget is fixed at start-up -- and that
 * therefore has no device buffer to hand gg_heap_set_workspace.
 *
 * Same arguments, validation and results as gg_all_gather (automatic data
 * path, claim policy of gg_set_claim_policy; the heap's workspace, if any, is
 * not used).  When the launch claims runs of tiles, its counter lives in a
 * 256-byte static device array inside this library instead of a workspace;
 * the call zeroes that counter with one memset on `stream` before the kernel
 * and allocates nothing.  The scratch needed does not grow with M, N,
 * world_size or comm_programs (one 8-byte counter), so no size the all-gather
 * accepts is rejected for lack of scratch.
 * Limits: every GPU that loads the library holds the 256 bytes until the
 * process exits; all calls on a device share the one counter, so calls that
 * may overlap on the GPU (different streams, not ordered) race and may skip
 * or repeat tiles -- order them on one stream.  The first call on each device
 * (with that device current) looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * The address found then is kept for the life of the process: after a
 * cudaDeviceReset of that device it is stale, so do not call this entry
 * point on a device that was reset after its first call.
 * ------------------------------------------------------------------------- */
gg_status gg_all_gather_noalloc(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                                void *output, int64_t ld_out, int64_t M, int64_t N,
                                gg_dtype dtype, gg_tile tile, int comm_programs, gg_group group,
                                int *dev_status, gg_stream_t stream);

/* Data-path variants of gg_all_gather (same arguments and result):
 *   GG_AG_AUTO      tensor-map path when it applies, else bulk, else vector
 *                   (what gg_all_gather does)
 *   GG_AG_TMA       each tile moved by one TMA tensor load into shared memory
 *                   and one TMA tensor store per destination, through tensor
 *                   maps built on the host from the heap-bases table; needs
 *                   16-byte aligned input, output, pitches and
 *                   block_n*elem_size, and block_n <= 256 (N may be ragged)
 *   GG_AG_BULK      tiles staged in shared memory by bulk copies (TMA engine),
 *                   stored to each destination by bulk copies; needs 16-byte
 *                   aligned pointers, pitches, block_n*elem_size and
 *                   N*elem_size (else GG_ERR_ALIGNMENT)
 *   GG_AG_VECTOR    16/8/4/2-byte vector loads into registers, then one vector
 *                   store per destination (widest width the alignment allows)
 */
typedef enum { GG_AG_AUTO = 0, GG_AG_BULK = 1, GG_AG_VECTOR = 2, GG_AG_TMA = 3 } gg_ag_path;

gg_status gg_all_gather_path(const gg_heap *heap, int rank, const void *input,
                             int64_t ld_in, void *output, int64_t ld_out, int64_t M,
                             int64_t N, gg_dtype dtype, gg_tile tile, int comm_programs,
                             gg_group group, int *dev_status, gg_stream_t stream,
                             gg_ag_path path);

/* Validate a gg_all_gather_path call exactly as the launching call does and
 * launch nothing.  *chosen (nullable) receives the path a launch would take
 * (GG_AG_TMA, GG_AG_BULK or GG_AG_VECTOR; GG_AG_AUTO when there is nothing
 * to launch). */
gg_status gg_all_gather_check(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                              void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                              gg_tile tile, int comm_programs, gg_group group, gg_ag_path path,
                              gg_ag_path *chosen);

/* ---------------------------------------------------------------------------
 * gg_all_gather_grouped — gg_all_gather_path whose tile stores go out
 * `dests_per_wait` destinations at a time: each group of stores waits until
 * the previous group has finished reading shared memory (the "INLINE"
 * grouping of iris #594, "Compiler inspection and grouping", and iris #591,
 * Description §2: a bounded number of destination stores per wait).
 * dests_per_wait = 0 (or >= world_size) stores to all destinations at once,
 * as gg_all_gather does.  Same result.  Applies to the tensor-map and bulk
 * paths; the vector path ignores it.
 * ------------------------------------------------------------------------- */
gg_status gg_all_gather_grouped(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                                void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                                gg_tile tile, int comm_programs, gg_group group,
                                int dests_per_wait, int *dev_status, gg_stream_t stream,
                                gg_ag_path path);

/* ---------------------------------------------------------------------------
 * gg_all_gather_partitioned — the same result as gg_all_gather, with the
 * programs partitioned across the destinations (iris PR #626, "Triton CCL
 * all-gather": persistent_all_gather_partitioned): program p serves group
 * member p mod world_size only, and the programs of one destination share
 * all tiles; every tile is therefore read once per destination.  Requires
 * comm_programs >= world_size (else GG_ERR_INVALID_ARG).  path: GG_AG_AUTO,
 * GG_AG_TMA or GG_AG_VECTOR (GG_AG_BULK returns GG_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------- */
gg_status gg_all_gather_partitioned(const gg_heap *heap, int rank, const void *input,
                                    int64_t ld_in, void *output, int64_t ld_out, int64_t M,
                                    int64_t N, gg_dtype dtype, gg_tile tile, int comm_programs,
                                    gg_group group, int *dev_status, gg_stream_t stream,
                                    gg_ag_path path);

/* ---------------------------------------------------------------------------
 * gg_all_to_all — the all-to-all over the same heap (iris #594, "Compiler
 * inspection and grouping", and iris #591, Work: Gluon all_to_all).  Member
 * i's input is world_size*M x N (row pitch ld_in): row block d
 * (rows d*M .. d*M+M-1) is meant for member d.  Member d's output
 * (world_size*M x N, pitch ld_out) receives, in row block i, member i's
 * block d -- torch.distributed.all_to_all_single with equal splits.  Each
 * tile is read once and stored once; every source sends to its destinations
 * in rotated order (its own block first).
 * rank >= 0: only that member's W blocks go out (input: any device memory);
 * rank == -1: every member, input symmetric.  Other arguments, alignment and
 * errors as gg_all_gather; path: GG_AG_AUTO, GG_AG_TMA or GG_AG_VECTOR.
 * ------------------------------------------------------------------------- */
gg_status gg_all_to_all(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                        void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                        gg_tile tile, int comm_programs, gg_group group, int *dev_status,
                        gg_stream_t stream, gg_ag_path path);

/* Collectives of gg_collective_check. */
typedef enum {
    GG_COLL_ALL_GATHER = 0,
    GG_COLL_ALL_GATHER_PARTITIONED = 1,
    GG_COLL_ALL_TO_ALL = 2
} gg_collective;

/* Validate a call of one of the collectives above exactly as the launching
 * call does and launch nothing; *chosen (nullable) receives the path a launch
 * would take (GG_AG_AUTO when there is nothing to launch). */
gg_status gg_collective_check(gg_collective kind, const gg_heap *heap, int rank, const void *input,
                              int64_t ld_in, void *output, int64_t ld_out, int64_t M, int64_t N,
                              gg_dtype dtype, gg_tile tile, int comm_programs, gg_group group,
                              int dests_per_wait, gg_ag_path path, gg_ag_path *chosen);

/* ---------------------------------------------------------------------------
 * gg_matmul_all_gather — the fused form (iris PR #626, "Summary" and
 * "Benchmark": the matmul's epilogue all-gathers each output tile).
 * Member r computes C_r = A_r @ B (A_r: M x K row-major, row pitch lda;
 * B: K x N row-major, row pitch ldb, one buffer shared by all members),
 * accumulating in float32 on the tensor cores, rounds C_r to `dtype`
 * (round to nearest even) and writes it into row block i (its group index)
 * of the world_size*M x N output of every member, local copy first.
 * dtype: GG_F16 or GG_BF16 (A, B and the output share it).
 * rank >= 0: only that member computes and gathers its block; `A` is any
 *   device pointer.  rank == -1: every member, in one launch; `A` is then a
 *   symmetric heap buffer.
 * tile: the output tile of one CTA, exactly as given (never remapped):
 *   {GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N} = 128 x 256: one tcgen05 MMA tile
 *     per CTA, 256 x 256 per CTA pair (or 128 x 256 on the 1-SM path);
 *   {GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N_WIDE} = 128 x 512: two 128 x 256 MMA
 *     tiles side by side per CTA, sharing each A stage, 256 x 512 per CTA
 *     pair; needs the CTA pairs (comm_programs >= 2, not GG_MAG_1SM).  It
 *     reads a quarter fewer operand bytes per MMA and is the faster choice
 *     wherever N is not padded much more by 512-column tiles (N = 3584:
 *     95-98% of cuBLAS's rate on the plain GEMM, against 89-90%).
 *   Anything else returns GG_ERR_UNSUPPORTED.
 * Alignment (GG_ERR_ALIGNMENT otherwise): A, B, output 16-byte aligned;
 *   lda, ldb, ld_out multiples of 8; N a multiple of 8.
 * comm_programs: number of persistent CTAs (one per SM at most is useful).
 *   By default they run as CTA pairs (comm_programs/2 clusters of two CTAs,
 *   each pair on twice the tile's rows); a single program runs alone on
 *   128 x 256 tiles.
 * dev_status: as for gg_all_gather (NULL: the library's status word).
 * M or N == 0: nothing is launched, GG_OK.
 * K == 0: every product is the empty sum, the zero matrix: the call writes
 *   zeros into the gathered rows of its sources (all of them for rank == -1)
 *   in every member's output, padding columns untouched.  A and B are not
 *   read and may be NULL; the output is validated as above.  No matmul
 *   kernel runs (a plain fill).
 * ------------------------------------------------------------------------- */
gg_status gg_matmul_all_gather(const gg_heap *heap, int rank, const void *A, int64_t lda,
                               const void *B, int64_t ldb, void *output, int64_t ld_out,
                               int64_t M, int64_t N, int64_t K, gg_dtype dtype,
                               gg_tile tile, int comm_programs, gg_group group,
                               int *dev_status, gg_stream_t stream);

/* Kernel variants of gg_matmul_all_gather (same arguments and result):
 *   GG_MAG_AUTO  2-SM pairs when comm_programs >= 2, else 1-SM
 *   GG_MAG_1SM   one CTA per 128 x 256 tile (tcgen05.mma.cta_group::1);
 *                GG_ERR_UNSUPPORTED for the 128 x 512 tile
 *   GG_MAG_2SM   a CTA pair per two tiles (tcgen05.mma.cta_group::2);
 *                needs comm_programs >= 2 (else GG_ERR_INVALID_ARG) */
typedef enum { GG_MAG_AUTO = 0, GG_MAG_1SM = 1, GG_MAG_2SM = 2 } gg_mag_path;

gg_status gg_matmul_all_gather_path(const gg_heap *heap, int rank, const void *A, int64_t lda,
                                    const void *B, int64_t ldb, void *output, int64_t ld_out,
                                    int64_t M, int64_t N, int64_t K, gg_dtype dtype, gg_tile tile,
                                    int comm_programs, gg_group group, int *dev_status,
                                    gg_stream_t stream, gg_mag_path path);

/* Validate a gg_matmul_all_gather_path call exactly as the launching call
 * does and launch nothing; *chosen (nullable) receives the kernel variant a
 * launch would run: GG_MAG_1SM (a single program, or asked for) or
 * GG_MAG_2SM; GG_MAG_AUTO when no matmul kernel would run (M or N == 0:
 * nothing; K == 0: the zero fill). */
gg_status gg_matmul_all_gather_plan(const gg_heap *heap, int rank, const void *A, int64_t lda,
                                    const void *B, int64_t ldb, void *output, int64_t ld_out,
                                    int64_t M, int64_t N, int64_t K, gg_dtype dtype,
                                    gg_tile tile, int comm_programs, gg_group group,
                                    gg_mag_path path, gg_mag_path *chosen);

/* Validate a gg_matmul_all_gather call exactly as the launching call does
 * and launch nothing. */
gg_status gg_matmul_all_gather_check(const gg_heap *heap, int rank, const void *A, int64_t lda,
                                     const void *B, int64_t ldb, void *output, int64_t ld_out,
                                     int64_t M, int64_t N, int64_t K, gg_dtype dtype,
                                     gg_tile tile, int comm_programs, gg_group group);

/* ---------------------------------------------------------------------------
 * Bounded waits.  Every wait of a kernel on an mbarrier gives up after this
 * many nanoseconds of wall time (default 2e9), stores GG_ERR_TIMEOUT in the
 * call's dev_status, drains the copies it has in flight and returns.  Applies
 * to launches made after the call, from any thread.  0 restores the default.
 * ------------------------------------------------------------------------- */
gg_status gg_set_wait_limit_ns(uint64_t ns);
uint64_t gg_get_wait_limit_ns(void);

/* The library's status word of the current device: where launches whose
 * caller passed dev_status == NULL store GG_ERR_TIMEOUT when a bounded wait
 * gives up (first error wins; 0 while no such launch stopped early).
 * gg_device_status waits for `stream` to finish the work queued on it so far,
 * then copies the word to *host_out (host memory); gg_clear_device_status
 * enqueues its reset to 0 on `stream`.  Both look the word's address up once
 * per device (cudaGetSymbolAddress, with that device current) at their first
 * use, or at the first launch given no status word; make that first use
 * before any stream capture, and do not use the word on a device after a
 * cudaDeviceReset of it.  Every launch on a device without a status word of
 * its own shares this one word. */
gg_status gg_device_status(gg_stream_t stream, int *host_out);
gg_status gg_clear_device_status(gg_stream_t stream);

/* Test hook for the bounded waits (failure detection without a GPU fault).
 * While enabled, launches of the bulk all-gather path and of the fused
 * kernel leave the first ring stage of program 0 unarmed, so the wait on it
 * can never complete: it runs out after the wait limit, GG_ERR_TIMEOUT lands
 * in the status word and the kernel drains and returns.  Nothing faults or
 * hangs.  Off by default; 0 turns it off. */
gg_status gg_debug_inject_stall(int enable);

/* Message describing the last error returned on this thread ("" if none). */
const char *gg_last_error(void);

/* Short name of a status code. */
const char *gg_status_string(gg_status s);

/* Library version, major*10000 + minor*100 + patch. */
int gg_version(void);

/* ---------------------------------------------------------------------------
 * Tracing: the SM clock a kernel ran at.  The pages have no counterpart
 * (their evidence is the compiler's assembly); here it shows how a kernel's
 * time splits into SM cycles and clock.
 *
 * gg_set_trace(enable): launches after this call (enable != 0) record, from
 * one thread of their first CTA, the wall time (%globaltimer, ns) and the SM
 * cycle counter (clock64) at that CTA's start and end, into the library's
 * trace records of the device: one record for the all-gather family (also
 * gg_all_gather_noalloc), one for gg_matmul_all_gather.  enable == 0 (the
 * default) stops it.  The cost is four 8-byte stores per launch.  The
 * records are shared by every launch on the device, so with launches in
 * flight on several streams the record is the last one written.
 * (end_cycles - start_cycles) * 1e3 / (end_ns - start_ns) is the clock in
 * MHz; the first CTA runs from a kernel's start to about its end.
 *
 * gg_trace_read(stream, gather, fused): copies the two records to the host
 * after stream's queued work (either pointer may be NULL).  A record no
 * traced launch has written holds zeros.  Like the status word, the records'
 * address is looked up once per device and goes stale after a
 * cudaDeviceReset of that device.
 * ------------------------------------------------------------------------- */
typedef struct {
    uint64_t start_ns, start_cycles, end_ns, end_cycles;
} gg_trace_record;

gg_status gg_set_trace(int enable);
gg_status gg_trace_read(gg_stream_t stream, gg_trace_record *gather, gg_trace_record *fused);

/* ---------------------------------------------------------------------------
 * gg_checked_build — 1 in the checked build of the library
 * (libgemm_gather_checked.so), 0 in the release build (libgemm_gather.so).
 * The pages have no counterpart.
 *
 * Both builds export the same calls with the same arguments and results.  The
 * checked build adds device-side checks to the all-gather, partitioned
 * all-gather and all-to-all kernels, for finding a wrong heap-bases table or
 * an indexing fault while developing:
 *  - every program compares the device heap-bases table with the heap's
 *    layout (entry h == partition h's address, as gg_heap_bases reports it);
 *    an entry that differs is reported and not used: the member is reached
 *    at its partition's address, so the results stay those of a correct
 *    table;
 *  - the validated input and output extents must fit inside a partition
 *    (else the launch reports and returns before its first access);
 *  - every decoded work item must lie inside the tile grid, and every load
 *    and store the bulk and vector paths address must lie inside the source
 *    block or the member's gathered output that the host validated (else
 *    that access is skipped).
 * A failed check stores GG_ERR_NOT_IN_HEAP in the launch's status word
 * (dev_status, or the library's word when it is NULL); first error wins, as
 * for GG_ERR_TIMEOUT.  The tensor-map paths and the fused kernels address
 * memory only through tensor maps the host encodes from its own copy of the
 * bases, clipped to the validated extents by the TMA unit: of these checks
 * the tensor-map all-gather paths run the table comparison, the extent check
 * and the item check, the fused kernels none.  The checks cost time: the
 * checked build is not for measurement. */
int gg_checked_build(void);

#ifdef __cplusplus
}
#endif
#endif /* GEMM_GATHER_H */
