// C ABI of gemm_gather: heap handles, argument validation, path selection and
// launches.  Declared in include/gemm_gather.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gemm_gather.h"
#include "gg_internal.h"

struct gg_heap {
    uint64_t base;
    size_t part;
    int H;
    uint64_t *dev_table;
    std::vector<uint64_t> host_bases;
    unsigned long long *work = nullptr;  // workspace slots (claimed-run counters)
    int work_slots = 0;
    mutable std::atomic<uint32_t> work_next{0};  // round-robin slot of the next launch

    unsigned long long *next_work_slot() const
    {
        if (!work)
            return nullptr;
        const uint32_t s = work_next.fetch_add(1, std::memory_order_relaxed) % (uint32_t)work_slots;
        return work + (size_t)s * (GG_WORKSPACE_SLOT_BYTES / sizeof(unsigned long long));
    }
};

static_assert(GG_WORKSPACE_SLOT_BYTES == gg::kWorkSlotBytes, "one counter per workspace slot");
static_assert(GG_CLAIM_AUTO == gg::kClaimAuto && GG_CLAIM_ALWAYS == gg::kClaimAlways &&
                  GG_CLAIM_NEVER == gg::kClaimNever,
              "claim policies");

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_claim_policy{GG_CLAIM_AUTO};
std::atomic<int> g_store_policy{GG_STORE_EVICT_FIRST};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

gg_status fail(gg_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

gg_status ok()
{
    g_last_error.clear();
    return GG_OK;
}

gg_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(GG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int elem_size(gg_dtype d)
{
    switch (d) {
    case GG_F16: return 2;
    case GG_BF16: return 2;
    case GG_F32: return 4;
    }
    return 0;
}

// Group checks shared by every collective; on success *gi is the group index
// of `rank` (or -1 for a launch over all members).
gg_status check_group(const gg_heap *heap, gg_group g, int rank, int *gi)
{
    if (!heap)
        return fail(GG_ERR_INVALID_ARG, "heap is NULL");
    if (g.world_size < 1 || g.world_size > GG_MAX_WORLD)
        return fail(GG_ERR_INVALID_ARG, "world_size %d outside [1, %d]", g.world_size,
                    GG_MAX_WORLD);
    if (g.rank_stride < 1)
        return fail(GG_ERR_INVALID_ARG, "rank_stride %d must be >= 1", g.rank_stride);
    if (g.rank_start < 0)
        return fail(GG_ERR_INVALID_ARG, "rank_start %d must be >= 0", g.rank_start);
    const int64_t last = (int64_t)g.rank_start + (int64_t)(g.world_size - 1) * g.rank_stride;
    if (last >= heap->H)
        return fail(GG_ERR_INVALID_ARG, "group member %lld is not a heap (heaps: %d)",
                    (long long)last, heap->H);
    if (rank == -1) {
        *gi = -1;
        return GG_OK;
    }
    if (rank < 0 || rank >= heap->H)
        return fail(GG_ERR_INVALID_ARG, "rank %d is neither -1 nor a heap index", rank);
    const int d = rank - g.rank_start;
    if (d < 0 || d % g.rank_stride != 0 || d / g.rank_stride >= g.world_size)
        return fail(GG_ERR_INVALID_ARG, "rank %d is not a member of the group (%d, %d, %d)", rank,
                    g.rank_start, g.rank_stride, g.world_size);
    *gi = d / g.rank_stride;
    return GG_OK;
}

// Byte offset of a symmetric buffer within its partition, checking that
// `extent` bytes from there stay inside the partition.
gg_status symmetric_offset(const gg_heap *heap, const void *p, int64_t extent, const char *what,
                           int64_t *off)
{
    const uint64_t a = reinterpret_cast<uint64_t>(p);
    const uint64_t end = heap->base + (uint64_t)heap->part * (uint64_t)heap->H;
    if (a < heap->base || a >= end)
        return fail(GG_ERR_NOT_IN_HEAP, "%s (0x%llx) is not inside the heap", what,
                    (unsigned long long)a);
    const uint64_t o = (a - heap->base) % heap->part;
    if ((uint64_t)extent > heap->part - o)
        return fail(GG_ERR_NOT_IN_HEAP,
                    "%s: %lld bytes at offset %llu overrun the %llu-byte partition", what,
                    (long long)extent, (unsigned long long)o, (unsigned long long)heap->part);
    *off = (int64_t)o;
    return GG_OK;
}

bool overlap(uint64_t a0, uint64_t a1, uint64_t b0, uint64_t b1) { return a0 < b1 && b0 < a1; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool checked_mul(int64_t a, int64_t b, int64_t *out)
{
    if (a != 0 && b > INT64_MAX / a)
        return false;
    *out = a * b;
    return true;
}

// Device address of a file-scope __device__ object on the current device.
// Host code only holds a host-side stand-in for such an object, so its
// device address is looked up (cudaGetSymbolAddress) once per device, with
// that device current, and kept in cache[device].
constexpr int kMaxDevices = 64;

gg_status device_symbol(const void *symbol, void **cache, std::mutex &mu, const char *what,
                        void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(GG_ERR_UNSUPPORTED, "device %d: the library serves devices 0..%d", dev,
                    kMaxDevices - 1);
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, symbol);
        if (e != cudaSuccess)
            return cuda_fail(e, what);
        cache[dev] = p;
    }
    *out = cache[dev];
    return GG_OK;
}

}  // namespace

// The library's own status word (one int per device): launches whose caller
// passes no dev_status report a bounded wait that gave up here, so a launch
// that stopped early never goes unreported.  Read and cleared with
// gg_device_status / gg_clear_device_status.
static __device__ int g_library_status;

namespace {

std::mutex g_status_mu;
void *g_status_ptr[kMaxDevices];

gg_status library_status(int **out)
{
    void *p = nullptr;
    gg_status st = device_symbol(&g_library_status, g_status_ptr, g_status_mu,
                                 "cudaGetSymbolAddress of the library status word", &p);
    *out = static_cast<int *>(p);
    return st;
}

// The status word a launch reports to: the caller's, else the library's.
gg_status resolve_status(int **status)
{
    return *status ? GG_OK : library_status(status);
}

}  // namespace

// The library's trace records (one per device, gg_set_trace): the all-gather
// family's last traced launch in words 0..3, the fused call's in words 4..7.
static __device__ unsigned long long g_trace[gg::kTraceWords];

namespace {

std::mutex g_trace_mu;
void *g_trace_ptr[kMaxDevices];
std::atomic<int> g_trace_on{0};

gg_status trace_records(unsigned long long **out)
{
    void *p = nullptr;
    gg_status st = device_symbol(&g_trace, g_trace_ptr, g_trace_mu,
                                 "cudaGetSymbolAddress of the trace records", &p);
    *out = static_cast<unsigned long long *>(p);
    return st;
}

// The trace record a launch writes: NULL unless tracing is on.
gg_status resolve_trace(unsigned long long **trace, int which)
{
    *trace = nullptr;
    if (!g_trace_on.load(std::memory_order_relaxed))
        return GG_OK;
    unsigned long long *base = nullptr;
    gg_status st = trace_records(&base);
    if (st == GG_OK)
        *trace = base + which;
    return st;
}

}  // namespace

extern "C" {

gg_status gg_heap_wrap(void *dev_base, size_t bytes_per_rank, int num_heaps,
                       uint64_t *dev_bases_table, gg_heap **out)
{
    if (!out)
        return fail(GG_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!dev_base || !dev_bases_table)
        return fail(GG_ERR_INVALID_ARG, "dev_base and dev_bases_table must be non-NULL");
    if (reinterpret_cast<uint64_t>(dev_base) % 256 != 0)
        return fail(GG_ERR_ALIGNMENT, "dev_base must be 256-byte aligned");
    if (reinterpret_cast<uint64_t>(dev_bases_table) % 8 != 0)
        return fail(GG_ERR_ALIGNMENT, "dev_bases_table must be 8-byte aligned");
    if (bytes_per_rank == 0 || bytes_per_rank % 256 != 0)
        return fail(GG_ERR_INVALID_ARG, "bytes_per_rank must be a positive multiple of 256");
    if (num_heaps < 1 || num_heaps > GG_MAX_HEAPS)
        return fail(GG_ERR_INVALID_ARG, "num_heaps %d outside [1, %d]", num_heaps, GG_MAX_HEAPS);
    gg_heap *h = new gg_heap;
    h->base = reinterpret_cast<uint64_t>(dev_base);
    h->part = bytes_per_rank;
    h->H = num_heaps;
    h->dev_table = dev_bases_table;
    h->host_bases.resize(num_heaps);
    for (int i = 0; i < num_heaps; ++i)
        h->host_bases[i] = h->base + (uint64_t)i * bytes_per_rank;
    *out = h;
    return ok();
}

gg_status gg_heap_create(void *dev_base, size_t bytes_per_rank, int num_heaps,
                         uint64_t *dev_bases_table, gg_stream_t stream, gg_heap **out)
{
    gg_status st = gg_heap_wrap(dev_base, bytes_per_rank, num_heaps, dev_bases_table, out);
    if (st != GG_OK)
        return st;
    gg_heap *h = *out;
    cudaError_t e = cudaMemcpyAsync(dev_bases_table, h->host_bases.data(),
                                    sizeof(uint64_t) * num_heaps, cudaMemcpyHostToDevice,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        delete h;
        *out = nullptr;
        return cuda_fail(e, "writing the heap-bases table");
    }
    return ok();
}

gg_status gg_heap_bases(const gg_heap *heap, uint64_t *host_out, int n)
{
    if (!heap || !host_out)
        return fail(GG_ERR_INVALID_ARG, "heap and host_out must be non-NULL");
    if (n < 0 || n > heap->H)
        return fail(GG_ERR_INVALID_ARG, "n %d outside [0, %d]", n, heap->H);
    std::copy(heap->host_bases.begin(), heap->host_bases.begin() + n, host_out);
    return ok();
}

gg_status gg_heap_info(const gg_heap *heap, int *num_heaps, size_t *bytes_per_rank)
{
    if (!heap)
        return fail(GG_ERR_INVALID_ARG, "heap is NULL");
    if (num_heaps)
        *num_heaps = heap->H;
    if (bytes_per_rank)
        *bytes_per_rank = heap->part;
    return ok();
}

gg_status gg_heap_destroy(gg_heap *heap)
{
    delete heap;
    return ok();
}

gg_status gg_heap_set_workspace(gg_heap *heap, void *dev_work, size_t bytes)
{
    if (!heap)
        return fail(GG_ERR_INVALID_ARG, "heap is NULL");
    if (!dev_work || bytes == 0) {
        if (dev_work || bytes)
            return fail(GG_ERR_INVALID_ARG, "a workspace needs both a pointer and a size");
        heap->work = nullptr;
        heap->work_slots = 0;
        return ok();
    }
    if (reinterpret_cast<uint64_t>(dev_work) % 256 != 0)
        return fail(GG_ERR_ALIGNMENT, "the workspace must be 256-byte aligned");
    if (bytes % GG_WORKSPACE_SLOT_BYTES != 0 || bytes / GG_WORKSPACE_SLOT_BYTES > (1u << 20))
        return fail(GG_ERR_INVALID_ARG,
                    "workspace bytes %zu: a multiple of %d, at most 2^20 slots", bytes,
                    GG_WORKSPACE_SLOT_BYTES);
    heap->work = static_cast<unsigned long long *>(dev_work);
    heap->work_slots = (int)(bytes / GG_WORKSPACE_SLOT_BYTES);
    return ok();
}

}  // extern "C"

namespace {

// Validation and argument set-up of a gather; *launch is false when there is
// nothing to do (M == 0 or N == 0).
// Data path a gather launch takes.
enum GatherKind { kVector = 0, kBulk = 1, kTma = 2 };

gg_status prepare_gather(const gg_heap *heap, int mode, int rank, const void *input,
                         int64_t ld_in, void *output, int64_t ld_out, int64_t M, int64_t N,
                         gg_dtype dtype, gg_tile tile, int comm_programs, gg_group group,
                         int dests_per_wait, int *dev_status, gg_ag_path path,
                         gg::GatherArgs *out_args, int *kind, int *vec_bytes, CUtensorMap *in_map,
                         gg::OutMaps *maps, bool *launch)
{
    *launch = false;
    int gi = -1;
    gg_status st = check_group(heap, group, rank, &gi);
    if (st != GG_OK)
        return st;
    const int es = elem_size(dtype);
    if (es == 0)
        return fail(GG_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (path != GG_AG_AUTO && path != GG_AG_BULK && path != GG_AG_VECTOR && path != GG_AG_TMA)
        return fail(GG_ERR_INVALID_ARG, "unknown path %d", (int)path);
    if (M < 0 || N < 0)
        return fail(GG_ERR_INVALID_ARG, "M and N must be >= 0");
    if (ld_in < N || ld_out < N)
        return fail(GG_ERR_INVALID_ARG, "ld_in (%lld) and ld_out (%lld) must be >= N (%lld)",
                    (long long)ld_in, (long long)ld_out, (long long)N);
    if (tile.block_m < 1 || tile.block_m > 256 || tile.block_n < 1)
        return fail(GG_ERR_UNSUPPORTED,
                    "tile %dx%d: block_m must be in [1, 256] and block_n >= 1 (tiles are never "
                    "remapped)",
                    tile.block_m, tile.block_n);
    if ((int64_t)tile.block_m * tile.block_n * es > 32768)
        return fail(GG_ERR_UNSUPPORTED,
                    "tile %dx%d of %d-byte elements exceeds 32768 bytes (tiles are never remapped)",
                    tile.block_m, tile.block_n, es);
    if (comm_programs < 1 || comm_programs > 65535)
        return fail(GG_ERR_INVALID_ARG, "comm_programs %d outside [1, 65535]", comm_programs);
    if (dests_per_wait < 0)
        return fail(GG_ERR_INVALID_ARG, "dests_per_wait %d must be >= 0", dests_per_wait);
    if (mode == gg::kModePartitioned && comm_programs < group.world_size)
        return fail(GG_ERR_INVALID_ARG,
                    "the partitioned all-gather needs comm_programs (%d) >= world_size (%d): one "
                    "destination per program",
                    comm_programs, group.world_size);
    if (mode != gg::kModeGather && path == GG_AG_BULK)
        return fail(GG_ERR_UNSUPPORTED,
                    "the partitioned all-gather and the all-to-all run the tensor-map or the "
                    "vector path");
    if (!output || (!input && M > 0 && N > 0))
        return fail(GG_ERR_INVALID_ARG, "input and output must be non-NULL");
    if (M == 0 || N == 0)
        return ok();

    const int W = group.world_size;
    // the all-to-all input holds W row blocks (one per destination)
    const int64_t in_rows = mode == gg::kModeAllToAll ? (int64_t)W * M : M;
    int64_t rows_out, out_ext, in_ext, tmp;
    if (!checked_mul(W, M, &rows_out) || !checked_mul(rows_out - 1, ld_out, &tmp) ||
        !checked_mul(tmp + N, es, &out_ext) || !checked_mul(in_rows - 1, ld_in, &tmp) ||
        !checked_mul(tmp + N, es, &in_ext))
        return fail(GG_ERR_INVALID_ARG, "sizes overflow");
    int64_t out_off = 0;
    st = symmetric_offset(heap, output, out_ext, "output", &out_off);
    if (st != GG_OK)
        return st;

    gg::GatherArgs a{};
    a.bases = heap->dev_table;
    a.heap_lo = heap->base;
    a.part_bytes = (uint64_t)heap->part;
    a.in_ext_b = in_ext;
    a.out_ext_b = out_ext;
    a.W = W;
    a.rank_start = group.rank_start;
    a.rank_stride = group.rank_stride;
    uint64_t in_align;
    if (rank == -1) {
        int64_t in_off;
        st = symmetric_offset(heap, input, in_ext, "input", &in_off);
        if (st != GG_OK)
            return st;
        if (overlap(in_off, in_off + in_ext, out_off, out_off + out_ext))
            return fail(GG_ERR_INVALID_ARG, "input and output overlap inside the partition");
        a.n_src = W;
        a.src_first = 0;
        a.in_abs = nullptr;
        a.in_off = in_off;
        in_align = (uint64_t)in_off;
    } else {
        const uint64_t i0 = reinterpret_cast<uint64_t>(input);
        for (int q = 0; q < W; ++q) {
            const uint64_t o0 = heap->host_bases[group.rank_start + q * group.rank_stride] + out_off;
            if (overlap(i0, i0 + in_ext, o0, o0 + out_ext))
                return fail(GG_ERR_INVALID_ARG, "input overlaps the output of member %d", q);
        }
        a.n_src = 1;
        a.src_first = gi;
        a.in_abs = static_cast<const uint8_t *>(input);
        a.in_off = 0;
        in_align = i0;
    }
    a.out_off = out_off;
    a.ld_in_b = ld_in * es;
    a.ld_out_b = ld_out * es;
    a.M = M;
    a.row_b = N * es;
    a.bm = tile.block_m;
    a.bn_b = (int64_t)tile.block_n * es;
    a.tiles_n = ceil_div(N, tile.block_n);
    a.tiles_per_src = ceil_div(M, tile.block_m) * a.tiles_n;
    a.total_items = a.tiles_per_src * a.n_src * (mode == gg::kModeAllToAll ? W : 1);
    a.es = es;
    a.mode = mode;
    a.dests_per_wait = dests_per_wait;
    a.status = dev_status;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.inject_stall = g_inject_stall.load();
    a.work = nullptr;  // a slot is taken at launch time
    a.chunk = 0;
    a.claim_policy = g_claim_policy.load();
    a.store_hint = g_store_policy.load() == GG_STORE_EVICT_FIRST ? gg::kStoreEvictFirst
                                                                 : gg::kStorePlain;

    // widest power-of-two granule dividing every address, pitch and length
    uint64_t g = in_align | (uint64_t)out_off | (uint64_t)a.ld_in_b | (uint64_t)a.ld_out_b |
                 (uint64_t)a.bn_b | (uint64_t)a.row_b | 16u;
    const int granule = (int)(g & (~g + 1));  // lowest set bit, <= 16
    const bool bulk_ok = granule == 16;
    // tensor maps: 16-byte aligned bases and pitches, a box of at most 256 x 256
    // elements whose rows are whole 16-byte units (N itself may be ragged)
    const bool tma_ok = ((in_align | (uint64_t)out_off | (uint64_t)a.ld_in_b |
                          (uint64_t)a.ld_out_b | (uint64_t)a.bn_b) % 16 == 0) &&
                        tile.block_n <= 256 && tile.block_m <= 256;
    if (path == GG_AG_BULK && !bulk_ok)
        return fail(GG_ERR_ALIGNMENT,
                    "bulk path needs 16-byte aligned input, output, pitches, block_n and N "
                    "(in bytes)");
    if (path == GG_AG_TMA && !tma_ok)
        return fail(GG_ERR_ALIGNMENT,
                    "tensor-map path needs 16-byte aligned input, output, pitches and "
                    "block_n*elem_size, and block_n <= 256");
    int k;
    if (path == GG_AG_TMA || (path == GG_AG_AUTO && tma_ok))
        k = kTma;
    else if (path == GG_AG_BULK || (path == GG_AG_AUTO && bulk_ok && mode == gg::kModeGather))
        k = kBulk;
    else
        k = kVector;
    *kind = k;
    *vec_bytes = granule;
    if (k == kTma && in_map && maps) {
        const CUtensorMapDataType dt =
            es == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
        const void *ibase = rank == -1 ? reinterpret_cast<const void *>(heap->base + a.in_off)
                                       : input;
        const uint64_t whole = (uint64_t)(in_rows * a.ld_in_b);  // one source's input
        bool enc;
        if (mode == gg::kModeAllToAll) {
            // sources as {N, M, W blocks, heaps}: a tile clips at the end of its block
            const uint32_t box[4] = {(uint32_t)tile.block_n, (uint32_t)tile.block_m, 1, 1};
            const uint64_t dims[4] = {(uint64_t)N, (uint64_t)M, (uint64_t)W,
                                      (uint64_t)(rank == -1 ? heap->H : 1)};
            const uint64_t strides[3] = {(uint64_t)a.ld_in_b, (uint64_t)(M * a.ld_in_b),
                                         rank == -1 ? (uint64_t)heap->part : whole};
            enc = gg::encode_map(in_map, dt, 4, ibase, dims, strides, box,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
        } else {
            const uint32_t box[3] = {(uint32_t)tile.block_n, (uint32_t)tile.block_m, 1};
            const uint64_t dims[3] = {(uint64_t)N, (uint64_t)M,
                                      (uint64_t)(rank == -1 ? heap->H : 1)};
            const uint64_t strides[2] = {(uint64_t)a.ld_in_b,
                                         rank == -1 ? (uint64_t)heap->part : whole};
            enc = gg::encode_map(in_map, dt, 3, ibase, dims, strides, box,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
        }
        if (!enc)
            return fail(GG_ERR_CUDA, "encoding the input tensor map");
        uint64_t member_out[GG_MAX_WORLD];
        for (int q = 0; q < W; ++q)
            member_out[q] = heap->host_bases[group.rank_start + q * group.rank_stride] +
                            (uint64_t)out_off;
        if (!gg::encode_out_maps(maps, member_out, W, M, N, a.ld_out_b, es,
                                 (uint32_t)tile.block_n, (uint32_t)tile.block_m, dt,
                                 CU_TENSOR_MAP_SWIZZLE_NONE))
            return fail(GG_ERR_CUDA, "encoding the output tensor maps");
    }
    *out_args = a;
    *launch = true;
    return ok();
}

}  // namespace

extern "C" {

// Validate, build and launch one collective of the gather kernels.
gg_status run_collective(const gg_heap *heap, int mode, int rank, const void *input, int64_t ld_in,
                         void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                         gg_tile tile, int comm_programs, gg_group group, int dests_per_wait,
                         int *dev_status, gg_stream_t stream, gg_ag_path path)
{
    gg::GatherArgs a;
    int kind = kVector, vec = 0;
    bool launch = false;
    static thread_local CUtensorMap in_map;
    static thread_local gg::OutMaps maps;
    gg_status st = prepare_gather(heap, mode, rank, input, ld_in, output, ld_out, M, N, dtype, tile,
                                  comm_programs, group, dests_per_wait, dev_status, path, &a, &kind,
                                  &vec, &in_map, &maps, &launch);
    if (st != GG_OK || !launch)
        return st;
    st = resolve_status(&a.status);
    if (st == GG_OK)
        st = resolve_trace(&a.trace, gg::kTraceGather);
    if (st != GG_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // a workspace slot for launches that may claim runs (see prepare_claims)
    if (kind == kTma && mode != gg::kModePartitioned && a.claim_policy != GG_CLAIM_NEVER)
        a.work = heap->next_work_slot();
    cudaError_t e;
    if (kind == kTma)
        e = gg::launch_gather_tma(in_map, maps, a, comm_programs, s);
    else if (kind == kBulk)
        e = gg::launch_gather_bulk(a, comm_programs, s);
    else
        e = gg::launch_gather_vec(a, comm_programs, vec, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the collective");
    return ok();
}

gg_status gg_all_gather_path(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                             void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                             gg_tile tile, int comm_programs, gg_group group, int *dev_status,
                             gg_stream_t stream, gg_ag_path path)
{
    return run_collective(heap, gg::kModeGather, rank, input, ld_in, output, ld_out, M, N, dtype,
                          tile, comm_programs, group, 0, dev_status, stream, path);
}

gg_status gg_all_gather_grouped(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                                void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                                gg_tile tile, int comm_programs, gg_group group,
                                int dests_per_wait, int *dev_status, gg_stream_t stream,
                                gg_ag_path path)
{
    return run_collective(heap, gg::kModeGather, rank, input, ld_in, output, ld_out, M, N, dtype,
                          tile, comm_programs, group, dests_per_wait, dev_status, stream, path);
}

gg_status gg_all_gather_partitioned(const gg_heap *heap, int rank, const void *input,
                                    int64_t ld_in, void *output, int64_t ld_out, int64_t M,
                                    int64_t N, gg_dtype dtype, gg_tile tile, int comm_programs,
                                    gg_group group, int *dev_status, gg_stream_t stream,
                                    gg_ag_path path)
{
    return run_collective(heap, gg::kModePartitioned, rank, input, ld_in, output, ld_out, M, N,
                          dtype, tile, comm_programs, group, 0, dev_status, stream, path);
}

gg_status gg_all_to_all(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                        void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                        gg_tile tile, int comm_programs, gg_group group, int *dev_status,
                        gg_stream_t stream, gg_ag_path path)
{
    return run_collective(heap, gg::kModeAllToAll, rank, input, ld_in, output, ld_out, M, N, dtype,
                          tile, comm_programs, group, 0, dev_status, stream, path);
}

gg_status gg_collective_check(gg_collective kind, const gg_heap *heap, int rank, const void *input,
                              int64_t ld_in, void *output, int64_t ld_out, int64_t M, int64_t N,
                              gg_dtype dtype, gg_tile tile, int comm_programs, gg_group group,
                              int dests_per_wait, gg_ag_path path, gg_ag_path *chosen)
{
    if (kind != GG_COLL_ALL_GATHER && kind != GG_COLL_ALL_GATHER_PARTITIONED &&
        kind != GG_COLL_ALL_TO_ALL)
        return fail(GG_ERR_INVALID_ARG, "unknown collective %d", (int)kind);
    const int mode = kind == GG_COLL_ALL_GATHER
                         ? gg::kModeGather
                         : (kind == GG_COLL_ALL_TO_ALL ? gg::kModeAllToAll : gg::kModePartitioned);
    gg::GatherArgs a;
    int k = kVector, vec = 0;
    bool launch = false;
    gg_status st = prepare_gather(heap, mode, rank, input, ld_in, output, ld_out, M, N, dtype, tile,
                                  comm_programs, group, dests_per_wait, nullptr, path, &a, &k, &vec,
                                  nullptr, nullptr, &launch);
    if (chosen)
        *chosen = !launch ? GG_AG_AUTO
                          : (k == kTma ? GG_AG_TMA : (k == kBulk ? GG_AG_BULK : GG_AG_VECTOR));
    return st;
}

gg_status gg_all_gather_check(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                              void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                              gg_tile tile, int comm_programs, gg_group group, gg_ag_path path,
                              gg_ag_path *chosen)
{
    return gg_collective_check(GG_COLL_ALL_GATHER, heap, rank, input, ld_in, output, ld_out, M, N,
                               dtype, tile, comm_programs, group, 0, path, chosen);
}

gg_status gg_all_gather(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                        void *output, int64_t ld_out, int64_t M, int64_t N, gg_dtype dtype,
                        gg_tile tile, int comm_programs, gg_group group, int *dev_status,
                        gg_stream_t stream)
{
    return gg_all_gather_path(heap, rank, input, ld_in, output, ld_out, M, N, dtype, tile,
                              comm_programs, group, dev_status, stream, GG_AG_AUTO);
}

}  // extern "C"

namespace {

// Path checks of the fused calls (before the argument checks of prepare_fused).
gg_status check_fused_path(gg_mag_path path, gg_tile tile, int comm_programs)
{
    if (path != GG_MAG_AUTO && path != GG_MAG_1SM && path != GG_MAG_2SM)
        return fail(GG_ERR_INVALID_ARG, "unknown fused path %d", (int)path);
    if (path == GG_MAG_2SM && comm_programs < 2)
        return fail(GG_ERR_INVALID_ARG, "the 2-SM path needs comm_programs >= 2 (one CTA pair)");
    if (tile.block_m == GG_FUSED_BLOCK_M && tile.block_n == GG_FUSED_BLOCK_N_WIDE) {
        if (path == GG_MAG_1SM)
            return fail(GG_ERR_UNSUPPORTED, "the %dx%d tile runs on CTA pairs only, not the 1-SM "
                        "path (tiles are never remapped)", GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N_WIDE);
        if (comm_programs < 2)
            return fail(GG_ERR_INVALID_ARG, "the %dx%d tile needs comm_programs >= 2 (one CTA "
                        "pair)", GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N_WIDE);
    }
    return GG_OK;
}

// What a validated fused call runs.
enum FusedWork { kFusedNothing = 0, kFusedMatmul = 1, kFusedZeros = 2 };

// Validation and argument set-up of a fused call.  *work: nothing (M == 0 or
// N == 0), the matmul kernel (*out_args, *maps), or, for K == 0, the zero
// fill of the gathered rows (*zeros).  maps and zeros may be NULL (checks).
gg_status prepare_fused(const gg_heap *heap, int rank, const void *A, int64_t lda, const void *B,
                        int64_t ldb, void *output, int64_t ld_out, int64_t M, int64_t N,
                        int64_t K, gg_dtype dtype, gg_tile tile, int comm_programs,
                        gg_group group, int *dev_status, gg::FusedArgs *out_args,
                        gg::OutMaps *maps, gg::ZeroArgs *zeros, FusedWork *work)
{
    *work = kFusedNothing;
    int gi = -1;
    gg_status st = check_group(heap, group, rank, &gi);
    if (st != GG_OK)
        return st;
    if (dtype != GG_F16 && dtype != GG_BF16)
        return fail(GG_ERR_UNSUPPORTED, "matmul_all_gather takes GG_F16 or GG_BF16");
    if (tile.block_m != GG_FUSED_BLOCK_M ||
        (tile.block_n != GG_FUSED_BLOCK_N && tile.block_n != GG_FUSED_BLOCK_N_WIDE))
        return fail(GG_ERR_UNSUPPORTED,
                    "fused tile %dx%d is not supported; the library runs %dx%d and %dx%d (tiles are "
                    "never remapped)",
                    tile.block_m, tile.block_n, GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N,
                    GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N_WIDE);
    if (M < 0 || N < 0 || K < 0)
        return fail(GG_ERR_INVALID_ARG, "M, N and K must be >= 0");
    if (lda < K || ldb < N || ld_out < N)
        return fail(GG_ERR_INVALID_ARG, "lda >= K, ldb >= N and ld_out >= N are required");
    if (comm_programs < 1 || comm_programs > 65535)
        return fail(GG_ERR_INVALID_ARG, "comm_programs %d outside [1, 65535]", comm_programs);
    if (!output || ((!A || !B) && M > 0 && N > 0 && K > 0))
        return fail(GG_ERR_INVALID_ARG, "A, B and output must be non-NULL");
    if (M == 0 || N == 0)
        return ok();
    const uint64_t ua = reinterpret_cast<uint64_t>(A), ub = reinterpret_cast<uint64_t>(B),
                   uo = reinterpret_cast<uint64_t>(output);
    // with K == 0 the operands are never read (every product is the empty sum)
    const uint64_t operands = K > 0 ? (ua | ub) : 0;
    if ((operands | uo) % 16 != 0 || (K > 0 && (lda % 8 || ldb % 8)) || ld_out % 8 || N % 8)
        return fail(GG_ERR_ALIGNMENT,
                    "A, B and output must be 16-byte aligned; lda, ldb, ld_out and N multiples "
                    "of 8");
    if (K > (int64_t)1 << 31 || M > (int64_t)1 << 31 || N > (int64_t)1 << 31)
        return fail(GG_ERR_UNSUPPORTED, "M, N and K must be below 2^31");
    const int W = group.world_size;
    const int64_t out_ext = ((W * M - 1) * ld_out + N) * 2;
    const int64_t a_ext = ((M - 1) * lda + K) * 2;
    int64_t out_off;
    st = symmetric_offset(heap, output, out_ext, "output", &out_off);
    if (st != GG_OK)
        return st;
    if (K == 0) {
        // C_r = A_r @ B over an empty k range is the zero matrix: the gathered
        // rows of the call's sources become zeros in every member's output
        if (zeros) {
            for (int q = 0; q < W; ++q)
                zeros->out[q] =
                    heap->host_bases[group.rank_start + q * group.rank_stride] + (uint64_t)out_off;
            zeros->W = W;
            zeros->src_first = rank == -1 ? 0 : gi;
            zeros->n_src = rank == -1 ? W : 1;
            zeros->M = M;
            zeros->ld_out_b = ld_out * 2;
            zeros->row_b = N * 2;
        }
        *work = kFusedZeros;
        return ok();
    }

    gg::FusedArgs f{};
    f.W = W;
    f.rank_start = group.rank_start;
    f.rank_stride = group.rank_stride;
    f.b = B;
    f.lda = lda;
    f.ldb = ldb;
    f.out_off = out_off;
    f.ld_out = ld_out;
    f.M = M;
    f.N = N;
    f.K = K;
    f.is_bf16 = dtype == GG_BF16;
    f.wide = tile.block_n == GG_FUSED_BLOCK_N_WIDE;
    f.heap_base = heap->base;
    f.part_bytes = heap->part;
    f.num_heaps = heap->H;
    f.status = dev_status;
    f.wait_limit_ns = g_wait_limit_ns.load();
    f.inject_stall = g_inject_stall.load();
    const uint64_t b_ext = (uint64_t)(((K - 1) * ldb + N) * 2);
    if (rank == -1) {
        int64_t a_off;
        st = symmetric_offset(heap, A, a_ext, "A", &a_off);
        if (st != GG_OK)
            return st;
        if (overlap(a_off, a_off + a_ext, out_off, out_off + out_ext))
            return fail(GG_ERR_INVALID_ARG, "A and the output overlap inside the partition");
        f.n_src = W;
        f.src_first = 0;
        f.a_abs = nullptr;
        f.a_off = a_off;
    } else {
        for (int q = 0; q < W; ++q) {
            const uint64_t o0 = heap->host_bases[group.rank_start + q * group.rank_stride] + out_off;
            if (overlap(ua, ua + a_ext, o0, o0 + out_ext))
                return fail(GG_ERR_INVALID_ARG, "A overlaps the output of member %d", q);
        }
        f.n_src = 1;
        f.src_first = gi;
        f.a_abs = A;
        f.a_off = 0;
    }
    for (int q = 0; q < W; ++q) {
        const uint64_t o0 = heap->host_bases[group.rank_start + q * group.rank_stride] + out_off;
        if (overlap(ub, ub + b_ext, o0, o0 + out_ext))
            return fail(GG_ERR_INVALID_ARG, "B overlaps the output of member %d", q);
    }
    if (maps) {
        // the per-peer translation, once per launch: member d's output address
        uint64_t member_out[GG_MAX_WORLD];
        for (int q = 0; q < W; ++q)
            member_out[q] = heap->host_bases[group.rank_start + q * group.rank_stride] +
                            (uint64_t)out_off;
        const CUtensorMapDataType dt =
            dtype == GG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (!gg::encode_out_maps(maps, member_out, W, M, N, ld_out * 2, 2, 64, 32, dt,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
            return fail(GG_ERR_CUDA, "encoding the output tensor maps");
    }
    *out_args = f;
    *work = kFusedMatmul;
    return ok();
}

}  // namespace

extern "C" {

gg_status gg_matmul_all_gather_path(const gg_heap *heap, int rank, const void *A, int64_t lda,
                                    const void *B, int64_t ldb, void *output, int64_t ld_out,
                                    int64_t M, int64_t N, int64_t K, gg_dtype dtype, gg_tile tile,
                                    int comm_programs, gg_group group, int *dev_status,
                                    gg_stream_t stream, gg_mag_path path)
{
    gg_status st = check_fused_path(path, tile, comm_programs);
    if (st != GG_OK)
        return st;
    gg::FusedArgs f;
    static thread_local gg::OutMaps maps;
    gg::ZeroArgs zeros;
    FusedWork work = kFusedNothing;
    st = prepare_fused(heap, rank, A, lda, B, ldb, output, ld_out, M, N, K, dtype, tile,
                       comm_programs, group, dev_status, &f, &maps, &zeros, &work);
    if (st != GG_OK || work == kFusedNothing)
        return st;
    if (work == kFusedZeros) {
        const cudaError_t e =
            gg::launch_zero_rows(zeros, comm_programs, reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? ok() : cuda_fail(e, "launching the zero fill (K == 0)");
    }
    st = resolve_status(&f.status);
    if (st == GG_OK)
        st = resolve_trace(&f.trace, gg::kTraceFused);
    if (st != GG_OK)
        return st;
    const char *why = nullptr;
    cudaError_t e = gg::launch_matmul_all_gather(f, maps, comm_programs, (int)path,
                                                 reinterpret_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess)
        return why ? fail(GG_ERR_CUDA, "%s: %s", why, cudaGetErrorName(e))
                   : cuda_fail(e, "launching matmul_all_gather");
    return ok();
}

gg_status gg_matmul_all_gather(const gg_heap *heap, int rank, const void *A, int64_t lda,
                               const void *B, int64_t ldb, void *output, int64_t ld_out,
                               int64_t M, int64_t N, int64_t K, gg_dtype dtype, gg_tile tile,
                               int comm_programs, gg_group group, int *dev_status,
                               gg_stream_t stream)
{
    return gg_matmul_all_gather_path(heap, rank, A, lda, B, ldb, output, ld_out, M, N, K, dtype,
                                     tile, comm_programs, group, dev_status, stream, GG_MAG_AUTO);
}

gg_status gg_matmul_all_gather_check(const gg_heap *heap, int rank, const void *A, int64_t lda,
                                     const void *B, int64_t ldb, void *output, int64_t ld_out,
                                     int64_t M, int64_t N, int64_t K, gg_dtype dtype,
                                     gg_tile tile, int comm_programs, gg_group group)
{
    gg_status st = check_fused_path(GG_MAG_AUTO, tile, comm_programs);
    if (st != GG_OK)
        return st;
    gg::FusedArgs f;
    FusedWork work = kFusedNothing;
    return prepare_fused(heap, rank, A, lda, B, ldb, output, ld_out, M, N, K, dtype, tile,
                         comm_programs, group, nullptr, &f, nullptr, nullptr, &work);
}

gg_status gg_matmul_all_gather_plan(const gg_heap *heap, int rank, const void *A, int64_t lda,
                                    const void *B, int64_t ldb, void *output, int64_t ld_out,
                                    int64_t M, int64_t N, int64_t K, gg_dtype dtype, gg_tile tile,
                                    int comm_programs, gg_group group, gg_mag_path path,
                                    gg_mag_path *chosen)
{
    if (chosen)
        *chosen = GG_MAG_AUTO;
    gg_status st = check_fused_path(path, tile, comm_programs);
    if (st != GG_OK)
        return st;
    gg::FusedArgs f;
    FusedWork work = kFusedNothing;
    st = prepare_fused(heap, rank, A, lda, B, ldb, output, ld_out, M, N, K, dtype, tile,
                       comm_programs, group, nullptr, &f, nullptr, nullptr, &work);
    if (st == GG_OK && work == kFusedMatmul && chosen)
        *chosen = (gg_mag_path)gg::fused_variant(comm_programs, (int)path);
    return st;
}

gg_status gg_set_wait_limit_ns(uint64_t ns)
{
    g_wait_limit_ns.store(ns == 0 ? kDefaultWaitNs : ns);
    return ok();
}

uint64_t gg_get_wait_limit_ns(void) { return g_wait_limit_ns.load(); }

gg_status gg_set_claim_policy(int policy)
{
    if (policy != GG_CLAIM_AUTO && policy != GG_CLAIM_ALWAYS && policy != GG_CLAIM_NEVER)
        return fail(GG_ERR_INVALID_ARG, "unknown claim policy %d", policy);
    g_claim_policy.store(policy);
    return ok();
}

int gg_get_claim_policy(void) { return g_claim_policy.load(); }

gg_status gg_set_store_policy(int policy)
{
    if (policy != GG_STORE_PLAIN && policy != GG_STORE_EVICT_FIRST)
        return fail(GG_ERR_INVALID_ARG, "unknown store policy %d", policy);
    g_store_policy.store(policy);
    return ok();
}

int gg_get_store_policy(void) { return g_store_policy.load(); }

gg_status gg_debug_inject_stall(int enable)
{
    g_inject_stall.store(enable ? 1 : 0);
    return ok();
}

gg_status gg_device_status(gg_stream_t stream, int *host_out)
{
    if (!host_out)
        return fail(GG_ERR_INVALID_ARG, "host_out is NULL");
    int *word = nullptr;
    gg_status st = library_status(&word);
    if (st != GG_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_out, word, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the library status word");
    return ok();
}

gg_status gg_clear_device_status(gg_stream_t stream)
{
    int *word = nullptr;
    gg_status st = library_status(&word);
    if (st != GG_OK)
        return st;
    cudaError_t e = cudaMemsetAsync(word, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "clearing the library status word");
    return ok();
}

gg_status gg_set_trace(int enable)
{
    g_trace_on.store(enable ? 1 : 0);
    return ok();
}

gg_status gg_trace_read(gg_stream_t stream, gg_trace_record *gather, gg_trace_record *fused)
{
    static_assert(sizeof(gg_trace_record) == 4 * sizeof(unsigned long long), "record layout");
    unsigned long long *rec = nullptr;
    gg_status st = trace_records(&rec);
    if (st != GG_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long host[gg::kTraceWords];
    cudaError_t e = cudaMemcpyAsync(host, rec, sizeof(host), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the trace records");
    if (gather)
        memcpy(gather, host + gg::kTraceGather, sizeof(*gather));
    if (fused)
        memcpy(fused, host + gg::kTraceFused, sizeof(*fused));
    return ok();
}

const char *gg_last_error(void) { return g_last_error.c_str(); }

const char *gg_status_string(gg_status s)
{
    switch (s) {
    case GG_OK: return "GG_OK";
    case GG_ERR_INVALID_ARG: return "GG_ERR_INVALID_ARG";
    case GG_ERR_ALIGNMENT: return "GG_ERR_ALIGNMENT";
    case GG_ERR_NOT_IN_HEAP: return "GG_ERR_NOT_IN_HEAP";
    case GG_ERR_UNSUPPORTED: return "GG_ERR_UNSUPPORTED";
    case GG_ERR_CUDA: return "GG_ERR_CUDA";
    case GG_ERR_TIMEOUT: return "GG_ERR_TIMEOUT";
    }
    return "GG_UNKNOWN";
}

int gg_version(void) { return 100; }

#ifndef GG_CHECKED
#define GG_CHECKED 0
#endif
int gg_checked_build(void) { return GG_CHECKED ? 1 : 0; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free all-gather (gg_all_gather_noalloc).
//
// For callers that cannot allocate device memory at all (no cudaMalloc, no
// allocator of their own to carve a workspace from), the claim counter of the
// load-balanced tensor-map path lives in this file-scope device array instead
// of a heap workspace.  It is a single region shared by every call on a
// device, and holds the last call's counter until the next claiming call
// zeroes it: prepare_claims (ag_kernels.cu) enqueues that memset on the
// call's stream before the kernel, for a workspace slot and for this array
// alike.  Every GPU that loads the library keeps these bytes until the
// process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned long long g_noalloc_scratch[kNoAllocScratchBytes / 8];
static_assert(sizeof(unsigned long long) <= kNoAllocScratchBytes,
              "a call needs one claim counter, whatever its sizes");

namespace {

std::mutex g_noalloc_mu;
void *g_noalloc_dev_ptr[kMaxDevices];

// Device address of the scratch array on the current device: looked up at the
// first call on each device (with that device current), then reused.
gg_status noalloc_scratch(unsigned long long **out)
{
    void *p = nullptr;
    gg_status st = device_symbol(g_noalloc_scratch, g_noalloc_dev_ptr, g_noalloc_mu,
                                 "cudaGetSymbolAddress of the static scratch array", &p);
    *out = static_cast<unsigned long long *>(p);
    return st;
}

}  // namespace

extern "C" {

gg_status gg_all_gather_noalloc(const gg_heap *heap, int rank, const void *input, int64_t ld_in,
                                void *output, int64_t ld_out, int64_t M, int64_t N,
                                gg_dtype dtype, gg_tile tile, int comm_programs, gg_group group,
                                int *dev_status, gg_stream_t stream)
{
    unsigned long long *scratch = nullptr;
    gg_status st = noalloc_scratch(&scratch);  // first call on a device: set-up
    if (st != GG_OK)
        return st;
    gg::GatherArgs a;
    int kind = kVector, vec = 0;
    bool launch = false;
    static thread_local CUtensorMap in_map;
    static thread_local gg::OutMaps maps;
    st = prepare_gather(heap, gg::kModeGather, rank, input, ld_in, output, ld_out, M, N, dtype,
                        tile, comm_programs, group, 0, dev_status, GG_AG_AUTO, &a, &kind, &vec,
                        &in_map, &maps, &launch);
    if (st != GG_OK || !launch)
        return st;
    st = resolve_status(&a.status);
    if (st == GG_OK)
        st = resolve_trace(&a.trace, gg::kTraceGather);
    if (st != GG_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the static counter stands in for a heap workspace slot; when the launch
    // claims runs, prepare_claims zeroes it on `s` before the kernel
    if (kind == kTma && a.claim_policy != GG_CLAIM_NEVER)
        a.work = scratch;
    cudaError_t e;
    if (kind == kTma)
        e = gg::launch_gather_tma(in_map, maps, a, comm_programs, s);
    else if (kind == kBulk)
        e = gg::launch_gather_bulk(a, comm_programs, s);
    else
        e = gg::launch_gather_vec(a, comm_programs, vec, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "launching the allocation-free all-gather");
    return ok();
}

}  // extern "C"
