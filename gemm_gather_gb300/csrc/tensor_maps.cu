// Host-side TMA tensor maps: the CUDA driver API's encoder, reached through the
// runtime's entry-point query (no link against libcuda), and the
// per-destination output maps of the gathers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gg_internal.h"

namespace gg {

namespace {

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

bool tensor_maps_available() { return encode_fn() != nullptr; }

bool encode_map(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                const uint64_t *dims, const uint64_t *strides_b, const uint32_t *box,
                CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i)
        st[i] = strides_b[i];
    return enc(map, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_out_maps(OutMaps *out, const uint64_t *member_out, int W, int64_t M, int64_t N,
                     int64_t ld_out_b, int es, uint32_t box_cols, uint32_t box_rows,
                     CUtensorMapDataType dt, CUtensorMapSwizzle swizzle)
{
    // destination d: its gathered output viewed as {N, M, W} (column, row within a
    // block, block), so a box is clipped at the end of its own row block
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)M, (uint64_t)W};
    const uint64_t strides[2] = {(uint64_t)ld_out_b, (uint64_t)(M * ld_out_b)};
    const uint32_t box[3] = {box_cols, box_rows, 1};
    (void)es;
    for (int d = 0; d < W; ++d)
        if (!encode_map(&out->map[d], dt, 3, reinterpret_cast<const void *>(member_out[d]), dims,
                        strides, box, swizzle))
            return false;
    return true;
}

}  // namespace gg
