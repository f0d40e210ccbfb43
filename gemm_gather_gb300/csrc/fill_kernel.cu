// The fused matmul + all-gather with an empty contraction (K == 0).
//
// C_r = A_r @ B sums over k in [0, K); with K == 0 every element is the empty
// sum, +0, so the gathered output holds zero blocks: row block i of every
// member's output is all zeros (binary16 and bfloat16 +0 are both the
// all-zero bit pattern), for each source i of the launch.  No operand is
// read and padding columns between N and the row pitch are left alone.
#include <cuda_runtime.h>

#include "gg_internal.h"
#include "ptx.cuh"

namespace gg {
namespace {

constexpr int kFillThreads = 256;

// One 16-byte store per thread and step: rows are whole 16-byte units (the
// fused call requires 16-byte aligned outputs, pitches and rows).
__global__ void __launch_bounds__(kFillThreads) zero_rows_kernel(const ZeroArgs z)
{
    const int64_t rows = (int64_t)z.n_src * z.M;  // rows per member
    const int64_t vecs = z.row_b / 16;             // 16-byte units per row
    const int64_t total = (int64_t)z.W * rows * vecs;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += step) {
        const int64_t t = i / vecs;
        const int64_t v = i - t * vecs;
        const int d = (int)(t / rows);
        const int64_t r = t - (int64_t)d * rows;
        uint8_t *row = reinterpret_cast<uint8_t *>(z.out[d]) +
                       ((int64_t)z.src_first * z.M + r) * z.ld_out_b;
        *reinterpret_cast<uint4 *>(row + v * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace

cudaError_t launch_zero_rows(const ZeroArgs &z, int programs, cudaStream_t s)
{
    const int64_t units = (int64_t)z.W * z.n_src * z.M * (z.row_b / 16);
    const int64_t need = (units + kFillThreads - 1) / kFillThreads;
    const int grid = (int)gg_min64(programs, need > 0 ? need : 1);
    zero_rows_kernel<<<grid, kFillThreads, 0, s>>>(z);
    return cudaGetLastError();
}

}  // namespace gg
