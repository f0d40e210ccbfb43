/*
 * Oracle for the tiled all-gather over a symmetric heap and for the fused
 * matmul + all-gather.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may call this code; the product
 * (the CUDA library and its Python binding) never does, and the two share no
 * code, header, table or helper.
 *
 * Everything here is the plain definition, written for a reader to check by
 * eye, not for speed.  Sources (ROCm/iris pages):
 *
 *  - iris PR #626, "Summary": an all-gather writes the caller's tile to every
 *    destination of the group, the local copy included ("the local copy goes
 *    first"); the fused matmul_all_gather computes the tile and all-gathers it
 *    in the epilogue.
 *  - iris #594, "Multi-GPU CI": results are compared with
 *    torch.distributed.all_gather_into_tensor, i.e. block i of the gathered
 *    output is group member i's input, concatenated along rows.
 *  - iris #594, "Local validation": logical ranks are independent allocations
 *    (here: partitions of one heap image); checks cover outputs, padding,
 *    guards and inactive heaps.  So nothing but the gathered blocks changes.
 *  - iris #591 "Gluon all-gather reloads peer heap bases inside the tile
 *    loop", Description §1: group membership from rank_start, rank_stride and
 *    world_size; heap_bases gives each rank's partition.
 *
 * Parity pins (tests/test_oracle_pins.py): index-coded brute force,
 * all_to_all applied twice is the identity,
 * invariants, torch.distributed gloo all_gather_into_tensor, numpy float64
 * matmul, integer-exact products, one-hot/identity/ones closed forms, numpy
 * float16 and torch bfloat16 conversions.  No function here is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * Group resolution (iris #591, Description §1; iris #594 "Local validation"
 * on strided subgroups): member i of the group is heap
 * rank_start + i * rank_stride.  Returns the group index of heap h, or -1
 * when h is not a member.
 * ------------------------------------------------------------------------- */
int oracle_group_index(int h, int rank_start, int rank_stride, int world_size)
{
    for (int i = 0; i < world_size; ++i)
        if (rank_start + i * rank_stride == h)
            return i;
    return -1;
}

/* ---------------------------------------------------------------------------
 * One rank's contribution (iris PR #626 "Summary"; iris #594 "Multi-GPU CI"):
 * source heap `src_rank` (a group member) writes its M x N block `src`
 * (row pitch ld_in elements) into row block i = group index of src_rank of
 * the gathered output of EVERY member d of the group, the source itself
 * included.  The gathered output of member d starts `out_off` bytes into
 * partition d and has row pitch ld_out elements; element (i*M + m, n) is
 * element (m, n) of the source.  Bytes are copied unchanged (no conversion).
 * heap: H partitions of part_bytes each, laid out one after another.
 * Returns 0, or -1 if src_rank is not a member or a write leaves a partition.
 * ------------------------------------------------------------------------- */
int oracle_gather_contribution(uint8_t *heap, int64_t part_bytes, int H,
                               const uint8_t *src, int64_t ld_in,
                               int64_t out_off, int64_t ld_out,
                               int64_t M, int64_t N, int esize,
                               int rank_start, int rank_stride, int world_size,
                               int src_rank)
{
    int i = oracle_group_index(src_rank, rank_start, rank_stride, world_size);
    if (i < 0)
        return -1;
    for (int q = 0; q < world_size; ++q) {
        int d = rank_start + q * rank_stride;
        if (d < 0 || d >= H)
            return -1;
        uint8_t *part = heap + (int64_t)d * part_bytes;
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t n = 0; n < N; ++n) {
                int64_t dst = out_off + ((i * M + m) * ld_out + n) * esize;
                if (dst < 0 || dst + esize > part_bytes)
                    return -1;
                memcpy(part + dst, src + (m * ld_in + n) * esize, (size_t)esize);
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * The whole collective: every member i contributes the block that sits
 * `in_off` bytes into its own partition (row pitch ld_in).  The sources are
 * read from a snapshot `src_heap` of the heap taken before the collective, so
 * an output that overlaps an input cannot feed a later contribution.
 * ------------------------------------------------------------------------- */
int oracle_all_gather(uint8_t *heap, const uint8_t *src_heap, int64_t part_bytes,
                      int H, int64_t in_off, int64_t ld_in, int64_t out_off,
                      int64_t ld_out, int64_t M, int64_t N, int esize,
                      int rank_start, int rank_stride, int world_size)
{
    for (int i = 0; i < world_size; ++i) {
        int r = rank_start + i * rank_stride;
        if (r < 0 || r >= H)
            return -1;
        const uint8_t *src = src_heap + (int64_t)r * part_bytes + in_off;
        int rc = oracle_gather_contribution(heap, part_bytes, H, src, ld_in,
                                            out_off, ld_out, M, N, esize,
                                            rank_start, rank_stride,
                                            world_size, r);
        if (rc)
            return rc;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * All-to-all (iris #594, "Compiler inspection and grouping", and iris #591
 * Work: the Gluon all_to_all over the same symmetric heap).  Each member i
 * holds W blocks of M x N rows (block d at rows d*M..d*M+M-1 of its W*M x N
 * input, pitch ld_in, at in_off); block d is meant for member d.  The output
 * of member d (W*M x N, pitch ld_out, at out_off) holds, in row block i, the
 * block member i meant for d:
 *     out_d[(i*M + m), n] = in_i[(d*M + m), n]
 * -- torch.distributed.all_to_all_single with equal splits.  Sources are read
 * from the snapshot src_heap; bytes are copied unchanged; nothing else changes.
 * ------------------------------------------------------------------------- */
int oracle_all_to_all(uint8_t *heap, const uint8_t *src_heap, int64_t part_bytes,
                      int H, int64_t in_off, int64_t ld_in, int64_t out_off,
                      int64_t ld_out, int64_t M, int64_t N, int esize,
                      int rank_start, int rank_stride, int world_size)
{
    for (int i = 0; i < world_size; ++i) {
        int src = rank_start + i * rank_stride;
        for (int d = 0; d < world_size; ++d) {
            int dst = rank_start + d * rank_stride;
            if (src < 0 || src >= H || dst < 0 || dst >= H)
                return -1;
            const uint8_t *in = src_heap + (int64_t)src * part_bytes + in_off;
            uint8_t *out = heap + (int64_t)dst * part_bytes + out_off;
            for (int64_t m = 0; m < M; ++m) {
                for (int64_t n = 0; n < N; ++n) {
                    int64_t from = ((d * M + m) * ld_in + n) * esize;
                    int64_t to = ((i * M + m) * ld_out + n) * esize;
                    if (in_off + from + esize > part_bytes || out_off + to + esize > part_bytes)
                        return -1;
                    memcpy(out + to, in + from, (size_t)esize);
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * 16-bit floating-point formats, from their definitions.
 *   binary16 (IEEE 754-2008): 1 sign, 5 exponent (bias 15), 10 fraction bits.
 *   bfloat16: the upper half of IEEE binary32: 1 sign, 8 exponent (bias 127),
 *             7 fraction bits.
 * fmt 0 = binary16, fmt 1 = bfloat16.
 * ------------------------------------------------------------------------- */
static void fmt_params(int fmt, int *ebits, int *mbits, int *bias)
{
    if (fmt == 0) { *ebits = 5; *mbits = 10; *bias = 15; }
    else          { *ebits = 8; *mbits = 7;  *bias = 127; }
}

double oracle_decode16(uint16_t h, int fmt)
{
    int ebits, mbits, bias;
    fmt_params(fmt, &ebits, &mbits, &bias);
    int sign = (h >> 15) & 1;
    int e = (h >> mbits) & ((1 << ebits) - 1);
    int f = h & ((1 << mbits) - 1);
    double v;
    if (e == 0)                          /* zero and subnormals */
        v = ldexp((double)f, 1 - bias - mbits);
    else if (e == (1 << ebits) - 1)      /* infinities and NaN */
        v = f ? NAN : INFINITY;
    else                                 /* normal: (1.f) * 2^(e-bias) */
        v = ldexp((double)((1 << mbits) + f), e - bias - mbits);
    return sign ? -v : v;
}

/* Round half to even of a non-negative double below 2^52. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double d = q - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/* Round-to-nearest-even encoding of a double into binary16 / bfloat16. */
uint16_t oracle_encode16(double x, int fmt)
{
    int ebits, mbits, bias;
    fmt_params(fmt, &ebits, &mbits, &bias);
    const int emax = (1 << ebits) - 2 - bias;   /* largest normal exponent */
    const int emin = 1 - bias;                  /* smallest normal exponent */
    const uint16_t inf_bits = (uint16_t)(((1 << ebits) - 1) << mbits);
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return (uint16_t)(inf_bits | (1 << (mbits - 1)));
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | inf_bits);
    int ex;
    frexp(a, &ex);              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;             /* a in [2^e, 2^(e+1)) */
    if (e < emin)
        e = emin;               /* subnormal range: fixed quantum */
    double q = ldexp(a, mbits - e);          /* exact: power-of-two scaling */
    double qi = round_half_even(q);
    if (qi >= ldexp(1.0, mbits + 1)) {       /* rounding carried into the next binade */
        qi = ldexp(qi, -1);
        e += 1;
    }
    if (e > emax)
        return (uint16_t)(sign | inf_bits);
    uint32_t iq = (uint32_t)qi;
    if (iq < (1u << mbits))                  /* subnormal (or rounded to zero) */
        return (uint16_t)(sign | iq);
    uint32_t efield = (uint32_t)(e + bias);
    return (uint16_t)(sign | (efield << mbits) | (iq - (1u << mbits)));
}

/* ---------------------------------------------------------------------------
 * C = A @ B in float64 (iris PR #626 "Summary"/"Benchmark": the fused
 * kernel's tile is the product of the rank's A rows and the shared B).
 * A: M x K, row pitch lda; B: K x N, row pitch ldb; both 16-bit (fmt);
 * C: M x N doubles, row pitch ldc.  C[m][n] = sum over k of A[m][k]*B[k][n],
 * each product and the sum in double precision, k ascending.
 * The operands are decoded to double first (B into a transposed copy, so that
 * each sum reads one contiguous row of it); the products and the order of
 * the sum are exactly those of the definition.
 * Only the rows listed in `rows` (n_rows of them) are computed when rows is
 * non-NULL; row j of the result then holds row rows[j].
 * Returns 0, or -1 if memory for the decoded operands is not available.
 * ------------------------------------------------------------------------- */
int oracle_matmul_f64(const uint16_t *A, int64_t lda, const uint16_t *B,
                      int64_t ldb, double *C, int64_t ldc, int64_t M,
                      int64_t N, int64_t K, int fmt, const int64_t *rows,
                      int64_t n_rows)
{
    int64_t R = rows ? n_rows : M;
    double *bt = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!bt)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            bt[n * K + k] = oracle_decode16(B[k * ldb + n], fmt);
    int failed = 0;
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!a) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t j = 0; j < R; ++j) {
            if (!a)
                continue;
            int64_t m = rows ? rows[j] : j;
            for (int64_t k = 0; k < K; ++k)
                a[k] = oracle_decode16(A[m * lda + k], fmt);
            for (int64_t n = 0; n < N; ++n) {
                const double *b = bt + n * K;
                double s = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    s += a[k] * b[k];
                C[j * ldc + n] = s;
            }
        }
        free(a);
    }
    free(bt);
    return failed ? -1 : 0;
}

/* Round an M x N block of doubles into 16-bit values (round to nearest even),
 * the conversion the fused epilogue applies before gathering. */
void oracle_round16(const double *C, int64_t ldc, uint16_t *out, int64_t ldo,
                    int64_t M, int64_t N, int fmt)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            out[m * ldo + n] = oracle_encode16(C[m * ldc + n], fmt);
}

/* Thread control for the row-parallel loops above (OpenMP; results do not
 * depend on the thread count: each output element is summed by one thread). */
#ifdef _OPENMP
#include <omp.h>
void oracle_set_threads(int n) { if (n > 0) omp_set_num_threads(n); }
int oracle_max_threads(void) { return omp_get_max_threads(); }
#else
void oracle_set_threads(int n) { (void)n; }
int oracle_max_threads(void) { return 1; }
#endif
