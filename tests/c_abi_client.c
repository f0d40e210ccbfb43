/*
 * A plain C client of the library (no Python, no torch): the caller owns all
 * device memory (cudaMalloc), builds the symmetric heap, runs one group
 * all-gather and one fused matmul + all-gather through the C ABI of
 * include/gemm_gather.h, and checks the results on the host.
 *
 *   all-gather: W=4 members, 96 x 264 binary16 bit patterns per member (every
 *     element encodes its member, row and column), tile 8x256, 16 programs;
 *     every member's row block i must equal member i's input bit for bit, and
 *     the padding columns of the output must keep their fill byte;
 *   fused: W=2 members, M=128, N=256, K=64, integer-valued f16 operands in
 *     {-2..2}: every product and partial sum is an exact integer in float32
 *     and |C| <= 256 is exact in binary16, so each output element must equal
 *     the integer dot product computed here.
 *   status: a launch given no status word leaves the library's word at 0.
 *   the gather runs with plain stores (gg_set_store_policy) and traced
 *   (gg_set_trace): its trace record must show time and cycles passing.
 *
 * Prints "c abi client ok" and returns 0 on success; any mismatch or error
 * prints what failed and returns 1.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm_gather.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 1;                                                              \
        }                                                                          \
    } while (0)
#define CHECK_GG(x)                                                                \
    do {                                                                           \
        gg_status s_ = (x);                                                        \
        if (s_ != GG_OK) {                                                         \
            fprintf(stderr, "%s: %s (%s)\n", #x, gg_status_string(s_), gg_last_error()); \
            return 1;                                                              \
        }                                                                          \
    } while (0)

/* binary16 encoding of a small integer (|v| <= 2048): exact */
static uint16_t f16_of_int(int v)
{
    if (v == 0)
        return 0;
    uint16_t sign = v < 0 ? 0x8000 : 0;
    unsigned a = (unsigned)(v < 0 ? -v : v);
    int e = 0;
    while ((a >> e) > 1)
        ++e;                                   /* a = 1.f * 2^e */
    unsigned frac = (a << (10 - e)) & 0x3FF;   /* e <= 10 */
    return (uint16_t)(sign | (unsigned)((e + 15) << 10) | frac);
}

static uint16_t code_of(int member, int row, int col)
{
    uint32_t h = (uint32_t)member * 2654435761u ^ (uint32_t)row * 40503u ^ (uint32_t)col * 9176u;
    h ^= h >> 13;
    h *= 0x5bd1e995u;
    h ^= h >> 15;
    return (uint16_t)h;
}

static int run_gather(void)
{
    const int W = 4, M = 96, N = 264, LD_OUT = 272;
    const size_t in_off = 4096, in_bytes = (size_t)M * N * 2;
    const size_t out_off = 65536, out_bytes = (size_t)W * M * LD_OUT * 2;
    const size_t part = 1 << 20;
    void *heap_mem = NULL, *status = NULL;
    uint64_t *table = NULL;
    CHECK_CUDA(cudaMalloc(&heap_mem, part * W));
    CHECK_CUDA(cudaMalloc((void **)&table, sizeof(uint64_t) * W));
    CHECK_CUDA(cudaMalloc(&status, sizeof(int)));
    CHECK_CUDA(cudaMemset(heap_mem, 0x5A, part * W));
    CHECK_CUDA(cudaMemset(status, 0, sizeof(int)));
    uint16_t *host = (uint16_t *)malloc(in_bytes);
    for (int r = 0; r < W; ++r) {
        for (int m = 0; m < M; ++m)
            for (int n = 0; n < N; ++n)
                host[(size_t)m * N + n] = code_of(r, m, n);
        CHECK_CUDA(cudaMemcpy((char *)heap_mem + r * part + in_off, host, in_bytes,
                              cudaMemcpyHostToDevice));
    }
    gg_heap *heap = NULL;
    CHECK_GG(gg_heap_create(heap_mem, part, W, table, NULL, &heap));
    gg_tile tile = {8, 256};
    gg_group group = {0, 1, W};
    /* plain stores (no L2 hint) and a traced launch */
    CHECK_GG(gg_set_store_policy(GG_STORE_PLAIN));
    if (gg_get_store_policy() != GG_STORE_PLAIN || gg_set_store_policy(5) != GG_ERR_INVALID_ARG) {
        fprintf(stderr, "store policy round trip\n");
        return 1;
    }
    CHECK_GG(gg_set_trace(1));
    CHECK_GG(gg_all_gather(heap, -1, (char *)heap_mem + in_off, N, (char *)heap_mem + out_off,
                           LD_OUT, M, N, GG_F16, tile, 16, group, (int *)status, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    gg_trace_record rec;
    CHECK_GG(gg_trace_read(NULL, &rec, NULL));
    CHECK_GG(gg_set_trace(0));
    CHECK_GG(gg_set_store_policy(GG_STORE_EVICT_FIRST));
    if (!(rec.end_ns > rec.start_ns && rec.end_cycles > rec.start_cycles)) {
        fprintf(stderr, "trace record not written\n");
        return 1;
    }
    int st = -1;
    CHECK_CUDA(cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost));
    if (st != 0) {
        fprintf(stderr, "all-gather status %d\n", st);
        return 1;
    }
    uint16_t *out = (uint16_t *)malloc(out_bytes);
    for (int d = 0; d < W; ++d) {
        CHECK_CUDA(cudaMemcpy(out, (char *)heap_mem + d * part + out_off, out_bytes,
                              cudaMemcpyDeviceToHost));
        for (int i = 0; i < W; ++i)
            for (int m = 0; m < M; ++m) {
                const uint16_t *row = out + ((size_t)i * M + m) * LD_OUT;
                for (int n = 0; n < N; ++n)
                    if (row[n] != code_of(i, m, n)) {
                        fprintf(stderr, "member %d block %d row %d col %d: %04x != %04x\n", d,
                                i, m, n, row[n], code_of(i, m, n));
                        return 1;
                    }
                for (int n = N; n < LD_OUT; ++n)
                    if (row[n] != 0x5A5A) {
                        fprintf(stderr, "member %d padding changed at row %d\n", d, i * M + m);
                        return 1;
                    }
            }
    }
    free(out);
    free(host);
    CHECK_GG(gg_heap_destroy(heap));
    CHECK_CUDA(cudaFree(status));
    CHECK_CUDA(cudaFree(table));
    CHECK_CUDA(cudaFree(heap_mem));
    return 0;
}

static int run_fused(void)
{
    const int W = 2, M = 128, N = 256, K = 64;
    const size_t part = 1 << 20, a_off = 0, out_off = 65536;
    const size_t out_bytes = (size_t)W * M * N * 2;
    void *heap_mem = NULL, *Bd = NULL;
    uint64_t *table = NULL;
    CHECK_CUDA(cudaMalloc(&heap_mem, part * W));
    CHECK_CUDA(cudaMalloc((void **)&table, sizeof(uint64_t) * W));
    CHECK_CUDA(cudaMalloc(&Bd, (size_t)K * N * 2));
    CHECK_CUDA(cudaMemset(heap_mem, 0, part * W));
    int *Ai = (int *)malloc(sizeof(int) * W * M * K), *Bi = (int *)malloc(sizeof(int) * K * N);
    uint16_t *buf = (uint16_t *)malloc((size_t)(M > K ? M : K) * (K > N ? K : N) * 2);
    srand(7);
    for (int r = 0; r < W; ++r) {
        for (int i = 0; i < M * K; ++i) {
            Ai[r * M * K + i] = rand() % 5 - 2;
            buf[i] = f16_of_int(Ai[r * M * K + i]);
        }
        CHECK_CUDA(cudaMemcpy((char *)heap_mem + r * part + a_off, buf, (size_t)M * K * 2,
                              cudaMemcpyHostToDevice));
    }
    for (int i = 0; i < K * N; ++i) {
        Bi[i] = rand() % 5 - 2;
        buf[i] = f16_of_int(Bi[i]);
    }
    CHECK_CUDA(cudaMemcpy(Bd, buf, (size_t)K * N * 2, cudaMemcpyHostToDevice));
    gg_heap *heap = NULL;
    CHECK_GG(gg_heap_create(heap_mem, part, W, table, NULL, &heap));
    gg_tile tile = {GG_FUSED_BLOCK_M, GG_FUSED_BLOCK_N};
    gg_group group = {0, 1, W};
    CHECK_GG(gg_clear_device_status(NULL));
    /* no status word: a wait that gave up would land in the library's word */
    CHECK_GG(gg_matmul_all_gather(heap, -1, (char *)heap_mem + a_off, K, Bd, N,
                                  (char *)heap_mem + out_off, N, M, N, K, GG_F16, tile, 4, group,
                                  NULL, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int st = -1;
    CHECK_GG(gg_device_status(NULL, &st));
    if (st != 0) {
        fprintf(stderr, "fused: library status word %d\n", st);
        return 1;
    }
    uint16_t *out = (uint16_t *)malloc(out_bytes);
    for (int d = 0; d < W; ++d) {
        CHECK_CUDA(cudaMemcpy(out, (char *)heap_mem + d * part + out_off, out_bytes,
                              cudaMemcpyDeviceToHost));
        for (int i = 0; i < W; ++i)
            for (int m = 0; m < M; ++m)
                for (int n = 0; n < N; ++n) {
                    int acc = 0;
                    for (int k = 0; k < K; ++k)
                        acc += Ai[(i * M + m) * K + k] * Bi[k * N + n];
                    const uint16_t got = out[((size_t)i * M + m) * N + n];
                    if (got != f16_of_int(acc)) {
                        fprintf(stderr, "fused member %d block %d (%d,%d): %04x != %04x (%d)\n", d,
                                i, m, n, got, f16_of_int(acc), acc);
                        return 1;
                    }
                }
    }
    free(out);
    free(buf);
    free(Ai);
    free(Bi);
    CHECK_GG(gg_heap_destroy(heap));
    CHECK_CUDA(cudaFree(Bd));
    CHECK_CUDA(cudaFree(table));
    CHECK_CUDA(cudaFree(heap_mem));
    return 0;
}

int main(void)
{
    if (run_gather() != 0 || run_fused() != 0)
        return 1;
    printf("c abi client ok\n");
    return 0;
}
