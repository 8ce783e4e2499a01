/* A plain C client of libtb: the C ABI used without Python or PyTorch.
 *
 *   c_client <out_dir>
 *
 * Allocates with the CUDA runtime, fills three 16 MiB sources with the
 * default pattern, runs one 3-source reduce-copy, a 2-iteration transfer of
 * source 1 on the copy engines (DMA executor), and one batch of 1000
 * scattered copies through tb_batch_copy and again through
 * tb_batch_copy_noalloc, and writes what came back to <out_dir>/reduce.bin,
 * dma.bin, batch.bin and batch_noalloc.bin, for the caller to compare with
 * the oracle.  The batch layout is fixed arithmetic:
 * copy i moves 64 + 13 * i bytes from source offset 16384 * i + i % 13 to
 * destination offset 16384 * ((i * 7919) % 1000) + i % 5 (distinct 16 KiB
 * slots, so no two destinations overlap).  Exit status 0 on
 * success, else the failing call is printed. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "tb.h"

#define CHECK_TB(call)                                                                   \
    do {                                                                                 \
        int rc_ = (call);                                                                \
        if (rc_ != TB_OK) {                                                              \
            fprintf(stderr, "%s -> %s (%s)\n", #call, tb_strerror(rc_),                  \
                    ctx ? tb_last_error(ctx) : "");                                      \
            return 1;                                                                    \
        }                                                                                \
    } while (0)
#define CHECK_CUDA(call)                                                                 \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess) {                                                         \
            fprintf(stderr, "%s -> %s\n", #call, cudaGetErrorString(e_));                \
            return 1;                                                                    \
        }                                                                                \
    } while (0)

static int write_file(const char *dir, const char *name, const void *data, size_t n)
{
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(data, 1, n, f) != n) {
        fprintf(stderr, "cannot write %s\n", path);
        if (f)
            fclose(f);
        return 1;
    }
    fclose(f);
    return 0;
}

int main(int argc, char **argv)
{
    if (argc != 2) {
        fprintf(stderr, "usage: %s <out_dir>\n", argv[0]);
        return 2;
    }
    tb_ctx *ctx = NULL;
    CHECK_TB(tb_create(&ctx, 0, NULL));

    /* Reduce-copy: dst = src0 + src1 + src2 over 16 MiB. */
    const uint64_t nb = 16u << 20;
    void *src[3] = {NULL, NULL, NULL};
    void *dst = NULL;
    for (int k = 0; k < 3; ++k)
        CHECK_CUDA(cudaMalloc(&src[k], nb));
    CHECK_CUDA(cudaMalloc(&dst, nb));
    tb_pattern pat;
    memset(&pat, 0, sizeof pat);
    pat.kind = TB_PATTERN_DEFAULT;
    for (int k = 0; k < 3; ++k)
        CHECK_TB(tb_fill_source(ctx, src[k], nb, &pat, k, NULL));
    CHECK_TB(tb_reduce_copy(ctx, (const void *const *)src, 3, dst, nb, 0, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    void *host = malloc(nb);
    if (!host)
        return 1;
    CHECK_CUDA(cudaMemcpy(host, dst, nb, cudaMemcpyDeviceToHost));
    if (write_file(argv[1], "reduce.bin", host, nb))
        return 1;

    /* DMA executor: dst2 = src[1], one copy-engine copy per iteration. */
    void *dst2 = NULL;
    CHECK_CUDA(cudaMalloc(&dst2, nb));
    CHECK_CUDA(cudaMemset(dst2, 0, nb));
    tb_transfer t;
    memset(&t, 0, sizeof t);
    t.srcs = &src[1];
    t.n_src = 1;
    t.dst = dst2;
    t.num_bytes = nb;
    t.iters = 2;
    t.rotate_bytes = 0;
    t.executor = TB_EXEC_DMA;
    tb_result res;
    CHECK_TB(tb_run_transfer_ex(ctx, &t, &res));
    if (res.executor != TB_EXEC_DMA || res.iters != 2) {
        fprintf(stderr, "DMA result: executor %d, iters %d\n", (int)res.executor, (int)res.iters);
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(host, dst2, nb, cudaMemcpyDeviceToHost));
    if (write_file(argv[1], "dma.bin", host, nb))
        return 1;

    /* Batch copy from src[0] into a zeroed pool. */
    const size_t n = 1000;
    const uint64_t pool = 16384ull * 1000 + 64;
    void *dpool = NULL;
    CHECK_CUDA(cudaMalloc(&dpool, pool));
    CHECK_CUDA(cudaMemset(dpool, 0, pool));
    tb_copy_desc *desc = calloc(n, sizeof *desc);
    if (!desc)
        return 1;
    for (size_t i = 0; i < n; ++i) {
        desc[i].src = (uint64_t)(uintptr_t)src[0] + 16384 * i + i % 13;
        desc[i].dst = (uint64_t)(uintptr_t)dpool + 16384 * ((i * 7919) % 1000) + i % 5;
        desc[i].len = 64 + 13 * i;
    }
    cudaStream_t s;
    CHECK_CUDA(cudaStreamCreate(&s));
    CHECK_TB(tb_batch_copy(ctx, desc, n, (tb_stream)s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    tb_batch_stats st;
    CHECK_TB(tb_last_batch_stats(ctx, &st));
    if (st.descs != n) {
        fprintf(stderr, "batch stats: %llu descriptors\n", (unsigned long long)st.descs);
        return 1;
    }
    void *hpool = malloc(pool);
    if (!hpool)
        return 1;
    CHECK_CUDA(cudaMemcpy(hpool, dpool, pool, cudaMemcpyDeviceToHost));
    if (write_file(argv[1], "batch.bin", hpool, pool))
        return 1;

    /* The same batch without any allocation, into a second zeroed pool. */
    void *dpool2 = NULL;
    CHECK_CUDA(cudaMalloc(&dpool2, pool));
    CHECK_CUDA(cudaMemset(dpool2, 0, pool));
    for (size_t i = 0; i < n; ++i)
        desc[i].dst = (uint64_t)(uintptr_t)dpool2 + 16384 * ((i * 7919) % 1000) + i % 5;
    CHECK_TB(tb_batch_copy_noalloc(desc, n, (tb_stream)s));
    CHECK_CUDA(cudaStreamSynchronize(s));
    CHECK_TB(tb_batch_copy_noalloc(NULL, 0, (tb_stream)s)); /* no expired wait to report */
    CHECK_CUDA(cudaMemcpy(hpool, dpool2, pool, cudaMemcpyDeviceToHost));
    if (write_file(argv[1], "batch_noalloc.bin", hpool, pool))
        return 1;
    CHECK_CUDA(cudaFree(dpool2));
    CHECK_CUDA(cudaFree(dst2));

    free(desc);
    free(host);
    free(hpool);
    CHECK_CUDA(cudaStreamDestroy(s));
    CHECK_CUDA(cudaFree(dpool));
    CHECK_CUDA(cudaFree(dst));
    for (int k = 0; k < 3; ++k)
        CHECK_CUDA(cudaFree(src[k]));
    tb_destroy(ctx);
    printf("ok\n");
    return 0;
}
