/*
 * c_abi_smoke.c -- a plain C consumer of libdlrm_sparse.so: the header
 * compiles as C, the library links without Python, and the entry points
 * behave as declared.
 *
 *   c_abi_smoke          host-only checks (no GPU needed): ABI version,
 *                        status strings, argument checks, workspace sizes
 *   c_abi_smoke --gpu    also fused forwards on the device with identity
 *                        tables (E_t = I), whose outputs are known exactly:
 *                        out[b] = [x_b, z(i,j)] with z(0, 1+t) = x_b[r_t] and
 *                        z(1+i, 1+j) = [r_i == r_j]  ("DLRM", robocikowo.com,
 *                        "Forward pass" steps (2)-(4)); the x values carry at
 *                        most 16 significant bits, which every Gram path of the
 *                        library reproduces exactly.
 * Exit status 0 on success; the first failure is printed.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dlrm_sparse.h"

static int failures = 0;
#define CHECK(cond)                                                            \
    do {                                                                       \
        if (!(cond)) {                                                         \
            fprintf(stderr, "c_abi_smoke: check failed at line %d: %s\n",      \
                    __LINE__, #cond);                                          \
            ++failures;                                                        \
        }                                                                      \
    } while (0)

static int host_checks(void)
{
    void *ptrs[2] = {(void *)0x1000, (void *)0x1000};
    int64_t rows[2] = {10, 10};
    dlrm_tables tb = {2, 128, DLRM_F32, ptrs, rows};
    dlrm_bags bags = {4, 8, DLRM_I32, (const void *)0x2000, (const void *)0x3000};
    size_t need = 0;

    CHECK(dlrm_abi_version() == 2);
    CHECK(strcmp(dlrm_status_string(DLRM_OK), "ok") == 0);
    CHECK(strcmp(dlrm_status_string(DLRM_ERR_INDEX_OOB), "index out of range") == 0);
    CHECK(dlrm_sparse_fwd(NULL, &bags, DLRM_POOL_SUM, (const float *)0x4000, (float *)0x5000,
                          NULL, NULL, 0) == DLRM_ERR_INVALID_ARG);
    tb.num_tables = 0;
    CHECK(dlrm_embbag_fwd(&tb, &bags, DLRM_POOL_SUM, (float *)0x4000, NULL, 0) ==
          DLRM_ERR_INVALID_ARG);
    tb.num_tables = 2;
    tb.dim = 48;
    CHECK(dlrm_embbag_fwd(&tb, &bags, DLRM_POOL_SUM, (float *)0x4000, NULL, 0) ==
          DLRM_ERR_UNSUPPORTED);
    tb.dim = 128;
    CHECK(dlrm_sparse_bwd_workspace_size(&tb, &bags, &need) == DLRM_OK);
    CHECK(need >= (size_t)4 * 2 * 128 * 4 + 16 * 8);
    CHECK(dlrm_embbag_bwd_workspace_size(&tb, &bags, DLRM_POOL_SUM, &need) == DLRM_OK);
    {
        dlrm_update upd = {DLRM_RULE_SGD, 0.1f, 0.0f, NULL};
        bags.batch = (int64_t)1 << 31;
        bags.index_type = DLRM_I64;
        CHECK(dlrm_embbag_bwd_update(&tb, &bags, DLRM_POOL_SUM, (const float *)0x10, &upd,
                                     (void *)0x10, (size_t)1 << 62, NULL, 0, 0) ==
              DLRM_ERR_UNSUPPORTED); /* T * B = 2^32 */
        upd.rule = 7;
        bags.batch = 4;
        CHECK(dlrm_embbag_bwd_update(&tb, &bags, DLRM_POOL_SUM, (const float *)0x10, &upd,
                                     (void *)0x10, (size_t)1 << 62, NULL, 0, 0) ==
              DLRM_ERR_INVALID_ARG);
        /* the split training step: a workspace too small for the sort, an unknown rule */
        bags.index_type = DLRM_I32;
        CHECK(dlrm_sparse_bwd_sort(&tb, &bags, (void *)0x10, 64, NULL, 0) == DLRM_ERR_INVALID_ARG);
        CHECK(dlrm_sparse_bwd_update_sorted(&tb, &bags, DLRM_POOL_SUM, (const float *)0x10,
                                            (const float *)0x10, (const float *)0x10, (float *)0x10,
                                            &upd, (void *)0x10, (size_t)1 << 62, NULL,
                                            (cudaEvent_t)0, (cudaEvent_t)0, 0) == DLRM_ERR_INVALID_ARG);
    }
    {
        int32_t shard[2] = {0, 0}, slot[2] = {0, 0}; /* slot 0 twice: inconsistent */
        int64_t start[2] = {0, 4};
        dlrm_shard_plan plan = {1, 1, 2, 128, 4, shard, slot, start};
        float *bt[1] = {(float *)0x100}, *bs[1] = {(float *)0x200};
        CHECK(dlrm_pooled_exchange(&plan, bt, bs, 1, 0) == DLRM_ERR_INVALID_ARG);
    }
    return failures;
}

/* One identity-table forward of T tables of D rows, B one-hot samples. */
static int identity_forward(int T, int D, int B)
{
    const int N = T + 1, W = D + N * (N - 1) / 2;
    float *tab_h = calloc((size_t)D * D, sizeof(float));
    float *x_h = malloc(sizeof(float) * (size_t)B * D);
    float *out_h = malloc(sizeof(float) * (size_t)B * W);
    int32_t *idx_h = malloc(sizeof(int32_t) * (size_t)T * B);
    int32_t *off_h = malloc(sizeof(int32_t) * ((size_t)T * B + 1));
    void *tab_d[DLRM_MAX_TABLES];
    int64_t rows[DLRM_MAX_TABLES];
    float *x_d = NULL, *out_d = NULL;
    int32_t *idx_d = NULL, *off_d = NULL, *st_d = NULL, st_h = -1;
    unsigned seed = 12345u;
    int bad = 0;

    for (int d = 0; d < D; ++d)
        tab_h[d * D + d] = 1.0f;
    for (int i = 0; i < B * D; ++i) { /* x with 16 significant bits: k / 2^12, |k| < 2^15 */
        seed = seed * 1103515245u + 12345u;
        x_h[i] = (float)((int)(seed >> 16) % 32768 - 16384) / 4096.0f;
    }
    for (int i = 0; i < T * B; ++i) {
        seed = seed * 1103515245u + 12345u;
        idx_h[i] = (int32_t)((seed >> 16) % (unsigned)D);
        off_h[i] = i;
    }
    off_h[T * B] = T * B;

    if (cudaMalloc((void **)&x_d, sizeof(float) * (size_t)B * D) != cudaSuccess ||
        cudaMalloc((void **)&out_d, sizeof(float) * (size_t)B * W) != cudaSuccess ||
        cudaMalloc((void **)&idx_d, sizeof(int32_t) * (size_t)T * B) != cudaSuccess ||
        cudaMalloc((void **)&off_d, sizeof(int32_t) * ((size_t)T * B + 1)) != cudaSuccess ||
        cudaMalloc((void **)&st_d, sizeof(int32_t)) != cudaSuccess) {
        fprintf(stderr, "c_abi_smoke: cudaMalloc failed\n");
        return 1;
    }
    for (int t = 0; t < T; ++t) {
        rows[t] = D;
        if (cudaMalloc(&tab_d[t], sizeof(float) * (size_t)D * D) != cudaSuccess) return 1;
        cudaMemcpy(tab_d[t], tab_h, sizeof(float) * (size_t)D * D, cudaMemcpyHostToDevice);
    }
    cudaMemcpy(x_d, x_h, sizeof(float) * (size_t)B * D, cudaMemcpyHostToDevice);
    cudaMemcpy(idx_d, idx_h, sizeof(int32_t) * (size_t)T * B, cudaMemcpyHostToDevice);
    cudaMemcpy(off_d, off_h, sizeof(int32_t) * ((size_t)T * B + 1), cudaMemcpyHostToDevice);
    cudaMemset(st_d, 0, sizeof(int32_t));
    {
        dlrm_tables tb = {T, D, DLRM_F32, tab_d, rows};
        dlrm_bags bags = {B, (int64_t)T * B, DLRM_I32, idx_d, off_d};
        CHECK(dlrm_sparse_fwd(&tb, &bags, DLRM_POOL_SUM, x_d, out_d, NULL, st_d, 0) == DLRM_OK);
    }
    CHECK(cudaDeviceSynchronize() == cudaSuccess);
    cudaMemcpy(out_h, out_d, sizeof(float) * (size_t)B * W, cudaMemcpyDeviceToHost);
    cudaMemcpy(&st_h, st_d, sizeof(int32_t), cudaMemcpyDeviceToHost);
    CHECK(st_h == DLRM_OK);
    for (int b = 0; b < B && !bad; ++b) {
        const float *o = out_h + (size_t)b * W;
        int k = D;
        for (int d = 0; d < D; ++d)
            if (o[d] != x_h[b * D + d]) bad = 1;
        for (int i = 0; i < N; ++i)
            for (int j = i + 1; j < N; ++j, ++k) {
                const int rj = idx_h[(j - 1) * B + b];
                const float want = i == 0 ? x_h[b * D + rj] : (float)(idx_h[(i - 1) * B + b] == rj);
                if (o[k] != want) {
                    fprintf(stderr, "c_abi_smoke: T=%d D=%d sample %d pair (%d,%d): %g, want %g\n", T, D, b,
                            i, j, o[k], want);
                    bad = 1;
                    break;
                }
            }
    }
    CHECK(!bad);
    for (int t = 0; t < T; ++t) cudaFree(tab_d[t]);
    cudaFree(x_d);
    cudaFree(out_d);
    cudaFree(idx_d);
    cudaFree(off_d);
    cudaFree(st_d);
    free(tab_h);
    free(x_h);
    free(out_h);
    free(idx_h);
    free(off_h);
    return bad;
}

int main(int argc, char **argv)
{
    const int gpu = argc > 1 && strcmp(argv[1], "--gpu") == 0;
    host_checks();
    if (gpu) {
        identity_forward(4, 16, 37);    /* register-blocked FFMA Gram */
        identity_forward(26, 128, 333); /* tensor-core Gram, several tiles per CTA */
        identity_forward(40, 64, 257);  /* tensor-core Gram, two samples per tile */
    }
    if (failures) {
        fprintf(stderr, "c_abi_smoke: %d check(s) failed\n", failures);
        return 1;
    }
    printf("c abi smoke ok%s\n", gpu ? " (with device forwards)" : "");
    return 0;
}
