/*
 * roundtrip_gpu.c -- a plain C99 user of the library on the GPU, with no Python and no
 * torch: device pools from cudaMalloc, chunks from kvx_host_alloc, one kvx_roundtrip_chunks
 * (store the request's pages into host chunks, load them into other pages, one launch),
 * then one kvx_transform_hbm gather of the loaded pages into device chunks, then a store and
 * a load with the bulk-copy mapping on 2 SMs.  Every byte of the chunks and of the pools is
 * compared with the CPU oracle (oracle/kv_oracle.c, compiled into this test program), run on
 * host copies of the same inputs.
 *
 * Prints "name value" lines and exits 0 only when every comparison holds.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "kvx.h"
#include "kv_oracle.c"

#define L 3
#define KV 2
#define P 16
#define V 192 /* token bytes: a multiple of 16, not of 32 */
#define NP 64
#define NT 300 /* 19 pages, the last one holding 12 tokens */
#define NPG ((NT + P - 1) / P)
#define NCHUNK 3
#define CANARY 0xA5

static int failures = 0;

#define CHECK_CUDA(call)                                                                  \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess) {                                                          \
            printf("cuda_error %s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            exit(2);                                                                      \
        }                                                                                 \
    } while (0)

#define CHECK_KVX(ctx, call)                                                             \
    do {                                                                                 \
        kvx_status s_ = (call);                                                          \
        if (s_ != KVX_OK) {                                                              \
            printf("kvx_error %s:%d %s: %s\n", __FILE__, __LINE__, kvx_status_string(s_), \
                   kvx_last_error(ctx));                                                 \
            exit(3);                                                                     \
        }                                                                                \
    } while (0)

static uint32_t lcg(uint32_t *state)
{
    *state = *state * 1664525u + 1013904223u;
    return *state >> 8;
}

static void compare(const char *what, const unsigned char *got, const unsigned char *exp,
                    size_t n)
{
    size_t bad = 0, first = n;
    for (size_t i = 0; i < n; ++i)
        if (got[i] != exp[i]) {
            if (!bad)
                first = i;
            ++bad;
        }
    printf("%s_mismatches %zu\n", what, bad);
    if (bad) {
        printf("%s_first_mismatch %zu\n", what, first);
        ++failures;
    }
}

static int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int main(void)
{
    const size_t pool_bytes = (size_t)NP * P * V;
    uint32_t rng = 20260u;

    /* Pools: device copies for the library, host copies for the oracle. */
    void *dev_pools[KV * L];
    unsigned char *host_pools[KV * L], *exp_pools[KV * L];
    for (int i = 0; i < KV * L; ++i) {
        host_pools[i] = malloc(pool_bytes);
        exp_pools[i] = malloc(pool_bytes);
        if (!host_pools[i] || !exp_pools[i])
            return 4;
        for (size_t b = 0; b < pool_bytes; ++b)
            host_pools[i][b] = (unsigned char)lcg(&rng);
        CHECK_CUDA(cudaMalloc(&dev_pools[i], pool_bytes));
        CHECK_CUDA(cudaMemcpy(dev_pools[i], host_pools[i], pool_bytes, cudaMemcpyHostToDevice));
    }

    /* Page tables: a seeded permutation of the pool; the store's pages first, then the
     * load's, disjoint. */
    int32_t perm[NP];
    for (int i = 0; i < NP; ++i)
        perm[i] = i;
    for (int i = NP - 1; i > 0; --i) {
        int j = (int)(lcg(&rng) % (uint32_t)(i + 1));
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    int32_t *dev_src_table, *dev_dst_table;
    CHECK_CUDA(cudaMalloc((void **)&dev_src_table, NPG * sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc((void **)&dev_dst_table, NPG * sizeof(int32_t)));
    CHECK_CUDA(cudaMemcpy(dev_src_table, perm, NPG * sizeof(int32_t), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dev_dst_table, perm + NPG, NPG * sizeof(int32_t),
                          cudaMemcpyHostToDevice));

    /* Three chunks of the request, one per layout; the last is partial (44 tokens). */
    const int32_t t0[NCHUNK] = {0, 128, 256}, nt[NCHUNK] = {128, 128, 44};
    const int32_t layout[NCHUNK] = {KVX_CHUNK_LAYER_MAJOR, KVX_CHUNK_TOKEN_MAJOR,
                                    KVX_CHUNK_STRIPED};
    int64_t off[NCHUNK], arena_bytes = 0;
    for (int c = 0; c < NCHUNK; ++c) {
        int64_t bytes = layout[c] == KVX_CHUNK_STRIPED
                            ? (int64_t)L * KV * round_up((int64_t)nt[c] * V, KVX_STRIPE_ALIGN)
                            : (int64_t)L * KV * nt[c] * V;
        off[c] = arena_bytes;
        arena_bytes = round_up(arena_bytes + bytes, 4096);
    }
    const size_t total = (size_t)arena_bytes + 4096; /* canary tail */
    unsigned char *arena = NULL, *exp_arena = malloc(total), *got = malloc(total);
    if (!exp_arena || !got)
        return 4;
    CHECK_KVX(NULL, kvx_host_alloc((void **)&arena, total));
    memset(arena, CANARY, total);

    void *k_pages[L], *v_pages[L];
    for (int l = 0; l < L; ++l) {
        k_pages[l] = dev_pools[l];
        v_pages[l] = dev_pools[L + l];
    }
    kvx_pool pool = {L, KV, P, NP, V, (void *const *)k_pages, (void *const *)v_pages};
    kvx_request src = {dev_src_table, perm, NT, 0};
    kvx_request dst = {dev_dst_table, perm + NPG, NT, 0};
    kvx_chunk chunks[NCHUNK];
    for (int c = 0; c < NCHUNK; ++c) {
        kvx_chunk ch = {0, t0[c], nt[c], 0, L, layout[c], arena + off[c]};
        chunks[c] = ch;
    }

    /* The round trip, through the C ABI. */
    kvx_ctx *ctx = NULL;
    CHECK_KVX(NULL, kvx_create(&ctx, 0, 0));
    CHECK_KVX(ctx, kvx_set_validation(ctx, 2));
    CHECK_KVX(ctx, kvx_roundtrip_chunks(ctx, &pool, &src, &dst, 1, chunks, NCHUNK, 0, L, NULL,
                                        NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    uint32_t flags = 0;
    CHECK_KVX(ctx, kvx_get_status(ctx, NULL, &flags));
    printf("roundtrip_device_flags %u\n", flags);

    /* The oracle on host copies: store from the source pages into a canary arena, then
     * load that arena into the destination pages. */
    memset(exp_arena, CANARY, total);
    ora_pool opool = {L, KV, P, NP, V, host_pools};
    ora_request osrc = {perm, NT, NPG}, odst = {perm + NPG, NT, NPG};
    ora_chunk ochunks[NCHUNK];
    for (int c = 0; c < NCHUNK; ++c) {
        ora_chunk oc = {0, t0[c], nt[c], 0, L, layout[c], exp_arena + off[c]};
        ochunks[c] = oc;
    }
    if (ora_store(&opool, &osrc, 1, ochunks, NCHUNK, 0, L) != ORA_OK)
        return 5;
    for (int i = 0; i < KV * L; ++i)
        memcpy(exp_pools[i], host_pools[i], pool_bytes);
    ora_pool oexp = {L, KV, P, NP, V, exp_pools};
    if (ora_load(&oexp, &odst, 1, ochunks, NCHUNK, 0, L) != ORA_OK)
        return 5;
    compare("roundtrip_chunks", arena, exp_arena, total);
    for (int i = 0; i < KV * L; ++i) {
        CHECK_CUDA(cudaMemcpy(got, dev_pools[i], pool_bytes, cudaMemcpyDeviceToHost));
        char name[32];
        snprintf(name, sizeof name, "roundtrip_pool%d", i);
        compare(name, got, exp_pools[i], pool_bytes);
    }

    /* HBM transform: gather the loaded destination pages into device chunks. */
    unsigned char *dev_arena = NULL;
    CHECK_CUDA(cudaMalloc((void **)&dev_arena, total));
    CHECK_CUDA(cudaMemset(dev_arena, CANARY, total));
    for (int c = 0; c < NCHUNK; ++c)
        chunks[c].ptr = dev_arena + off[c];
    CHECK_KVX(ctx, kvx_set_validation(ctx, 1));
    CHECK_KVX(ctx, kvx_transform_hbm(ctx, KVX_DIR_GATHER, &pool, &dst, 1, chunks, NCHUNK, 0, L,
                                     NULL, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_KVX(ctx, kvx_get_status(ctx, NULL, &flags));
    printf("transform_device_flags %u\n", flags);
    memset(exp_arena, CANARY, total);
    if (ora_store(&oexp, &odst, 1, ochunks, NCHUNK, 0, L) != ORA_OK)
        return 5;
    CHECK_CUDA(cudaMemcpy(got, dev_arena, total, cudaMemcpyDeviceToHost));
    compare("transform_chunks", got, exp_arena, total);

    /* The bulk-copy mapping on 2 SMs: store the destination pages into a second host arena
     * (the oracle's expectation is the arena just compared), then load that arena into the
     * source pages. */
    unsigned char *arena2 = NULL;
    CHECK_KVX(NULL, kvx_host_alloc((void **)&arena2, total));
    memset(arena2, CANARY, total);
    for (int c = 0; c < NCHUNK; ++c)
        chunks[c].ptr = arena2 + off[c];
    kvx_launch_cfg bcfg;
    CHECK_KVX(ctx, kvx_default_launch_cfg(ctx, KVX_OP_STORE, &bcfg));
    bcfg.sm_cap = 2;
    bcfg.mapping = KVX_MAP_BULK;
    bcfg.threads = 0;
    bcfg.unroll = 3;
    bcfg.stage_bytes = 4096;
    CHECK_KVX(ctx, kvx_store_chunks(ctx, &pool, &dst, 1, chunks, NCHUNK, 0, L, &bcfg, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_KVX(ctx, kvx_get_status(ctx, NULL, &flags));
    printf("bulk_store_device_flags %u\n", flags);
    compare("bulk_store_chunks", arena2, exp_arena, total);
    CHECK_KVX(ctx, kvx_default_launch_cfg(ctx, KVX_OP_LOAD, &bcfg));
    bcfg.sm_cap = 2;
    bcfg.mapping = KVX_MAP_BULK;
    bcfg.threads = 0;
    bcfg.unroll = 3;
    bcfg.stage_bytes = 4096;
    CHECK_KVX(ctx, kvx_load_chunks(ctx, &pool, &src, 1, chunks, NCHUNK, 0, L, &bcfg, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_KVX(ctx, kvx_get_status(ctx, NULL, &flags));
    printf("bulk_load_device_flags %u\n", flags);
    if (ora_load(&oexp, &osrc, 1, ochunks, NCHUNK, 0, L) != ORA_OK)
        return 5;
    for (int i = 0; i < KV * L; ++i) {
        CHECK_CUDA(cudaMemcpy(got, dev_pools[i], pool_bytes, cudaMemcpyDeviceToHost));
        char name[32];
        snprintf(name, sizeof name, "bulk_load_pool%d", i);
        compare(name, got, exp_pools[i], pool_bytes);
    }
    kvx_host_free(arena2);

    kvx_destroy(ctx);
    CHECK_CUDA(cudaFree(dev_arena));
    kvx_host_free(arena);
    for (int i = 0; i < KV * L; ++i) {
        CHECK_CUDA(cudaFree(dev_pools[i]));
        free(host_pools[i]);
        free(exp_pools[i]);
    }
    CHECK_CUDA(cudaFree(dev_src_table));
    CHECK_CUDA(cudaFree(dev_dst_table));
    free(exp_arena);
    free(got);
    printf("failures %d\n", failures);
    return failures ? 1 : 0;
}
