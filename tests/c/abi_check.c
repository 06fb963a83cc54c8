/*
 * abi_check.c -- uses the library through include/kvx.h from plain C99, with no GPU:
 * prints the sizes of the ABI structs and the results of the host-only entry points
 * (validation, work counts, chunk policy, time model), one "name value" pair per line,
 * for tests/test_c_abi.py to compare with the Python binding and the closed forms.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>

#include "kvx.h"

int main(void)
{
    /* One request of 1000 tokens on 16-token pages, K/V, 4 layers of 2 KiB token vectors.
     * The pool's "device" pointers are never dereferenced by these calls. */
    void *k[4], *v[4];
    for (int l = 0; l < 4; ++l) {
        k[l] = (void *)(uintptr_t)(0x100000u * (l + 1));
        v[l] = (void *)(uintptr_t)(0x1000000u * (l + 1));
    }
    kvx_pool pool = {4, 2, 16, 128, 2048, (void *const *)k, (void *const *)v};
    int32_t table[63];
    for (int i = 0; i < 63; ++i)
        table[i] = 2 * i;
    kvx_request req = {(const int32_t *)(uintptr_t)0x2000, table, 1000, 0};
    kvx_chunk chunks[3] = {
        {0, 0, 256, 0, 4, KVX_CHUNK_LAYER_MAJOR, (void *)(uintptr_t)0x10000000u},
        {0, 256, 300, 0, 4, KVX_CHUNK_TOKEN_MAJOR, (void *)(uintptr_t)0x20000000u},
        {0, 556, 444, 1, 2, KVX_CHUNK_STRIPED, (void *)(uintptr_t)0x30000000u},
    };

    printf("sizeof_pool %zu\n", sizeof(kvx_pool));
    printf("sizeof_request %zu\n", sizeof(kvx_request));
    printf("sizeof_chunk %zu\n", sizeof(kvx_chunk));
    printf("sizeof_cfg %zu\n", sizeof(kvx_launch_cfg));
    printf("sizeof_link_model %zu\n", sizeof(kvx_link_model));
    printf("version %d\n", kvx_version());
#define OFF(type, field) printf("off_%s_%s %zu\n", #type, #field, offsetof(type, field))
    OFF(kvx_pool, num_layers); OFF(kvx_pool, kv_factor); OFF(kvx_pool, page_size);
    OFF(kvx_pool, num_pages); OFF(kvx_pool, token_bytes); OFF(kvx_pool, k_pages);
    OFF(kvx_pool, v_pages);
    OFF(kvx_request, page_table); OFF(kvx_request, page_table_host);
    OFF(kvx_request, n_tokens); OFF(kvx_request, reserved);
    OFF(kvx_chunk, request); OFF(kvx_chunk, token_begin); OFF(kvx_chunk, n_tokens);
    OFF(kvx_chunk, layer_begin); OFF(kvx_chunk, n_layers); OFF(kvx_chunk, layout);
    OFF(kvx_chunk, ptr);
    OFF(kvx_launch_cfg, sm_cap); OFF(kvx_launch_cfg, ctas_per_sm); OFF(kvx_launch_cfg, threads);
    OFF(kvx_launch_cfg, unroll); OFF(kvx_launch_cfg, store_hint); OFF(kvx_launch_cfg, mapping);
    OFF(kvx_launch_cfg, stage_bytes); OFF(kvx_launch_cfg, batch); OFF(kvx_launch_cfg, overlap);
    OFF(kvx_link_model, h2d_gbs); OFF(kvx_link_model, d2h_gbs); OFF(kvx_link_model, hbm_gbs);
    OFF(kvx_link_model, bidir_gbs); OFF(kvx_link_model, latency_us);
    OFF(kvx_link_model, launch_us); OFF(kvx_link_model, num_sms); OFF(kvx_link_model, reserved);
#undef OFF

    char msg[256];
    printf("validate_ok %d\n",
           (int)kvx_validate(&pool, &req, 1, chunks, 3, 0, 4, KVX_OP_STORE, 1, msg, sizeof msg));
    kvx_chunk bad = chunks[0];
    bad.ptr = (void *)(uintptr_t)0x10000008u; /* not 16-byte aligned */
    printf("validate_misaligned %d\n",
           (int)kvx_validate(&pool, &req, 1, &bad, 1, 0, 4, KVX_OP_STORE, 1, msg, sizeof msg));
    bad = chunks[0];
    bad.n_tokens = 2000; /* past the request */
    printf("validate_tokens %d\n",
           (int)kvx_validate(&pool, &req, 1, &bad, 1, 0, 4, KVX_OP_STORE, 1, msg, sizeof msg));

    int64_t segments = 0, bytes = 0;
    kvx_plan_count(&pool, &req, 1, chunks, 3, 0, 4, &segments, &bytes);
    printf("segments %lld\n", (long long)segments);
    printf("bytes %lld\n", (long long)bytes);
    kvx_plan_count(&pool, &req, 1, chunks, 3, 1, 3, &segments, &bytes);
    printf("segments_window %lld\n", (long long)segments);
    printf("bytes_window %lld\n", (long long)bytes);

    int32_t tokens = 0, layers = 0;
    kvx_chunk_policy(&pool, 0, 0, &tokens, &layers);
    printf("policy_tokens %d\n", tokens);
    printf("policy_layers %d\n", layers);
    kvx_chunk_policy(&pool, 1, 1 << 20, &tokens, &layers);
    printf("policy_stream_tokens %d\n", tokens);
    printf("policy_stream_layers %d\n", layers);

    kvx_link_model m;
    kvx_default_link_model(&m);
    double us = 0;
    kvx_estimate_us(&m, KVX_OP_LOAD, (int64_t)1 << 32, NULL, &us);
    printf("estimate_load_us %.6f\n", us);
    kvx_estimate_pair_us(&m, KVX_OP_ROUNDTRIP, (int64_t)1 << 32, (int64_t)1 << 32, 32768, NULL,
                         &us);
    printf("estimate_roundtrip_us %.6f\n", us);
    printf("status_string_overlap %s\n", kvx_status_string(KVX_ERR_OVERLAP));
    return 0;
}
