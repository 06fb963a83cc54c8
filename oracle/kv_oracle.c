/*
 * kv_oracle.c -- plain CPU definition of paged KV gather (store) and scatter (load).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file.  Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (no approximation; the result is a permutation of bytes):
 *
 *   KV cache pages.  PagedAttention splits a request's KV cache into fixed pages of
 *   `page_size` tokens; a per-request page table maps logical page j to a physical page
 *   id in a pool ("Strata Guide", section "The Conflict Between PagedAttention and
 *   Transfer Efficiency", fragmentation figure: Page 12 -> Page 84 -> ...).  The GPU keeps
 *   a compute-friendly layer-first layout [L, P, H, D] (same page, section "Two-Dimensional
 *   Memory Layout Decoupling", item 1).  Here that is one pool per (kv, layer), each laid
 *   out as [num_pages][page_size][token_bytes]; kv = 0 is K, kv = 1 is V, and a latent
 *   (MLA) cache has kv_factor = 1.  Token t of a request lives in physical slot
 *   page_table[t / page_size] * page_size + t % page_size of every pool.
 *
 *   Chunks.  Host/storage memory keeps a transfer-friendly page-first layout [P, L, H, D]
 *   (same section, item 2): a chunk holds a run of tokens [t0, t0+n) of one request for a
 *   run of layers [l0, l0+nl).  Three layouts are defined:
 *     LAYER_MAJOR (0): [layer][kv][token][token_bytes]   -- page-first generalised to a
 *                      multi-page chunk; with one page per chunk and K/V folded it is the
 *                      page's host layout.
 *     TOKEN_MAJOR (1): [token][layer][kv][token_bytes]
 *     STRIPED     (2): one object per (layer, kv) in [layer][kv] order, each holding the
 *                      chunk's tokens of that layer and kv back to back, and each starting
 *                      at a multiple of 4096 bytes from the chunk start (the object's
 *                      length rounded up to 4096 is the stride).  This is the per-block
 *                      object layout of "Tutti: Making SSD-Backed KV Cache Practical",
 *                      section 2 Design 1 and Figure 4 (2L objects per KV block, stored
 *                      aligned to the block granularity of the NVMe file).
 *
 *   store: every token vector of every covered (layer, kv, token) is copied from its page
 *          slot into its chunk position.
 *   load:  the inverse assignment.
 *   Both are restricted to the half-open layer window [layer_begin, layer_end) intersected
 *   with each chunk's own layers; chunk positions stay relative to the chunk's l0.
 *
 * The loops follow the definition in the order chunk, layer, kv, token and move one whole
 * token vector with memcpy.  No blocking, fusion or reordering.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ORA_LAYER_MAJOR 0
#define ORA_TOKEN_MAJOR 1
#define ORA_STRIPED 2
#define ORA_STRIPE_ALIGN 4096

#define ORA_OK 0
#define ORA_EBADARG (-1)
#define ORA_ETOKENS (-2)
#define ORA_EPAGE (-3)
#define ORA_ELAYER (-4)

typedef struct {
    int32_t num_layers;
    int32_t kv_factor;      /* 2: separate K and V pools, 1: one latent pool */
    int32_t page_size;      /* tokens per page */
    int32_t num_pages;      /* pages in each pool */
    int64_t token_bytes;    /* bytes of one token's vector in one pool */
    unsigned char **pools;  /* [kv_factor * num_layers]; pools[kv * num_layers + layer] */
} ora_pool;

typedef struct {
    const int32_t *page_table; /* logical page -> physical page id */
    int32_t n_tokens;          /* tokens of the request */
    int32_t n_pages;           /* entries in page_table */
} ora_request;

typedef struct {
    int32_t request;
    int32_t token_begin;
    int32_t n_tokens;
    int32_t layer_begin;
    int32_t n_layers;
    int32_t layout;
    unsigned char *ptr;
} ora_chunk;

/* Address of token t's vector for (layer, kv) in the page pools. */
static unsigned char *page_slot(const ora_pool *pool, const ora_request *req,
                                int32_t layer, int32_t kv, int32_t t)
{
    int64_t page = req->page_table[t / pool->page_size];
    int64_t slot = page * pool->page_size + (t % pool->page_size);
    return pool->pools[(int64_t)kv * pool->num_layers + layer] + slot * pool->token_bytes;
}

/* Address of token t's vector for (layer, kv) inside chunk c, per its layout. */
static unsigned char *chunk_slot(const ora_pool *pool, const ora_chunk *c,
                                 int32_t layer, int32_t kv, int32_t t)
{
    int64_t v = pool->token_bytes;
    int64_t KV = pool->kv_factor;
    int64_t lr = layer - c->layer_begin;
    int64_t tr = t - c->token_begin;
    int64_t index;
    if (c->layout == ORA_STRIPED) {
        int64_t object_bytes = (int64_t)c->n_tokens * v;
        int64_t stride = (object_bytes + ORA_STRIPE_ALIGN - 1) / ORA_STRIPE_ALIGN * ORA_STRIPE_ALIGN;
        return c->ptr + (lr * KV + kv) * stride + tr * v;
    }
    if (c->layout == ORA_LAYER_MAJOR)
        index = (lr * KV + kv) * c->n_tokens + tr;
    else
        index = (tr * c->n_layers + lr) * KV + kv;
    return c->ptr + index * v;
}

static int check(const ora_pool *pool, const ora_request *reqs, int n_req,
                 const ora_chunk *chunks, int n_chunks, int layer_begin, int layer_end)
{
    if (!pool || !pool->pools || pool->num_layers <= 0 || pool->page_size <= 0 ||
        pool->num_pages <= 0 || pool->token_bytes <= 0 ||
        (pool->kv_factor != 1 && pool->kv_factor != 2))
        return ORA_EBADARG;
    if (n_req < 0 || n_chunks < 0 || (n_chunks > 0 && (!chunks || !reqs)))
        return ORA_EBADARG;
    if (layer_begin < 0 || layer_end > pool->num_layers || layer_begin > layer_end)
        return ORA_ELAYER;
    for (int i = 0; i < n_chunks; ++i) {
        const ora_chunk *c = &chunks[i];
        if (c->request < 0 || c->request >= n_req || !c->ptr ||
            (c->layout != ORA_LAYER_MAJOR && c->layout != ORA_TOKEN_MAJOR &&
             c->layout != ORA_STRIPED))
            return ORA_EBADARG;
        const ora_request *r = &reqs[c->request];
        if (c->token_begin < 0 || c->n_tokens < 0 ||
            (int64_t)c->token_begin + c->n_tokens > r->n_tokens)
            return ORA_ETOKENS;
        if (c->layer_begin < 0 || c->n_layers < 0 ||
            c->layer_begin + c->n_layers > pool->num_layers)
            return ORA_ELAYER;
        for (int32_t t = c->token_begin; t < c->token_begin + c->n_tokens; ++t) {
            int32_t j = t / pool->page_size;
            if (j >= r->n_pages)
                return ORA_ETOKENS;
            if (r->page_table[j] < 0 || r->page_table[j] >= pool->num_pages)
                return ORA_EPAGE;
        }
    }
    return ORA_OK;
}

/* dir 0 = store (pages -> chunks), dir 1 = load (chunks -> pages). */
static int transfer(int dir, const ora_pool *pool, const ora_request *reqs, int n_req,
                    const ora_chunk *chunks, int n_chunks, int layer_begin, int layer_end)
{
    int rc = check(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end);
    if (rc != ORA_OK)
        return rc;
    size_t v = (size_t)pool->token_bytes;
    for (int i = 0; i < n_chunks; ++i) {
        const ora_chunk *c = &chunks[i];
        const ora_request *r = &reqs[c->request];
        int32_t l_lo = c->layer_begin > layer_begin ? c->layer_begin : layer_begin;
        int32_t l_hi = c->layer_begin + c->n_layers < layer_end ? c->layer_begin + c->n_layers
                                                                : layer_end;
        for (int32_t l = l_lo; l < l_hi; ++l)
            for (int32_t kv = 0; kv < pool->kv_factor; ++kv)
                for (int32_t t = c->token_begin; t < c->token_begin + c->n_tokens; ++t) {
                    unsigned char *p = page_slot(pool, r, l, kv, t);
                    unsigned char *q = chunk_slot(pool, c, l, kv, t);
                    if (dir == 0)
                        memcpy(q, p, v);
                    else
                        memcpy(p, q, v);
                }
    }
    return ORA_OK;
}

int ora_store(const ora_pool *pool, const ora_request *reqs, int n_req,
              const ora_chunk *chunks, int n_chunks, int layer_begin, int layer_end)
{
    return transfer(0, pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end);
}

int ora_load(const ora_pool *pool, const ora_request *reqs, int n_req,
             const ora_chunk *chunks, int n_chunks, int layer_begin, int layer_end)
{
    return transfer(1, pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end);
}

/* Bytes the call moves: the sum over chunks of covered layers x kv x tokens x token_bytes. */
int64_t ora_bytes(const ora_pool *pool, const ora_chunk *chunks, int n_chunks,
                  int layer_begin, int layer_end)
{
    int64_t total = 0;
    for (int i = 0; i < n_chunks; ++i) {
        const ora_chunk *c = &chunks[i];
        int32_t l_lo = c->layer_begin > layer_begin ? c->layer_begin : layer_begin;
        int32_t l_hi = c->layer_begin + c->n_layers < layer_end ? c->layer_begin + c->n_layers
                                                                : layer_end;
        if (l_hi > l_lo)
            total += (int64_t)(l_hi - l_lo) * pool->kv_factor * c->n_tokens * pool->token_bytes;
    }
    return total;
}
