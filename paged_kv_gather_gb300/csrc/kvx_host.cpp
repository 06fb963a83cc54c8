// kvx_host.cpp -- host logic of the KV gather/scatter library: validation, descriptor
// packing, segment counting, the chunk-size policy.  Runs without a GPU except for the
// pointer-attribute checks of validation level 2.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "kvx_internal.h"
#include "kvx_rules.h"

namespace kvx {
namespace {

kvx_status fail(kvx_status st, char *msg, size_t len, const char *fmt, ...)
{
    if (msg && len > 0) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(msg, len, fmt, ap);
        va_end(ap);
    }
    return st;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool op_is_scatter(int op) { return op == KVX_OP_LOAD || op == KVX_OP_SCATTER_HBM; }

// Largest page (page_size x token_bytes) a pool may have: 2^30 16-byte units; and the
// largest token.
constexpr int64_t kMaxPageBytes = int64_t(1) << 34;
constexpr int64_t kMaxTokenBytes = int64_t(1) << 30;

int64_t pages_of(int64_t n_tokens, int64_t page_size)
{
    return (n_tokens + page_size - 1) / page_size;
}

// Level 2: the memory behind p must be reachable by the GPU at the same address.
kvx_status check_pointer(const void *p, bool want_host, const char *what, int index, char *msg,
                         size_t len)
{
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(KVX_ERR_CUDA, msg, len, "%s %d: cudaPointerGetAttributes: %s", what, index,
                    cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeUnregistered)
        return fail(KVX_ERR_NOT_DEVICE_ACCESSIBLE, msg, len,
                    "%s %d: pageable host memory; allocate with kvx_host_alloc or pin it with "
                    "kvx_host_register", what, index);
    if (a.devicePointer != p)
        return fail(KVX_ERR_NOT_DEVICE_ACCESSIBLE, msg, len,
                    "%s %d: not mapped at the same address on the device", what, index);
    if (want_host && a.type == cudaMemoryTypeDevice)
        return fail(KVX_ERR_INVALID_ARG, msg, len,
                    "%s %d: device memory; store/load take host chunks (use kvx_transform_hbm)",
                    what, index);
    if (!want_host && a.type == cudaMemoryTypeHost)
        return fail(KVX_ERR_INVALID_ARG, msg, len,
                    "%s %d: host memory where device memory is required", what, index);
    return KVX_OK;
}

struct SlotUse {
    int64_t slot;  // page * page_size + token % page_size
    int32_t lo, hi;  // layers written
    int32_t chunk;
};

}  // namespace

kvx_status validate(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                    const kvx_chunk *chunks, int n_chunks, int layer_begin, int layer_end,
                    int op, int level, bool have_gpu, char *msg, size_t len)
{
    if (msg && len > 0)
        msg[0] = '\0';
    if (op < KVX_OP_STORE || op > KVX_OP_SCATTER_HBM)
        return fail(KVX_ERR_INVALID_ARG, msg, len, "unknown operation %d", op);
    // Always: what the packer itself relies on.
    if (!pool)
        return fail(KVX_ERR_INVALID_ARG, msg, len, "pool is NULL");
    if (pool->num_layers <= 0 || (pool->kv_factor != 1 && pool->kv_factor != 2) ||
        pool->page_size <= 0 || pool->num_pages <= 0 || pool->token_bytes <= 0)
        return fail(KVX_ERR_INVALID_ARG, msg, len,
                    "pool: num_layers %d, kv_factor %d, page_size %d, num_pages %d, "
                    "token_bytes %lld", pool->num_layers, pool->kv_factor, pool->page_size,
                    pool->num_pages, (long long)pool->token_bytes);
    if (pool->token_bytes % 16 != 0)
        return fail(KVX_ERR_ALIGNMENT, msg, len, "token_bytes %lld is not a multiple of 16",
                    (long long)pool->token_bytes);
    // The kernels count a page segment's 16-byte units, and a token's bytes, in 32 bits.
    if (int64_t(pool->page_size) * pool->token_bytes > kMaxPageBytes ||
        pool->token_bytes > kMaxTokenBytes)
        return fail(KVX_ERR_INVALID_ARG, msg, len,
                    "a page of %d x %lld bytes exceeds 16 GiB, or a token 1 GiB",
                    pool->page_size, (long long)pool->token_bytes);
    if (!pool->k_pages || (pool->kv_factor == 2 && !pool->v_pages))
        return fail(KVX_ERR_INVALID_ARG, msg, len, "pool layer pointer array is NULL");
    if (n_req < 0 || n_chunks < 0 || (n_req > 0 && !reqs) || (n_chunks > 0 && !chunks))
        return fail(KVX_ERR_INVALID_ARG, msg, len, "bad request/chunk arrays (%d, %d)", n_req,
                    n_chunks);
    if (layer_begin < 0 || layer_end > pool->num_layers || layer_begin > layer_end)
        return fail(KVX_ERR_INVALID_ARG, msg, len, "layer window [%d, %d) outside [0, %d)",
                    layer_begin, layer_end, pool->num_layers);
    // Every index the kernel derives from a descriptor (request, page-table entry, layer,
    // pool) stays inside its array, whatever the level.
    for (int r = 0; r < n_req; ++r) {
        if (reqs[r].n_tokens < 0)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "request %d: n_tokens %d", r,
                        reqs[r].n_tokens);
        if (reqs[r].n_tokens > 0 && !reqs[r].page_table)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "request %d: page_table is NULL", r);
    }
    for (int c = 0; c < n_chunks; ++c) {
        const kvx_chunk &ch = chunks[c];
        if (ch.request < 0 || ch.request >= n_req)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "chunk %d: request %d of %d", c,
                        ch.request, n_req);
        if (ch.n_tokens < 0 || ch.n_layers < 0)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "chunk %d: negative size", c);
        const kvx_request &rq = reqs[ch.request];
        if (ch.token_begin < 0 || (int64_t)ch.token_begin + ch.n_tokens > rq.n_tokens)
            return fail(KVX_ERR_INVALID_ARG, msg, len,
                        "chunk %d: tokens [%d, %lld) outside request %d's %d tokens", c,
                        ch.token_begin, (long long)ch.token_begin + ch.n_tokens, ch.request,
                        rq.n_tokens);
        if (ch.layer_begin < 0 || (int64_t)ch.layer_begin + ch.n_layers > pool->num_layers)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "chunk %d: layers [%d, %lld) outside "
                        "[0, %d)", c, ch.layer_begin,
                        (long long)ch.layer_begin + ch.n_layers, pool->num_layers);
        if (ch.layout != KVX_CHUNK_LAYER_MAJOR && ch.layout != KVX_CHUNK_TOKEN_MAJOR &&
            ch.layout != KVX_CHUNK_STRIPED)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "chunk %d: layout %d", c, ch.layout);
    }
    if (level <= 0)
        return KVX_OK;

    // Level 1: O(layers + chunks) pointer and alignment checks.
    for (int k = 0; k < pool->kv_factor; ++k) {
        void *const *arr = k == 0 ? pool->k_pages : pool->v_pages;
        for (int l = 0; l < pool->num_layers; ++l) {
            if (!arr[l])
                return fail(KVX_ERR_INVALID_ARG, msg, len, "pool %c layer %d is NULL",
                            k ? 'V' : 'K', l);
            if (!aligned16(arr[l]))
                return fail(KVX_ERR_ALIGNMENT, msg, len, "pool %c layer %d not 16-B aligned",
                            k ? 'V' : 'K', l);
        }
    }
    for (int c = 0; c < n_chunks; ++c) {
        const kvx_chunk &ch = chunks[c];
        if (!ch.ptr)
            return fail(KVX_ERR_INVALID_ARG, msg, len, "chunk %d: ptr is NULL", c);
        if (!aligned16(ch.ptr))
            return fail(KVX_ERR_ALIGNMENT, msg, len, "chunk %d: ptr not 16-B aligned", c);
    }
    if (level <= 1)
        return KVX_OK;

    // Level 2: page ids against host copies, load-destination overlap, pointer attributes.
    for (int r = 0; r < n_req; ++r) {
        const int32_t *pt = reqs[r].page_table_host;
        if (!pt)
            continue;
        int64_t n = pages_of(reqs[r].n_tokens, pool->page_size);
        for (int64_t j = 0; j < n; ++j)
            if (pt[j] < 0 || pt[j] >= pool->num_pages)
                return fail(KVX_ERR_PAGE_OUT_OF_RANGE, msg, len,
                            "request %d: page_table[%lld] = %d outside [0, %d)", r,
                            (long long)j, pt[j], pool->num_pages);
    }
    if (op_is_scatter(op)) {
        std::vector<SlotUse> uses;
        for (int c = 0; c < n_chunks; ++c) {
            const kvx_chunk &ch = chunks[c];
            const int32_t *pt = reqs[ch.request].page_table_host;
            int lo, hi;
            chunk_layers(ch, layer_begin, layer_end, &lo, &hi);
            if (!pt || lo >= hi)
                continue;
            for (int32_t t = ch.token_begin; t < ch.token_begin + ch.n_tokens; ++t)
                uses.push_back({(int64_t)pt[t / pool->page_size] * pool->page_size +
                                    t % pool->page_size, lo, hi, c});
        }
        std::sort(uses.begin(), uses.end(), [](const SlotUse &a, const SlotUse &b) {
            return a.slot != b.slot ? a.slot < b.slot : a.lo < b.lo;
        });
        // Sorted by (slot, first layer): two uses of a slot overlap iff one starts below
        // the running end of the earlier ones.
        size_t i = 0;
        while (i < uses.size()) {
            size_t j = i + 1;
            int32_t run_hi = uses[i].hi;
            int32_t run_chunk = uses[i].chunk;
            while (j < uses.size() && uses[j].slot == uses[i].slot) {
                if (uses[j].lo < run_hi)
                    return fail(KVX_ERR_OVERLAP, msg, len,
                                "chunks %d and %d both write page slot %lld", run_chunk,
                                uses[j].chunk, (long long)uses[j].slot);
                if (uses[j].hi > run_hi) {
                    run_hi = uses[j].hi;
                    run_chunk = uses[j].chunk;
                }
                ++j;
            }
            i = j;
        }
    }
    if (have_gpu) {
        const bool chunks_on_host = op == KVX_OP_STORE || op == KVX_OP_LOAD;
        const void *last = nullptr;
        for (int c = 0; c < n_chunks; ++c) {
            if (chunks[c].ptr == last)
                continue;
            last = chunks[c].ptr;
            kvx_status st = check_pointer(chunks[c].ptr, chunks_on_host, "chunk", c, msg, len);
            if (st != KVX_OK)
                return st;
        }
        for (int k = 0; k < pool->kv_factor; ++k)
            for (int l = 0; l < pool->num_layers; ++l) {
                kvx_status st = check_pointer((k == 0 ? pool->k_pages : pool->v_pages)[l],
                                              false, "pool layer", l, msg, len);
                if (st != KVX_OK)
                    return st;
            }
    }
    return KVX_OK;
}

kvx_status validate_exchange(const kvx_pool *pool, const kvx_request *sreqs, int n_sreq,
                             const kvx_chunk *schunks, int n_schunks, const kvx_request *lreqs,
                             int n_lreq, const kvx_chunk *lchunks, int n_lchunks,
                             int layer_begin, int layer_end, int level, bool have_gpu,
                             char *msg, size_t len)
{
    kvx_status st = validate(pool, sreqs, n_sreq, schunks, n_schunks, layer_begin, layer_end,
                             KVX_OP_STORE, level, have_gpu, msg, len);
    if (st != KVX_OK)
        return st;
    st = validate(pool, lreqs, n_lreq, lchunks, n_lchunks, layer_begin, layer_end, KVX_OP_LOAD,
                  level, have_gpu, msg, len);
    if (st != KVX_OK || level < 2)
        return st;
    // A slot the store reads must not be one the load writes, for any common layer.
    auto slots = [&](const kvx_request *reqs, const kvx_chunk *chunks, int n) {
        std::vector<SlotUse> out;
        for (int c = 0; c < n; ++c) {
            const int32_t *pt = reqs[chunks[c].request].page_table_host;
            int lo, hi;
            chunk_layers(chunks[c], layer_begin, layer_end, &lo, &hi);
            if (!pt || lo >= hi)
                continue;
            for (int32_t t = chunks[c].token_begin;
                 t < chunks[c].token_begin + chunks[c].n_tokens; ++t)
                out.push_back({(int64_t)pt[t / pool->page_size] * pool->page_size +
                                   t % pool->page_size, lo, hi, c});
        }
        std::sort(out.begin(), out.end(), [](const SlotUse &a, const SlotUse &b) {
            return a.slot < b.slot;
        });
        return out;
    };
    const std::vector<SlotUse> reads = slots(sreqs, schunks, n_schunks);
    const std::vector<SlotUse> writes = slots(lreqs, lchunks, n_lchunks);
    size_t w = 0;
    for (const SlotUse &r : reads) {
        while (w < writes.size() && writes[w].slot < r.slot)
            ++w;
        for (size_t k = w; k < writes.size() && writes[k].slot == r.slot; ++k)
            if (writes[k].lo < r.hi && r.lo < writes[k].hi)
                return fail(KVX_ERR_OVERLAP, msg, len,
                            "store chunk %d reads page slot %lld that load chunk %d writes",
                            r.chunk, (long long)r.slot, writes[k].chunk);
    }
    return KVX_OK;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PackedLayout packed_layout(const kvx_pool *pool, int n_req, int n_chunks)
{
    PackedLayout lay;
    size_t off = 0;
    lay.off_item_begin = off;
    off = round_up(off + sizeof(int64_t) * (size_t)(n_chunks + 1), 128);
    lay.off_chunks = off;
    off = round_up(off + sizeof(DevChunk) * (size_t)n_chunks, 128);
    lay.off_reqs = off;
    off = round_up(off + sizeof(DevRequest) * (size_t)n_req, 128);
    lay.off_pools = off;
    off = round_up(off + sizeof(char *) * (size_t)pool->kv_factor * pool->num_layers, 128);
    lay.total = off;
    return lay;
}

Plan pack(const kvx_pool *pool, const kvx_request *reqs, int n_req, const kvx_chunk *chunks,
          int n_chunks, int layer_begin, int layer_end, int dir, const PackedLayout &lay,
          char *block, char *dev_block)
{
    int64_t *item_begin = reinterpret_cast<int64_t *>(block + lay.off_item_begin);
    DevChunk *dch = reinterpret_cast<DevChunk *>(block + lay.off_chunks);
    DevRequest *drq = reinterpret_cast<DevRequest *>(block + lay.off_reqs);
    char **pools = reinterpret_cast<char **>(block + lay.off_pools);
    const int64_t v = pool->token_bytes;
    const int32_t KV = pool->kv_factor;
    const int32_t P = pool->page_size;
    int64_t item = 0;
    for (int c = 0; c < n_chunks; ++c) {
        const kvx_chunk &ch = chunks[c];
        DevChunk &d = dch[c];
        int lo, hi;
        chunk_layers(ch, layer_begin, layer_end, &lo, &hi);
        d.ptr = static_cast<char *>(ch.ptr);
        if (ch.layout == KVX_CHUNK_LAYER_MAJOR) {
            d.slab_stride = (int64_t)ch.n_tokens * v;
            d.row_stride = v;
        } else if (ch.layout == KVX_CHUNK_STRIPED) {
            const int64_t obj = (int64_t)ch.n_tokens * v;
            d.slab_stride = (obj + KVX_STRIPE_ALIGN - 1) / KVX_STRIPE_ALIGN * KVX_STRIPE_ALIGN;
            d.row_stride = v;
        } else {
            d.slab_stride = v;
            d.row_stride = (int64_t)ch.n_layers * KV * v;
        }
        d.request = ch.request;
        d.t0 = ch.token_begin;
        d.t_end = ch.token_begin + ch.n_tokens;
        d.pf = ch.token_begin / P;
        d.np = (ch.n_tokens > 0 && lo < hi)
                   ? (ch.token_begin + ch.n_tokens - 1) / P - ch.token_begin / P + 1
                   : 0;
        d.la = lo;
        d.slab0 = (lo - ch.layer_begin) * KV;
        d.pad = 0;
        item_begin[c] = item;
        if (d.np > 0)
            item += (int64_t)(hi - lo) * KV * d.np;
    }
    item_begin[n_chunks] = item;
    for (int r = 0; r < n_req; ++r) {
        drq[r].page_table = reqs[r].page_table;
        drq[r].n_pages = (int32_t)pages_of(reqs[r].n_tokens, P);
        drq[r].pad = 0;
    }
    for (int k = 0; k < KV; ++k)
        for (int l = 0; l < pool->num_layers; ++l)
            pools[k * pool->num_layers + l] =
                static_cast<char *>((k == 0 ? pool->k_pages : pool->v_pages)[l]);

    Plan p;
    p.chunks = reinterpret_cast<const DevChunk *>(dev_block + lay.off_chunks);
    p.item_begin = reinterpret_cast<const int64_t *>(dev_block + lay.off_item_begin);
    p.reqs = reinterpret_cast<const DevRequest *>(dev_block + lay.off_reqs);
    p.pools = reinterpret_cast<char *const *>(dev_block + lay.off_pools);
    p.status = nullptr;
    p.total_items = item;
    p.token_bytes = v;
    p.n_chunks = n_chunks;
    p.kv_factor = KV;
    p.page_size = P;
    p.num_pages = pool->num_pages;
    p.num_layers = pool->num_layers;
    p.dir = dir;
    p.batch = default_batch(P, v);
    p.split = 1;
    return p;
}

// Round-trip units.  A load unit waits for its own store unit, and the grid's warps hold
// one unit each at the start (stores only) and at the end (loads only), so smaller units
// shorten that one-way fill and drain; but every unit also pays its hand-out, completion
// and wait, which only enough warps hide.  Measured on the MLA latent (1152-byte tokens,
// GB/s of both directions, 1.15 GB each way):
//  - 1, 2 and 4 tokens per page: 340.3-340.7 in units of about kRoundTripUnitBytes on 32
//    SMs, against 332.2-336.9 in 32 KiB units on 16 SMs; 8 KiB units on 16 SMs lose
//    (285-330), so fewer SMs keep 32 KiB units;
//  - 8 tokens per page (9 KiB segments, one per unit): 340.9 on 32 SMs in two runs, 333.2
//    and 341.9 on 16;
//  - 16 tokens and more (18 KiB segments and longer): 16 SMs is best (340.7 against 338.5);
//  - segments longer than kRoundTripMaxUnitBytes travel as row slices of at most that size
//    (72 KiB segments: 340.0 in three slices, 330.7-334.7 whole).
// Hence, with no configuration given, kRoundTripShortSms SMs for page segments shorter than
// kRoundTripShortSegment.
constexpr int64_t kRoundTripUnitBytes = 8192;
constexpr int64_t kRoundTripShortSegment = 16384;
constexpr int32_t kRoundTripShortSms = 32;
constexpr int64_t kRoundTripMaxUnitBytes = 32768;

RoundTripRule roundtrip_rule(int32_t page_size, int64_t token_bytes, bool user_cfg,
                             int32_t sm_cap, int32_t batch, int num_sms)
{
    RoundTripRule r{1, 1, sm_cap};
    if (page_size <= 0 || token_bytes <= 0)
        return r;
    const int64_t seg = token_bytes < kRoundTripMaxUnitBytes * 64
                            ? int64_t(page_size) * token_bytes
                            : kRoundTripMaxUnitBytes * 64;  // long enough for any rule
    if (!user_cfg && seg < kRoundTripShortSegment)
        r.sm_cap = kRoundTripShortSms;
    const int sms = r.sm_cap > 0 ? r.sm_cap : num_sms;
    if (batch > 0) {
        r.batch = batch;
    } else if (seg >= kRoundTripUnitBytes) {
        r.batch = 1;
        const int64_t k = (seg + kRoundTripMaxUnitBytes - 1) / kRoundTripMaxUnitBytes;
        r.slices = int32_t(std::min<int64_t>(std::max<int64_t>(k, 1), page_size));
    } else if (sms >= kRoundTripShortSms) {
        r.batch = int32_t(std::min<int64_t>((kRoundTripUnitBytes + seg - 1) / seg, 32));
    } else {
        r.batch = default_batch(page_size, token_bytes);
    }
    return r;
}


}  // namespace kvx

extern "C" {

kvx_status kvx_validate(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                        const kvx_chunk *chunks, int n_chunks, int layer_begin, int layer_end,
                        int op, int level, char *msg, size_t msg_len)
{
    int n_dev = 0;
    bool have_gpu = cudaGetDeviceCount(&n_dev) == cudaSuccess && n_dev > 0;
    if (!have_gpu)
        cudaGetLastError();
    return kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, op, level,
                         have_gpu, msg, msg_len);
}

kvx_status kvx_plan_count(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                          const kvx_chunk *chunks, int n_chunks, int layer_begin, int layer_end,
                          int64_t *n_segments, int64_t *n_bytes)
{
    kvx_status st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                                  KVX_OP_STORE, 0, false, nullptr, 0);
    if (st != KVX_OK)
        return st;
    int64_t segs = 0, bytes = 0;
    for (int c = 0; c < n_chunks; ++c) {
        int lo, hi;
        kvx::chunk_layers(chunks[c], layer_begin, layer_end, &lo, &hi);
        if (lo >= hi || chunks[c].n_tokens == 0)
            continue;
        int64_t np = (chunks[c].token_begin + chunks[c].n_tokens - 1) / pool->page_size -
                     chunks[c].token_begin / pool->page_size + 1;
        segs += (int64_t)(hi - lo) * pool->kv_factor * np;
        bytes += (int64_t)(hi - lo) * pool->kv_factor * chunks[c].n_tokens * pool->token_bytes;
    }
    if (n_segments)
        *n_segments = segs;
    if (n_bytes)
        *n_bytes = bytes;
    return KVX_OK;
}

// Default chunk size of the policy (bytes).  Chosen from the page/chunk-size sweep of the
// MLA-shaped workload: see kvx_chunk_policy.
static const int64_t kDefaultChunkBytes = 2ll << 20;

kvx_status kvx_chunk_policy(const kvx_pool *pool, int layer_streaming, int64_t target_bytes,
                            int32_t *tokens_per_chunk, int32_t *layers_per_chunk)
{
    if (!pool || !tokens_per_chunk || !layers_per_chunk || pool->num_layers <= 0 ||
        pool->page_size <= 0 || pool->token_bytes <= 0 ||
        (pool->kv_factor != 1 && pool->kv_factor != 2) || target_bytes < 0)
        return KVX_ERR_INVALID_ARG;
    int64_t target = target_bytes > 0 ? target_bytes : kDefaultChunkBytes;
    int32_t layers = layer_streaming ? 1 : pool->num_layers;
    int64_t page_bytes = (int64_t)layers * pool->kv_factor * pool->page_size * pool->token_bytes;
    int64_t pages = target / page_bytes;
    if (pages < 1)
        pages = 1;
    if (pages * pool->page_size > INT32_MAX)
        pages = INT32_MAX / pool->page_size;
    *tokens_per_chunk = (int32_t)(pages * pool->page_size);
    *layers_per_chunk = layers;
    return KVX_OK;
}

kvx_status kvx_default_link_model(kvx_link_model *m)
{
    if (!m)
        return KVX_ERR_INVALID_ARG;
    // GB300 with a Grace host over NVLink-C2C, as measured by the benchmark: pinned copies
    // 211.6 GB/s H2D and 193.7 GB/s D2H, 343.1 GB/s both at once; copy peak 6791.7 GB/s;
    // one SM with 128 KiB of
    // host reads in flight sustains ~50 GB/s (2.6 us round trip); ~10 us per call.
    m->h2d_gbs = 211.6;
    m->d2h_gbs = 193.7;
    m->hbm_gbs = 6791.7;
    m->bidir_gbs = 343.1;
    m->latency_us = 2.6;
    m->launch_us = 10.0;
    m->num_sms = 152;
    m->reserved = 0;
    return KVX_OK;
}

kvx_status kvx_estimate_us(const kvx_link_model *m, int op, int64_t bytes,
                           const kvx_launch_cfg *cfg, double *us)
{
    if (!m || !us || bytes < 0 || op < KVX_OP_STORE || op > KVX_OP_SCATTER_HBM ||
        m->latency_us <= 0 || m->num_sms <= 0)
        return KVX_ERR_INVALID_ARG;
    // The operation's defaults when no configuration is given (kept in step with the
    // library's kvx_default_launch_cfg).
    int sm_cap = op == KVX_OP_STORE ? 8 : (op == KVX_OP_LOAD ? 16 : 0);
    int ctas = op <= KVX_OP_LOAD ? 1 : 2;
    int threads = op <= KVX_OP_LOAD ? 1024 : 256, unroll = op <= KVX_OP_LOAD ? 8 : 4;
    bool bulk = false;
    double stage_bytes = 32768.0;
    if (cfg) {
        sm_cap = cfg->sm_cap;
        if (cfg->ctas_per_sm)
            ctas = cfg->ctas_per_sm;
        bulk = cfg->mapping == KVX_MAP_BULK;
        if (bulk) {
            unroll = cfg->unroll ? cfg->unroll : 3;
            if (cfg->stage_bytes)
                stage_bytes = cfg->stage_bytes;
        } else {
            if (cfg->threads)
                threads = cfg->threads;
            if (cfg->unroll)
                unroll = cfg->unroll;
        }
    }
    const double sms = sm_cap > 0 && sm_cap < m->num_sms ? sm_cap : m->num_sms;
    // Bytes in flight per CTA: threads x unroll 16-byte units (registers), or for the bulk
    // mapping its two rings' loading stages, 2 x (stages - 1) x stage_bytes.
    const double per_cta =
        bulk ? 2.0 * (unroll - 1) * stage_bytes : threads * (double)unroll * 16.0;
    const double in_flight = sms * ctas * per_cta;  // bytes
    const double little_gbs = in_flight / (m->latency_us * 1e3);           // B/ns = GB/s
    double peak;
    double moved = (double)bytes;
    if (op == KVX_OP_STORE)
        peak = m->d2h_gbs;
    else if (op == KVX_OP_LOAD)
        peak = m->h2d_gbs;
    else {
        peak = m->hbm_gbs;
        moved = 2.0 * bytes;  // read + write in HBM
    }
    const double gbs = op <= KVX_OP_LOAD ? (little_gbs < peak ? little_gbs : peak) : peak;
    *us = m->launch_us + (gbs > 0 ? moved / (gbs * 1e3) : 0.0);
    return KVX_OK;
}


kvx_status kvx_roundtrip_unit(int32_t page_size, int64_t token_bytes, const kvx_launch_cfg *cfg,
                              int32_t num_sms, int64_t *unit_bytes, int32_t *sm_cap)
{
    if (page_size <= 0 || token_bytes <= 0 || num_sms <= 0 || (cfg && cfg->sm_cap < 0) ||
        (cfg && (cfg->batch < 0 || cfg->batch > 32)))
        return KVX_ERR_INVALID_ARG;
    const kvx::RoundTripRule r = kvx::roundtrip_rule(page_size, token_bytes, cfg != nullptr,
                                                     cfg ? cfg->sm_cap : 16,
                                                     cfg ? cfg->batch : 0, num_sms);
    if (unit_bytes)
        *unit_bytes = r.slices > 1
                          ? (int64_t(page_size) + r.slices - 1) / r.slices * token_bytes
                          : int64_t(r.batch) * page_size * token_bytes;
    if (sm_cap)
        *sm_cap = r.sm_cap;
    return KVX_OK;
}

kvx_status kvx_estimate_pair_us(const kvx_link_model *m, int op, int64_t store_bytes,
                                int64_t load_bytes, int64_t unit_bytes,
                                const kvx_launch_cfg *cfg, double *us)
{
    if (!m || !us || store_bytes < 0 || load_bytes < 0 || unit_bytes < 0 ||
        (op != KVX_OP_EXCHANGE && op != KVX_OP_ROUNDTRIP) || m->latency_us <= 0 ||
        m->num_sms <= 0 || m->h2d_gbs <= 0 || m->d2h_gbs <= 0 || m->bidir_gbs <= 0 ||
        (op == KVX_OP_ROUNDTRIP && store_bytes != load_bytes))
        return KVX_ERR_INVALID_ARG;
    // Defaults in step with kvx_default_launch_cfg: exchange 40 SMs, round trip 16, both one
    // CTA of 1024 threads per SM with 8 loads in flight per lane.
    int sm_cap = op == KVX_OP_EXCHANGE ? 40 : 16, ctas = 1, threads = 1024, unroll = 8;
    if (cfg) {
        sm_cap = cfg->sm_cap;
        if (cfg->ctas_per_sm)
            ctas = cfg->ctas_per_sm;
        if (cfg->threads)
            threads = cfg->threads;
        if (cfg->unroll)
            unroll = cfg->unroll;
    }
    const double sms = sm_cap > 0 && sm_cap < m->num_sms ? sm_cap : m->num_sms;
    const double in_flight = sms * ctas * threads * (double)unroll * 16.0;
    const double little_gbs = in_flight / (m->latency_us * 1e3);
    const double both = little_gbs < m->bidir_gbs ? little_gbs : m->bidir_gbs;
    const double S = (double)store_bytes, Lb = (double)load_bytes;
    double t_ns;
    if (op == KVX_OP_EXCHANGE) {
        t_ns = S / m->d2h_gbs;
        if (Lb / m->h2d_gbs > t_ns)
            t_ns = Lb / m->h2d_gbs;
        if ((S + Lb) / both > t_ns)
            t_ns = (S + Lb) / both;
    } else {
        const double warps = sms * ctas * (threads / 32);
        double F = warps * (double)unit_bytes;
        if (F > S)
            F = S;
        t_ns = F / m->d2h_gbs + (2.0 * S - 2.0 * F) / both + F / m->h2d_gbs;
    }
    *us = m->launch_us + t_ns * 1e-3;
    return KVX_OK;
}

kvx_status kvx_estimate_stream_us(double io_us, double compute_us, int n_layers,
                                  double *e2e_us, double *bubble_us)
{
    if (n_layers <= 0 || io_us < 0 || compute_us < 0)
        return KVX_ERR_INVALID_ARG;
    const double step = io_us > compute_us ? io_us : compute_us;
    if (e2e_us)
        *e2e_us = io_us + (n_layers - 1) * step + compute_us;
    if (bubble_us)
        *bubble_us = io_us + (n_layers - 1) * (io_us > compute_us ? io_us - compute_us : 0.0);
    return KVX_OK;
}

const char *kvx_status_string(kvx_status s)
{
    switch (s) {
    case KVX_OK: return "ok";
    case KVX_ERR_INVALID_ARG: return "invalid argument";
    case KVX_ERR_ALIGNMENT: return "misaligned pointer or size";
    case KVX_ERR_NOT_DEVICE_ACCESSIBLE: return "memory not accessible by the device";
    case KVX_ERR_PAGE_OUT_OF_RANGE: return "page id out of range";
    case KVX_ERR_OVERLAP: return "overlapping load destinations";
    case KVX_ERR_CUDA: return "CUDA error";
    case KVX_ERR_DEVICE_STATUS: return "device reported an error";
    case KVX_ERR_CAPACITY: return "descriptor buffer too small";
    }
    return "unknown status";
}

int kvx_version(void) { return KVX_VERSION; }

}  // extern "C"
