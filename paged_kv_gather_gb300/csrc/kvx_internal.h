// kvx_internal.h -- descriptor formats shared by the host packer and the transfer kernels.
//
// The host turns a batch into O(chunks) descriptors (never O(layers x pages)): the
// device resolves pages through the page tables itself, following "Tutti: Making
// SSD-Backed KV Cache Practical", section 2 Design 1 (host work drops from
// O(layer x blocks) to O(layer)).
//
// Work is cut into items.  One item is one (chunk, layer, kv, page touched by the chunk):
// a run of tokens that is contiguous in the page pool.  Items of chunk c are numbered
//   item = slab * np + j,   slab = (layer - la) * kv_factor + kv,   j = page - pf
// and chunk c owns items [item_begin[c], item_begin[c + 1]).
#pragma once

#include <stdint.h>

#include "../../include/kvx.h"

namespace kvx {

struct DevChunk {
    char *ptr;           // chunk base
    int64_t slab_stride; // bytes between consecutive (layer, kv) slabs of the chunk
    int64_t row_stride;  // bytes between consecutive tokens of one slab
    int32_t request;
    int32_t t0;          // first token
    int32_t t_end;       // one past the last token
    int32_t pf;          // first logical page touched
    int32_t np;          // logical pages touched
    int32_t la;          // first layer moved (absolute)
    int32_t slab0;       // (la - chunk layer_begin) * kv_factor: first slab moved
    int32_t pad;
};
static_assert(sizeof(DevChunk) == 56, "descriptor layout");

struct DevRequest {
    const int32_t *page_table;
    int32_t n_pages;
    int32_t pad;
};
static_assert(sizeof(DevRequest) == 16, "descriptor layout");

// Kernel parameter block (passed by value).
struct Plan {
    const DevChunk *chunks;
    const int64_t *item_begin;  // [n_chunks + 1]
    const DevRequest *reqs;
    char *const *pools;         // [kv_factor * num_layers], pools[kv * num_layers + layer]
    unsigned int *status;       // device status word
    int64_t total_items;
    int64_t token_bytes;
    int32_t n_chunks;
    int32_t kv_factor;
    int32_t page_size;
    int32_t num_pages;
    int32_t num_layers;
    int32_t dir;                // KVX_DIR_GATHER (pages -> chunks) or KVX_DIR_SCATTER
    int32_t batch;              // segments a warp resolves at once (1..32)
    int32_t split;              // row slices per segment, one per warp (kvx_split_kernel);
                                // 1 = whole segments
};

// Segments a warp resolves in parallel by default: enough short segments to put ~32 KiB
// in flight per warp (one segment when page segments are >= 16 KiB).
inline int32_t default_batch(int64_t page_size, int64_t token_bytes)
{
    int64_t seg = page_size * token_bytes;
    int64_t b = seg > 0 ? (32768 + seg - 1) / seg : 1;
    if (seg >= 16384)
        b = 1;
    return int32_t(b < 1 ? 1 : (b > 32 ? 32 : b));
}

// Byte layout of one packed descriptor block (host staging == device copy).
struct PackedLayout {
    size_t off_item_begin, off_chunks, off_reqs, off_pools, total;
};

// Host-side helpers (kvx_host.cpp).
kvx_status validate(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                    const kvx_chunk *chunks, int n_chunks, int layer_begin, int layer_end,
                    int op, int level, bool have_gpu, char *msg, size_t msg_len);

// An exchange (store batch + load batch in one launch): each batch validated as its own
// operation, and, at level 2, no page slot read by the store and written by the load for a
// common layer.
kvx_status validate_exchange(const kvx_pool *pool, const kvx_request *sreqs, int n_sreq,
                             const kvx_chunk *schunks, int n_schunks, const kvx_request *lreqs,
                             int n_lreq, const kvx_chunk *lchunks, int n_lchunks,
                             int layer_begin, int layer_end, int level, bool have_gpu,
                             char *msg, size_t msg_len);

PackedLayout packed_layout(const kvx_pool *pool, int n_req, int n_chunks);

// Fill `block` (host memory of at least layout.total bytes) with descriptors whose device
// pointers are relative to `dev_block`; returns the plan for the launch.
Plan pack(const kvx_pool *pool, const kvx_request *reqs, int n_req, const kvx_chunk *chunks,
          int n_chunks, int layer_begin, int layer_end, int dir, const PackedLayout &lay,
          char *block, char *dev_block);

// Effective layer range of a chunk inside a call window; empty when lo >= hi.
inline void chunk_layers(const kvx_chunk &c, int layer_begin, int layer_end, int *lo, int *hi)
{
    *lo = c.layer_begin > layer_begin ? c.layer_begin : layer_begin;
    int e = c.layer_begin + c.n_layers;
    *hi = e < layer_end ? e : layer_end;
}

}  // namespace kvx
