/*
 * kvx.h -- C ABI of the GB300 paged KV-cache gather/scatter library (libkvx.so).
 *
 * The operation.  A serving engine keeps a request's KV cache in small fixed pages
 * (16-64 tokens) scattered through per-layer K and V pools in HBM and found through a
 * page table.  To move that cache to and from host memory in large contiguous chunks,
 * GPU threads gather the pages into chunk layout (store) or scatter chunks back into
 * freshly allocated pages (load), changing the layout on the fly, instead of issuing one
 * DMA per small page.  Sources:
 *   - "Strata Guide: Hierarchical Context Caching for Long LLMs", sections "The
 *     Conflict Between PagedAttention and Transfer Efficiency" (pages and page tables,
 *     per-page DMA cost), "The Mechanics of GPU-Assisted I/O", "Non-Intrusive Resource
 *     Sizing" (a small, capped SM count; cache-bypass stores), "Two-Dimensional Memory
 *     Layout Decoupling" (layer-first GPU layout, page-first host layout) and "Step 1:
 *     High-Performance GPU-Assisted I/O CUDA Kernel" (page-table lookup per unit);
 *   - "Tutti: Making SSD-Backed KV Cache Practical for Long-Context LLM Serving",
 *     section 2 Design 1 (host work O(layers), not O(layers x blocks)) and section 7
 *     (per-layer retrieve/store interface taking block ids).
 *
 * Layouts.
 *   Page pools (device memory): for each kv in [0, kv_factor) and layer in [0, num_layers)
 *   one array [num_pages][page_size][token_bytes].  kv 0 is K, kv 1 is V; an MLA latent
 *   cache uses kv_factor 1.  Token t of request r sits in slot
 *   page_table_r[t / page_size] * page_size + t % page_size of every pool.
 *   Chunks hold tokens [token_begin, token_begin + n_tokens) of one request for layers
 *   [layer_begin, layer_begin + n_layers):
 *     KVX_CHUNK_LAYER_MAJOR  [layer][kv][token][token_bytes]  (page-first, generalised to
 *                            a multi-page chunk)
 *     KVX_CHUNK_TOKEN_MAJOR  [token][layer][kv][token_bytes]
 *     KVX_CHUNK_STRIPED      [layer][kv] objects of [token][token_bytes], each starting at
 *                            a multiple of KVX_STRIPE_ALIGN from the chunk start
 *   A call moves only layers inside its window [layer_begin, layer_end) (half-open),
 *   intersected with each chunk's own layers; chunk offsets stay relative to the chunk's
 *   own layer_begin.
 *   In a TOKEN_MAJOR chunk of more than one (layer, kv) slab, a page of several tokens is
 *   a set of strided rows on the chunk side.  On their default grids stores and round
 *   trips move such pages at the rates of the other layouts, and loads and exchanges
 *   within 2-4 %; on a few SMs, loads from strided host rows run at about half the rate
 *   of contiguous ones.
 *
 * Ownership.  The caller owns the pools, page tables, chunk memory and streams.  A
 * kvx_ctx owns only a small ring of descriptor buffers (pinned host + device), a device
 * status word and a stream for descriptor copies.  Nothing on the transfer path
 * allocates; prepared plans allocate once, when created.
 *
 * Asynchrony and errors.  Every transfer call validates on the host, packs O(chunks)
 * descriptors, copies them to the device (on the context's copy stream, which the given
 * stream then waits for) and launches ONE kernel on the given stream, then returns.  A
 * host-detected error returns a non-zero kvx_status and launches nothing;
 * kvx_last_error() then holds a message.  Errors the kernel meets (a page id outside the
 * pool, a bounded wait that ran out) set a bit in the device status word and skip that
 * work, without trapping; kvx_get_status() reads and clears it.  A kvx_ctx must not be
 * used from two host threads at once.  Descriptor buffers are reused round-robin; before
 * reusing one the call waits for the kernel that last used it.
 */
#ifndef KVX_H
#define KVX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI version: bumped whenever a struct's layout changes (2: kvx_launch_cfg.overlap). */
#define KVX_VERSION 2

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *kvx_stream_t;

typedef enum kvx_status {
    KVX_OK = 0,
    KVX_ERR_INVALID_ARG = 1,            /* a size, index, range or pointer is invalid */
    KVX_ERR_ALIGNMENT = 2,              /* a pointer or token_bytes is not 16-byte aligned */
    KVX_ERR_NOT_DEVICE_ACCESSIBLE = 3,  /* chunk or pool memory the GPU cannot reach */
    KVX_ERR_PAGE_OUT_OF_RANGE = 4,      /* a page id outside [0, num_pages) */
    KVX_ERR_OVERLAP = 5,                /* two loads of one batch write the same page slot */
    KVX_ERR_CUDA = 6,                   /* a CUDA runtime call failed */
    KVX_ERR_DEVICE_STATUS = 7,          /* the kernel reported an error (see flags) */
    KVX_ERR_CAPACITY = 8                /* descriptors exceed the ctx's buffer size */
} kvx_status;

/* Bits of the device status word (kvx_get_status). */
#define KVX_DEV_PAGE_OUT_OF_RANGE 0x1u
#define KVX_DEV_WAIT_TIMEOUT 0x2u       /* a bulk copy, or the store a round-trip load
                                           waits for, did not complete within ~1 s; the
                                           kernel skipped work (output incomplete) */

typedef enum kvx_chunk_layout {
    KVX_CHUNK_LAYER_MAJOR = 0,
    KVX_CHUNK_TOKEN_MAJOR = 1,
    KVX_CHUNK_STRIPED = 2
} kvx_chunk_layout;

/* KVX_CHUNK_STRIPED: one object per (layer, kv), in [layer][kv] order, each holding the
 * chunk's tokens of that layer and kv back to back and each starting at a multiple of
 * KVX_STRIPE_ALIGN bytes from the chunk start (stride = object bytes rounded up to
 * KVX_STRIPE_ALIGN; the padding is never read or written).  A one-page chunk is the
 * per-block "GPU file" of 2L objects of "Tutti: Making SSD-Backed KV Cache Practical",
 * section 2 Design 1 and Figure 4, laid out for block-aligned (direct) storage I/O. */
#define KVX_STRIPE_ALIGN 4096

/* Direction of kvx_transform_hbm and kvx_dma_baseline. */
#define KVX_DIR_GATHER 0   /* pages -> chunks (a store) */
#define KVX_DIR_SCATTER 1  /* chunks -> pages (a load) */

typedef struct kvx_pool {
    int32_t num_layers;
    int32_t kv_factor;     /* 2: separate K and V pools; 1: one latent pool (MLA) */
    int32_t page_size;     /* tokens per page, > 0 */
    int32_t num_pages;     /* pages in each pool, > 0 */
    int64_t token_bytes;   /* one token's vector in one pool (heads x head_dim x dtype
                              bytes); a positive multiple of 16 up to 1 GiB, and a
                              page (page_size x token_bytes) at most 16 GiB */
    void *const *k_pages;  /* HOST array [num_layers] of device pointers: layer l's K pool
                              [num_pages][page_size][token_bytes], 16-byte aligned */
    void *const *v_pages;  /* same for V; ignored (may be NULL) when kv_factor == 1 */
} kvx_pool;

typedef struct kvx_request {
    const int32_t *page_table;       /* device-accessible [ceil(n_tokens / page_size)]
                                        physical page ids; read by the kernel */
    const int32_t *page_table_host;  /* optional host copy of the same table: enables the
                                        page-range and overlap checks of validation level 2;
                                        required by kvx_dma_baseline */
    int32_t n_tokens;                /* tokens in the request, >= 0 */
    int32_t reserved;                /* set to 0 */
} kvx_request;

typedef struct kvx_chunk {
    int32_t request;      /* index into the request array */
    int32_t token_begin;  /* first token, >= 0 */
    int32_t n_tokens;     /* tokens, token_begin + n_tokens <= request's n_tokens */
    int32_t layer_begin;  /* first layer held by the chunk */
    int32_t n_layers;     /* layers held, layer_begin + n_layers <= num_layers */
    int32_t layout;       /* kvx_chunk_layout */
    void *ptr;            /* chunk memory, 16-byte aligned, n_layers x kv_factor x n_tokens
                             x token_bytes bytes (STRIPED: n_layers x kv_factor x the
                             padded object stride): mapped pinned host memory for
                             store/load, device memory for kvx_transform_hbm */
} kvx_chunk;

/* Work mapping of the transfer kernel. */
#define KVX_MAP_WARP_SEGMENT 0  /* one warp per (chunk, layer, kv, page) segment; lanes move
                                   16-byte units through registers (32-byte units for an
                                   HBM transform on 32-byte-aligned memory) */
#define KVX_MAP_BULK 1          /* three warps per CTA: one resolves segments 32 at a
                                   time, and one lane of each of the other two streams
                                   alternate batches of them through its own ring of
                                   shared-memory stages with bulk async copies
                                   (cp.async.bulk, mbarrier completion); `unroll` is the
                                   number of stages per ring (2..8), `stage_bytes` their
                                   size.  Loads reach the host link's peak on the fewest
                                   SMs (4 on GB300) */
#define KVX_MAP_CTA 2           /* all threads of a CTA move one segment together (thread t
                                   takes units t, t + threads, ...), 32 segments resolved
                                   per batch by one warp; store, load and transform only */

/* Store cache hint for the destination of each 16-byte unit. */
#define KVX_HINT_DEFAULT 0      /* st.global (write-back) */
#define KVX_HINT_STREAMING 1    /* st.global.cs (evict-first, cache streaming) */

typedef struct kvx_launch_cfg {
    int32_t sm_cap;       /* CTAs launched = sm_cap x ctas_per_sm (fewer when the batch has
                             less work); with ctas_per_sm = 1 the kernel occupies at most
                             sm_cap SMs.  0 = every SM */
    int32_t ctas_per_sm;  /* 0 = the operation's default */
    int32_t threads;      /* threads per CTA, multiple of 32 in [32, 1024]; 0 = default
                             (the bulk mapping always runs three warps per CTA) */
    int32_t unroll;       /* warp-segment and CTA mappings: 16-byte loads in flight per
                             thread before its stores (1, 2, 4 or 8; where
                             kvx_transform_hbm moves 32-byte units, max(unroll / 2, 1)
                             32-byte loads; a single transfer whose chunks include a
                             token-major one of several (layer, kv) slabs walks its strided
                             rows min(unroll, 4) deep); bulk mapping: shared-memory stages
                             of each of its two rings (2..8).  0 = default (bulk: 3) */
    int32_t store_hint;   /* KVX_HINT_* (warp-segment and CTA mappings) */
    int32_t mapping;      /* KVX_MAP_* */
    int32_t stage_bytes;  /* bulk mapping: bytes per shared-memory stage, a multiple of 16;
                             2 x stages x stage_bytes <= 208 KiB.  0 = default (32 KiB) */
    int32_t batch;        /* warp-segment mapping: page segments a warp resolves at once,
                             one per lane (1..32); 0 = automatic (about 32 KiB of segments;
                             for page segments >= 16 KiB, 1 for host transfers and 2 for
                             the HBM transform; round trips: see kvx_roundtrip_chunks) */
    int32_t overlap;      /* 1: the launch may start while the previous kernel on its stream
                             is still running (programmatic dependent launch), so that its
                             ramp overlaps that kernel's drain; it still completes after that
                             kernel, so events recorded after it keep their meaning.  Use it
                             only when this transfer touches no memory the previous kernel
                             writes and writes none it reads (for example consecutive
                             per-layer loads).  A call made with it waits on the host for
                             its descriptor copy (a few microseconds) before it enqueues the
                             kernel.  Store, load and transform with the warp-segment
                             mapping; 0 elsewhere.  0 = off (default) */
} kvx_launch_cfg;

typedef struct kvx_ctx kvx_ctx;

/* Operation ids (kvx_default_launch_cfg, kvx_validate). */
#define KVX_OP_STORE 0        /* pages -> chunks in mapped pinned host memory */
#define KVX_OP_LOAD 1         /* chunks in mapped pinned host memory -> pages */
#define KVX_OP_GATHER_HBM 2   /* pages -> chunks in device memory */
#define KVX_OP_SCATTER_HBM 3  /* chunks in device memory -> pages */
#define KVX_OP_EXCHANGE 4     /* a store batch and a load batch in one launch (defaults only) */
#define KVX_OP_ROUNDTRIP 5    /* store to chunks, then load them elsewhere, in one launch
                                 (defaults only) */

/* ---------------------------------------------------------------- context */

/* Create a context on `device` whose descriptor buffers hold up to
 * max_descriptor_bytes each (0 = 8 MiB; 64 bytes per chunk, 16 per request, 8 per pool
 * layer).  Allocates four
 * pinned host + device descriptor buffers, a device status word and a non-blocking stream
 * on which each call copies its descriptors (the caller's stream waits for that copy with
 * an event, so the copy overlaps the previous kernel).  Calls therefore cannot be captured
 * into a CUDA graph; prepared plans (below) can.  Requires a GPU.
 *
 * Threads: a context is not thread-safe.  Its descriptor ring, last-launch record and
 * error text belong to whichever call is running, so calls on one context must not
 * overlap in time; give each host thread its own context.  Streams are independent of
 * this: one thread may issue calls on any number of streams.  kvx_plan_launch touches its
 * context only to report an error, and kvx_load_chunks_noalloc uses no context (it
 * serialises its own calls). */
kvx_status kvx_create(kvx_ctx **out, int device, size_t max_descriptor_bytes);

/* Synchronize with every kernel the context launched, then free its buffers. */
void kvx_destroy(kvx_ctx *ctx);

/* 0: no validation.  1 (default): O(chunks) arithmetic checks of every size, range and
 * alignment.  2: also page ids and load-destination overlap against page_table_host
 * (O(tokens)) and cudaPointerGetAttributes on every chunk and pool pointer. */
kvx_status kvx_set_validation(kvx_ctx *ctx, int level);

/* Default launch configuration of an operation (KVX_OP_*) on this context's GPU. */
kvx_status kvx_default_launch_cfg(const kvx_ctx *ctx, int op, kvx_launch_cfg *cfg);

/* ---------------------------------------------------------------- transfers */

/* store: gather every covered (layer, kv, token) vector from the page pools into the
 * chunks ("Strata Guide", section "Non-Intrusive Resource Sizing": eviction to host
 * memory; "Tutti", section 7: store_layer(layer_id, block_ids)).  Chunks live in mapped
 * pinned host memory.  cfg may be NULL: the defaults of kvx_default_launch_cfg (8 SMs,
 * which carry the device-to-host peak on GB300), except that page segments
 * (page_size x token_bytes) shorter than 4 KiB get 32 SMs, since a warp then moves one
 * short segment per pass.  Asynchronous on `stream`.
 * A store issued beside a load that needs the whole host-to-device peak (a prefetch on
 * another stream) takes link bandwidth from it in proportion to its SMs (on GB300 about
 * 10 GB/s per SM while the other direction is saturated), which is why the default grid
 * stays at 8 SMs; where two kernels land on the GPU still varies from run to run.  Batches
 * that can be issued together are best issued with kvx_exchange_chunks, which shares one
 * grid between them. */
kvx_status kvx_store_chunks(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *reqs,
                            int n_req, const kvx_chunk *chunks, int n_chunks,
                            int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                            kvx_stream_t stream);

/* load: scatter chunks from mapped pinned host memory into the pages named by the page
 * tables ("Strata Guide", section "Step 1: High-Performance GPU-Assisted I/O CUDA
 * Kernel"; "Tutti", section 7: retrieve_layer(layer_id, block_ids)).  Destination slots
 * must be disjoint across the batch (checked at validation level 2).  Slots of a page
 * past the request's last token are not written.  cfg = NULL: as for kvx_store_chunks. */
kvx_status kvx_load_chunks(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *reqs,
                           int n_req, const kvx_chunk *chunks, int n_chunks,
                           int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                           kvx_stream_t stream);

/* exchange: a store batch and a load batch moved by ONE kernel launch, so both
 * directions of the host link carry data at once (an eviction
 * and a prefetch issued together: "Strata Guide", section "Implementation: GPU-Assisted
 * I/O Kernels and Bubble-Filling Scheduler", steps "Dispatch Asynchronous Transfer" and
 * "Asynchronous Eviction").  Each batch follows the rules of kvx_store_chunks /
 * kvx_load_chunks; either may be empty.  The store's source slots and the load's
 * destination slots must not meet for a common layer (checked at validation level 2).
 * cfg->sm_cap counts the SMs of both directions together (default 40).  Batches of
 * similar size (within 1.5x in segments) of page segments of 4 KiB or more split the CTAs
 * by direction, half each; otherwise every warp takes units of both batches, so the larger
 * one keeps the whole grid after the smaller one is done, and short segments of both
 * directions are in flight in every warp.  Either way, nothing in the launch waits on
 * anything else. */
kvx_status kvx_exchange_chunks(kvx_ctx *ctx, const kvx_pool *pool,
                               const kvx_request *store_reqs, int n_store_req,
                               const kvx_chunk *store_chunks, int n_store_chunks,
                               const kvx_request *load_reqs, int n_load_req,
                               const kvx_chunk *load_chunks, int n_load_chunks,
                               int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                               kvx_stream_t stream);

/* round trip: store the pages of src_reqs into the chunks and load the chunks into the
 * pages of dst_reqs, in ONE launch: a swap-out to host memory followed by a swap-in to
 * another page set (a preempted request resumed on new pages).  The pages describe the
 * two transfers ("Strata Guide", section "Implementation: GPU-Assisted I/O Kernels and
 * Bubble-Filling Scheduler": asynchronous eviction and transfer dispatch) but no call
 * that orders one after the other inside a launch; this one does so per unit of work:
 * each (chunk, layer, kv, page) segment is loaded once its own store has reached host
 * memory, so both link directions carry data from the first finished store to the last
 * load, with no launch boundary in between.  Chunk c belongs to request
 * chunks[c].request of BOTH arrays (n_req entries each); the two page sets must not
 * share a slot for a common layer (checked at validation level 2), and each batch
 * follows the rules of kvx_store_chunks / kvx_load_chunks.  Its waits are bounded: a
 * unit whose store has not finished within about a second is skipped and
 * KVX_DEV_WAIT_TIMEOUT is set.  The descriptor buffer holds both plans plus 4 bytes per
 * unit (a unit is `batch` segments; by default one segment when page segments are 8 KiB
 * or longer, else about 8 KiB of segments on 32 SMs or more and about 32 KiB on fewer).
 * cfg->sm_cap counts all SMs (default 16; with cfg = NULL and page segments shorter than
 * 16 KiB, 32, because a warp then has at most one short segment in flight). */
kvx_status kvx_roundtrip_chunks(kvx_ctx *ctx, const kvx_pool *pool,
                                const kvx_request *src_reqs, const kvx_request *dst_reqs,
                                int n_req, const kvx_chunk *chunks, int n_chunks,
                                int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                                kvx_stream_t stream);

/* transform: the same gather (dir = KVX_DIR_GATHER) or scatter (KVX_DIR_SCATTER) with
 * the chunks in device memory: the explicit HBM-to-HBM layout pass that "Strata Guide",
 * section "Two-Dimensional Memory Layout Decoupling", names as the conventional cost.
 * With the warp-segment mapping, when token_bytes, every pool layer and every chunk pointer
 * are multiples of 32 bytes, lanes move 32-byte units (max(unroll / 2, 1) loads in
 * flight); otherwise 16-byte units.  The result is the same either way. */
kvx_status kvx_transform_hbm(kvx_ctx *ctx, int dir, const kvx_pool *pool,
                             const kvx_request *reqs, int n_req, const kvx_chunk *chunks,
                             int n_chunks, int layer_begin, int layer_end,
                             const kvx_launch_cfg *cfg, kvx_stream_t stream);

/* ---------------------------------------------------------------- prepared plans */

/* A store, load or transform (op = KVX_OP_STORE .. KVX_OP_SCATTER_HBM) validated and
 * packed once (cfg as for the call it prepares).  kvx_plan_create allocates device memory of its own for the descriptors,
 * copies them there on `stream` and waits for the copy.  kvx_plan_launch then only
 * enqueues the kernel: no validation, no host packing, no descriptor copy, no slot wait,
 * so repeated transfers (the same per-layer batches every prefill, for instance) cost one
 * launch each, and a sequence of launches can be captured into a CUDA graph.  The plan
 * keeps the addresses of the pools, page tables and chunks it was made with: their
 * contents may change between launches, their addresses may not.  Launches report to the
 * context's status word; destroy a plan (it synchronizes the device) before its context. */
typedef struct kvx_plan kvx_plan;

kvx_status kvx_plan_create(kvx_ctx *ctx, int op, const kvx_pool *pool, const kvx_request *reqs,
                           int n_req, const kvx_chunk *chunks, int n_chunks, int layer_begin,
                           int layer_end, const kvx_launch_cfg *cfg, kvx_stream_t stream,
                           kvx_plan **out);
/* The exchange of kvx_exchange_chunks (a store batch and a load batch in one launch),
 * validated and packed once; launched with kvx_plan_launch like any plan.  Same rules on
 * what may change between launches. */
kvx_status kvx_plan_create_exchange(kvx_ctx *ctx, const kvx_pool *pool,
                                    const kvx_request *store_reqs, int n_store_req,
                                    const kvx_chunk *store_chunks, int n_store_chunks,
                                    const kvx_request *load_reqs, int n_load_req,
                                    const kvx_chunk *load_chunks, int n_load_chunks,
                                    int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                                    kvx_stream_t stream, kvx_plan **out);
/* The round trip of kvx_roundtrip_chunks, validated and packed once.  Each launch first
 * zeroes the plan's work counters and completion words (a memset on `stream`, captured
 * with the kernel in a CUDA graph), so launches of one such plan must not overlap in time;
 * the same holds for an exchange plan whose batches differ by more than 1.5x. */
kvx_status kvx_plan_create_roundtrip(kvx_ctx *ctx, const kvx_pool *pool,
                                     const kvx_request *src_reqs, const kvx_request *dst_reqs,
                                     int n_req, const kvx_chunk *chunks, int n_chunks,
                                     int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                                     kvx_stream_t stream, kvx_plan **out);
kvx_status kvx_plan_launch(const kvx_plan *plan, kvx_stream_t stream);
void kvx_plan_destroy(kvx_plan *plan);

/* Comparison baseline only: the same transfer as one cudaMemcpyAsync per contiguous
 * (chunk, layer, kv, page) segment (cudaMemcpy2DAsync for token-major chunks), issued
 * from this host thread ("Strata Guide", section "The Conflict Between PagedAttention
 * and Transfer Efficiency": one DMA per page and layer).  Needs page_table_host on every
 * request.  n_copies (may be NULL) receives the number of copies issued. */
kvx_status kvx_dma_baseline(kvx_ctx *ctx, int dir, const kvx_pool *pool,
                            const kvx_request *reqs, int n_req, const kvx_chunk *chunks,
                            int n_chunks, int layer_begin, int layer_end,
                            kvx_stream_t stream, int64_t *n_copies);

/* Read the device status word (after synchronizing `stream`), clear it, and return
 * KVX_ERR_DEVICE_STATUS if any bit was set.  flags may be NULL. */
kvx_status kvx_get_status(kvx_ctx *ctx, kvx_stream_t stream, uint32_t *flags);

/* Message describing the last error of this context ("" if none). */
const char *kvx_last_error(const kvx_ctx *ctx);

/* Shape of the context's last kernel launch by a call (not by a plan): work items (page
 * segments; an exchange or round trip counts both directions), CTAs, threads per CTA and
 * bytes of descriptors copied to the device; zeros if the last call launched nothing.
 * Any output may be NULL. */
kvx_status kvx_last_launch(const kvx_ctx *ctx, int64_t *items, int32_t *ctas,
                           int32_t *threads, int64_t *descriptor_bytes);

/* ---------------------------------------------------------------- allocation-free load */

/* Size of the fixed scratch array behind kvx_load_chunks_noalloc: a 256-byte status
 * header plus the packed descriptors (64 bytes per chunk, 16 per request, 8 per pool
 * layer, each group padded to 128 bytes), so about 16,000 chunks per call. */
#define KVX_NOALLOC_SCRATCH_BYTES (1u << 20)

/* kvx_load_chunks without a context and without allocating anything.  The pages have no
 * counterpart of this call: it exists for callers that may not allocate device memory,
 * such as a serving engine that has handed nearly all of HBM to its KV page pool at
 * start-up (a later cudaMalloc fails or takes memory the pool was promised), or a plug-in
 * the engine calls without a place to keep a kvx_ctx between calls.
 *
 * Scratch: the descriptors and the status word live in one file-scope device array of
 * KVX_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds until the
 * process exits.  A batch whose descriptors do not fit returns KVX_ERR_CAPACITY and
 * launches nothing.  The call calls no cudaMalloc or cudaFree and allocates no host
 * memory.
 *
 * Runs on the calling thread's current device.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current.  Each call
 * copies its descriptors into the array (from a static host image; the copy call returns
 * once it has read it), which also clears the status word, then launches the load kernel
 * on `stream` with the launch shape kvx_load_chunks would use for the same cfg.  A stream
 * that is capturing is refused with KVX_ERR_INVALID_ARG before anything is done: a
 * captured copy would read the host image again at replay, when it holds another call's
 * descriptors.  All calls share the one array and it keeps the last call's contents:
 * calls whose work overlaps on the GPU (for example on two streams without ordering
 * between them) race on it.  Issue them on one stream, or order them with events.
 *
 * Arguments are those of kvx_load_chunks (validation level 1 always; the warp-segment
 * mapping only, without overlap).  device_flags, if not NULL, is a 4-byte aligned
 * device-accessible word that the kernel ORs KVX_DEV_* bits into (the caller clears it);
 * when NULL they go to the array's status word, which the next call clears, so they are
 * dropped. */
kvx_status kvx_load_chunks_noalloc(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                                   const kvx_chunk *chunks, int n_chunks, int layer_begin,
                                   int layer_end, const kvx_launch_cfg *cfg,
                                   kvx_stream_t stream, uint32_t *device_flags);

/* ---------------------------------------------------------------- host logic (no GPU) */

/* Validate a transfer of kind `op` (KVX_OP_*) at `level` (1 or 2; level 2's pointer
 * checks need a GPU and are skipped when none is present).  On failure a message is
 * written to msg (if msg_len > 0). */
kvx_status kvx_validate(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                        const kvx_chunk *chunks, int n_chunks, int layer_begin,
                        int layer_end, int op, int level, char *msg, size_t msg_len);

/* Count the page segments of a transfer -- one per (chunk, covered layer, kv, page the
 * chunk touches); each is one copy of the DMA baseline (a 2D copy for a token-major
 * chunk) and one work item of the kernel -- and its payload bytes (one direction).
 * Either output may be NULL. */
kvx_status kvx_plan_count(const kvx_pool *pool, const kvx_request *reqs, int n_req,
                          const kvx_chunk *chunks, int n_chunks, int layer_begin,
                          int layer_end, int64_t *n_segments, int64_t *n_bytes);

/* Chunk-size policy: tokens and layers per chunk for a request's KV ("Strata Guide",
 * section "The Physics of I/O Bandwidth and Little's Law": transfers of 1-4 MB are what
 * saturate a host link, where one page per layer is kilobytes).  layer_streaming != 0
 * asks for per-layer chunks (one layer per chunk, for transfers issued layer by layer);
 * otherwise chunks hold all layers (page-first).  target_bytes is the wanted chunk size,
 * for instance a storage tier's preferred I/O size; 0 = the library default, 2 MiB.
 * tokens_per_chunk is the largest positive multiple of page_size whose chunk fits
 * target_bytes (one page when even that does not), so no chunk boundary splits a page. */
kvx_status kvx_chunk_policy(const kvx_pool *pool, int layer_streaming, int64_t target_bytes,
                            int32_t *tokens_per_chunk, int32_t *layers_per_chunk);

/* ---------------------------------------------------------------- SM partitioning */

/* Hard split of one GPU's SMs into io_groups I/O partitions and one compute partition,
 * each a green context with one non-blocking stream ("Tutti: Making SSD-Backed KV Cache
 * Practical", section 2 Design 2: SM partitioning into a compute domain and an I/O domain
 * with green contexts).  Transfers launched on an I/O stream run only on that partition's
 * SMs; work launched on the compute stream (wrap it with torch.cuda.ExternalStream, for
 * instance) runs only on the rest, so neither waits for the other's SMs.  Two I/O
 * partitions give a store and a load that run at once fixed, disjoint SM sets.  io_sms is
 * a minimum per I/O partition: the driver rounds it up to its partition granularity (8 SMs
 * on this GPU).  Priorities follow CUDA's convention (lower = higher; 0 = default).  On
 * failure msg (if msg_len > 0) holds the failing driver step.  Requires a GPU and a driver
 * with green-context support. */
typedef struct kvx_partition kvx_partition;

kvx_status kvx_partition_create(int device, int io_groups, int io_sms, int io_priority,
                                int compute_priority, kvx_partition **out, char *msg,
                                size_t msg_len);

/* Stream and SM count of partition `group`: 0 .. io_groups-1 are the I/O partitions,
 * io_groups is the compute partition.  Either output may be NULL. */
kvx_status kvx_partition_info(const kvx_partition *partition, int group, kvx_stream_t *stream,
                              int *sms);

/* Synchronize the device, then destroy the streams and green contexts. */
void kvx_partition_destroy(kvx_partition *partition);

/* ---------------------------------------------------------------- I/O-time estimator */

/* A measured description of one GPU's data paths, for kvx_estimate_us.  Fill it from
 * measurements (bench.py prints them); kvx_default_link_model gives the GB300 + Grace
 * NVLink-C2C figures measured by this library's benchmark. */
typedef struct kvx_link_model {
    double h2d_gbs;      /* host -> device peak, GB/s (one 4 GiB pinned copy) */
    double d2h_gbs;      /* device -> host peak, GB/s */
    double hbm_gbs;      /* HBM copy peak, GB/s counting read + write */
    double bidir_gbs;    /* host link, both directions at once (H2D + D2H pinned copies on
                            two streams), GB/s counting both directions */
    double latency_us;   /* round trip of one host-memory access from an SM */
    double launch_us;    /* fixed cost of one call: host packing, descriptor copy, launch */
    int32_t num_sms;
    int32_t reserved;
} kvx_link_model;

kvx_status kvx_default_link_model(kvx_link_model *model);

/* Predicted duration (microseconds) of one store/load/transform call of the warp-segment
 * mapping moving `bytes` in each direction with launch configuration cfg (NULL = the
 * operation's defaults).  Little's law, as "Strata Guide: Hierarchical Context Caching for
 * Long LLMs", section "The Physics of I/O Bandwidth and Little's Law", states it
 * (X = C * S / L): each CTA keeps threads x unroll 16-byte units in flight (the bulk
 * mapping: 2 x (unroll - 1) x stage_bytes, the loading stages of its two rings), so the
 * CTAs sustain ctas x that / latency, capped by the link's peak in that direction; the HBM
 * transform is capped by the HBM peak (2 x bytes of traffic).
 * t = launch_us + bytes / min(peak, in_flight / latency). */
kvx_status kvx_estimate_us(const kvx_link_model *model, int op, int64_t bytes,
                           const kvx_launch_cfg *cfg, double *us);

/* Predicted duration (microseconds) of one exchange (op = KVX_OP_EXCHANGE) or round trip
 * (KVX_OP_ROUNDTRIP) moving store_bytes to the host and load_bytes to the device in one
 * launch with cfg (NULL = defaults).  Both directions share the link: each is capped by
 * its own peak, together they are capped by the bidirectional peak and by Little's law
 * on the launch's bytes in flight (as in kvx_estimate_us):
 *   t = launch_us + max(store / d2h, load / h2d, (store + load) / min(bidir, in_flight / L))
 * A round trip (store_bytes = load_bytes) first stores, and last loads, one unit of
 * unit_bytes per warp of its grid on its own at the one-way rates (its fill and drain;
 * kvx_roundtrip_unit gives the unit and SM cap kvx_roundtrip_chunks uses):
 *   t = launch_us + F / d2h + (2 x bytes - 2 F) / min(bidir, ...) + F / h2d,
 *   F = min(bytes, warps x unit_bytes). */
kvx_status kvx_estimate_pair_us(const kvx_link_model *model, int op, int64_t store_bytes,
                                int64_t load_bytes, int64_t unit_bytes,
                                const kvx_launch_cfg *cfg, double *us);

/* The unit and SM cap kvx_roundtrip_chunks uses for page segments of page_size tokens of
 * token_bytes each, on a device of num_sms SMs, with cfg (NULL = no configuration given):
 * unit_bytes = segments per unit x the segment, or the largest row slice when long segments
 * are cut.  Pass them to kvx_estimate_pair_us (unit_bytes, and sm_cap in its cfg).  Host
 * only; KVX_ERR_INVALID_ARG for non-positive sizes or an invalid SM cap or batch. */
kvx_status kvx_roundtrip_unit(int32_t page_size, int64_t token_bytes, const kvx_launch_cfg *cfg,
                              int32_t num_sms, int64_t *unit_bytes, int32_t *sm_cap);

/* Layer-streamed prefill: layer l + 1's KV is loaded while layer l computes (as "Strata
 * Guide", section "The Loading-Bound Scheduling Dilemma and Delay Hits", and the
 * step list "Layer-Overlapped Prefill" describe).  With per-layer load time io_us and
 * compute time compute_us, the predicted end-to-end time is
 *   io_us + (n_layers - 1) * max(io_us, compute_us) + compute_us
 * and the I/O bubble (time the compute stream waits) is n_layers' worth of
 * max(0, io_us - compute_us) after the first layer plus the first load itself. */
kvx_status kvx_estimate_stream_us(double io_us, double compute_us, int n_layers,
                                  double *e2e_us, double *bubble_us);

/* Pinned host memory, mapped into the device address space (allocate or register
 * once, up front, never on the transfer path). */
kvx_status kvx_host_alloc(void **ptr, size_t bytes);
kvx_status kvx_host_free(void *ptr);
kvx_status kvx_host_register(void *ptr, size_t bytes);
kvx_status kvx_host_unregister(void *ptr);

const char *kvx_status_string(kvx_status status);
int kvx_version(void);

/* ---------------------------------------------------------------- test support */

/* Makes the round trip's bounded wait run out, so that a test can check the timeout path
 * without faulting or hanging the GPU.  It launches the round trip of kvx_roundtrip_chunks
 * (same arguments and validation, all layers, default launch configuration) with every
 * store unit counted as handed out but none performed.  Each load unit's wait for its
 * store then ends after wait_ns nanoseconds (1 ms to 1 s; a transfer waits about 1 s).
 * The kernel sets KVX_DEV_WAIT_TIMEOUT in the context's device status word, skips that
 * load unit and returns; no page and no chunk is written.  The launch takes about
 * ceil(units / warps of the grid) x wait_ns.  Read the flag with kvx_get_status.  Not a
 * transfer: for tests of failure handling only. */
kvx_status kvx_test_roundtrip_timeout(kvx_ctx *ctx, const kvx_pool *pool,
                                      const kvx_request *src_reqs, const kvx_request *dst_reqs,
                                      int n_req, const kvx_chunk *chunks, int n_chunks,
                                      uint64_t wait_ns, kvx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVX_H */
