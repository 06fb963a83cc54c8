// kvx.cu -- C-ABI entry points of the paged KV gather/scatter library: contexts,
// descriptor staging, launch shapes, prepared plans, the per-page DMA baseline and the
// allocation-free load.  The kernels are in kvx_kernels.cuh; host-only validation and
// packing are in kvx_host.cpp.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <vector>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kvx_internal.h"
#include "kvx_kernels.cuh"
#include "kvx_rules.h"

// --------------------------------------------------------------------------------- host

namespace {

const int kSlots = 4;
const size_t kDefaultDescriptorBytes = 8u << 20;
const int kDefaultStageBytes = 32 << 10;
const int kDefaultStages = 3;  // per copy lane of the bulk mapping
const int64_t kShortSegmentBytes = 4096;  // store/load without a cfg: below this, 32 SMs
const int kShortSegmentSms = 32;
const int64_t kMaxBulkSmem = 208 << 10;  // the rings; the CTA's other shared state is ~14 KiB

struct Slot {
    char *host = nullptr;
    char *dev = nullptr;
    cudaEvent_t done = nullptr;    // recorded on the caller's stream after the kernel
    cudaEvent_t staged = nullptr;  // recorded on the copy stream after the descriptor copy
    bool used = false;
};

}  // namespace

struct kvx_ctx {
    int device = 0;
    int num_sms = 0;
    int validation = 1;
    size_t slot_bytes = 0;
    Slot slots[kSlots];
    int next = 0;
    // Descriptor copies run here, beside the caller's stream, so that a call's copy overlaps
    // the previous call's kernel instead of sitting between two kernels.
    cudaStream_t copy_stream = nullptr;
    unsigned int *status_dev = nullptr;
    unsigned int *status_host = nullptr;
    int64_t last_items = 0;
    int32_t last_ctas = 0;
    int32_t last_threads = 0;
    int64_t last_desc_bytes = 0;
    char err[512] = {0};
};

namespace {

kvx_status set_err(kvx_ctx *ctx, kvx_status st, const char *fmt, ...)
    __attribute__((format(printf, 3, 4)));

kvx_status set_err(kvx_ctx *ctx, kvx_status st, const char *fmt, ...)
{
    if (ctx) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(ctx->err, sizeof ctx->err, fmt, ap);
        va_end(ap);
    }
    return st;
}

kvx_status cuda_err(kvx_ctx *ctx, cudaError_t e, const char *what)
{
    return set_err(ctx, KVX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Copy a call's packed descriptors into its slot on the context's copy stream (zeroing
// `zero_bytes` at `zero_off` after them), and make the caller's stream wait for that.
// settle: the host waits for the copy first (a few microseconds), so that the caller's
// stream waits on an event that has already completed.  An overlapped launch needs that: a
// wait on a copy still in flight keeps it from starting before the kernel ahead of it ends,
// where a completed one does not.
cudaError_t stage(kvx_ctx *ctx, Slot &slot, size_t bytes, size_t zero_off, size_t zero_bytes,
                  cudaStream_t s, bool settle = false)
{
    cudaError_t e = cudaMemcpyAsync(slot.dev, slot.host, bytes, cudaMemcpyHostToDevice,
                                    ctx->copy_stream);
    if (e == cudaSuccess && zero_bytes)
        e = cudaMemsetAsync(slot.dev + zero_off, 0, zero_bytes, ctx->copy_stream);
    if (e == cudaSuccess)
        e = cudaEventRecord(slot.staged, ctx->copy_stream);
    if (e == cudaSuccess && settle)
        e = cudaEventSynchronize(slot.staged);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(s, slot.staged, 0);
    return e;
}

// Keeps ctx->device current for the duration of a call and restores the caller's device.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            prev = -1;
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess)
            ok = false;
    }
    ~DeviceGuard()
    {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

void defaults_for(const kvx_ctx *ctx, int op, kvx_launch_cfg *c)
{
    c->mapping = KVX_MAP_WARP_SEGMENT;
    c->stage_bytes = kDefaultStageBytes;
    c->batch = 0;
    c->overlap = 0;
    switch (op) {
    case KVX_OP_STORE:  // 8 SMs carry the device-to-host peak (about 45 GB/s each) and
                        // leave a concurrent load its own
        c->sm_cap = 8;
        c->ctas_per_sm = 1;
        c->threads = 1024;
        c->unroll = 8;
        c->store_hint = KVX_HINT_DEFAULT;
        break;
    case KVX_OP_LOAD:
        c->sm_cap = 16;
        c->ctas_per_sm = 1;
        c->threads = 1024;
        c->unroll = 8;
        c->store_hint = KVX_HINT_STREAMING;
        break;
    case KVX_OP_EXCHANGE:  // 20 SMs per direction
        c->sm_cap = 40;
        c->ctas_per_sm = 1;
        c->threads = 1024;
        c->unroll = 8;
        c->store_hint = KVX_HINT_DEFAULT;
        break;
    case KVX_OP_ROUNDTRIP:  // both directions mixed on 16 SMs
        c->sm_cap = 16;
        c->ctas_per_sm = 1;
        c->threads = 1024;
        c->unroll = 8;
        c->store_hint = KVX_HINT_DEFAULT;
        break;
    default:  // HBM transform: the whole GPU, two 256-thread CTAs per SM, 4 x 16 bytes in
              // flight per lane (2 x 32 bytes with 32-byte accesses)
        c->sm_cap = 0;
        c->ctas_per_sm = 2;
        c->threads = 256;
        c->unroll = 4;
        c->store_hint = KVX_HINT_STREAMING;
        break;
    }
    (void)ctx;
}

kvx_status resolve_cfg(kvx_ctx *ctx, int op, const kvx_launch_cfg *user, kvx_launch_cfg *out)
{
    kvx_launch_cfg d;
    defaults_for(ctx, op, &d);
    *out = d;
    if (!user)
        return KVX_OK;
    out->sm_cap = user->sm_cap;  // 0 means every SM
    if (user->ctas_per_sm)
        out->ctas_per_sm = user->ctas_per_sm;
    out->mapping = user->mapping;
    if (user->threads)
        out->threads = user->threads;
    if (user->unroll)
        out->unroll = user->unroll;
    out->store_hint = user->store_hint;
    out->stage_bytes = user->stage_bytes ? user->stage_bytes : kDefaultStageBytes;
    out->batch = user->batch;
    out->overlap = user->overlap;
    bool ok = out->sm_cap >= 0 && out->ctas_per_sm >= 1 && out->ctas_per_sm <= 32 &&
              out->batch >= 0 && out->batch <= 32 &&
              (out->store_hint == KVX_HINT_DEFAULT || out->store_hint == KVX_HINT_STREAMING);
    // Overlapped launches: single transfers on the warp-segment mapping only.
    if (out->overlap != 0)
        ok = ok && out->overlap == 1 && out->mapping == KVX_MAP_WARP_SEGMENT &&
             op >= KVX_OP_STORE && op <= KVX_OP_SCATTER_HBM;
    if (out->mapping == KVX_MAP_WARP_SEGMENT || out->mapping == KVX_MAP_CTA) {
        ok = ok && out->threads >= 32 && out->threads <= 1024 && out->threads % 32 == 0 &&
             pick_kernel(out->unroll, 0, 0);
    } else if (out->mapping == KVX_MAP_BULK) {
        // Three warps per CTA (segment lookups, two copy lanes); `unroll` counts the
        // shared-memory stages of each copy lane's ring.
        if (!user->unroll)
            out->unroll = kDefaultStages;
        out->threads = 32 * (1 + kBulkLanes);
        ok = ok && out->unroll >= 2 && out->unroll <= kBulkMaxStages &&
             out->stage_bytes >= 16 && out->stage_bytes % 16 == 0 &&
             int64_t(kBulkLanes) * out->unroll * out->stage_bytes <= kMaxBulkSmem;
    } else {
        ok = false;
    }
    if (!ok)
        return set_err(ctx, KVX_ERR_INVALID_ARG,
                       "launch cfg: sm_cap %d ctas_per_sm %d threads %d unroll %d hint %d "
                       "mapping %d stage_bytes %d batch %d overlap %d (overlap: store, load "
                       "and transform on the warp-segment mapping only)", user->sm_cap,
                       user->ctas_per_sm, user->threads, user->unroll, user->store_hint,
                       user->mapping, user->stage_bytes, user->batch, user->overlap);
    return KVX_OK;
}

// Kernel, grid and shared memory of one transfer launch.
struct LaunchShape {
    const void *fn = nullptr;
    int64_t ctas = 0;
    int threads = 0;
    size_t smem = 0;
    int bulk = 0;
    int stage_bytes = 0;
    int stages = 0;
    bool overlap = false;  // programmatic dependent launch (kvx_launch_cfg.overlap)
};

// Row slices per segment for a warp-segment launch of one segment per warp: when the batch
// has fewer segments than the grid has warps, each segment is cut into enough slices (at
// most 8, at most its page's rows) to give the spare warps work.
void choose_split(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, Plan *plan)
{
    plan->split = 1;
    if (cfg.mapping != KVX_MAP_WARP_SEGMENT || plan->batch != 1 || plan->total_items <= 0)
        return;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    const int64_t warps = int64_t(sms) * cfg.ctas_per_sm * (cfg.threads / 32);
    if (plan->total_items >= warps)
        return;
    int64_t split = (warps + plan->total_items - 1) / plan->total_items;
    split = std::min<int64_t>(split, std::min<int64_t>(8, plan->page_size));
    plan->split = int32_t(std::max<int64_t>(split, 1));
}

// True when every address an HBM transform touches is a multiple of 32 bytes: token_bytes,
// every pool layer and every chunk (then all strides and offsets are too), so the kernel
// may use 32-byte accesses.
bool aligned32(const kvx_pool *pool, const kvx_chunk *chunks, int n_chunks)
{
    if (pool->token_bytes % 32 != 0)
        return false;
    for (int k = 0; k < pool->kv_factor; ++k)
        for (int l = 0; l < pool->num_layers; ++l)
            if (reinterpret_cast<uintptr_t>((k == 0 ? pool->k_pages : pool->v_pages)[l]) % 32)
                return false;
    for (int c = 0; c < n_chunks; ++c)
        if (reinterpret_cast<uintptr_t>(chunks[c].ptr) % 32)
            return false;
    return true;
}

// 32-byte accesses for an HBM transform of the warp-segment mapping on aligned memory (on
// GB300 they move HBM-to-HBM 1.5-2 % faster; host transfers are link-bound either way).
bool use_w32(int op, const kvx_launch_cfg &cfg, const kvx_pool *pool, const kvx_chunk *chunks,
             int n_chunks)
{
    return (op == KVX_OP_GATHER_HBM || op == KVX_OP_SCATTER_HBM) &&
           cfg.mapping == KVX_MAP_WARP_SEGMENT && aligned32(pool, chunks, n_chunks);
}

// Whether page segments of more than one token are strided on the chunk side: the chunks
// include a token-major one of more than one (layer, kv) slab.
bool strided_rows(const kvx_pool *pool, const kvx_chunk *chunks, int n_chunks)
{
    if (pool->page_size == 1)
        return false;
    for (int c = 0; c < n_chunks; ++c)
        if (chunks[c].layout == KVX_CHUNK_TOKEN_MAJOR &&
            int64_t(chunks[c].n_layers) * pool->kv_factor > 1)
            return true;
    return false;
}

// The row-walking segment kernel (kvx_rows_kernel): a warp-segment launch, not with 32-byte
// accesses, with strided rows.
bool use_rows(const kvx_launch_cfg &cfg, const kvx_pool *pool, const kvx_chunk *chunks,
              int n_chunks, bool w32)
{
    return !w32 && cfg.mapping == KVX_MAP_WARP_SEGMENT && strided_rows(pool, chunks, n_chunks);
}

LaunchShape launch_shape(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &plan, int dir,
                         bool w32 = false, bool rows = false)
{
    LaunchShape sh;
    const int64_t warps_per_cta = cfg.threads / 32;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    int64_t ctas = int64_t(sms) * cfg.ctas_per_sm;
    const bool split = cfg.mapping == KVX_MAP_WARP_SEGMENT && plan.split > 1;
    const int64_t per_cta = cfg.mapping == KVX_MAP_CTA    ? 32
                            : cfg.mapping == KVX_MAP_BULK ? 1
                                                          : warps_per_cta * plan.batch;
    const int64_t work = split ? plan.total_items * plan.split : plan.total_items;
    const int64_t needed = (work + per_cta - 1) / per_cta;
    if (ctas > needed)
        ctas = needed;
    sh.ctas = ctas;
    if (cfg.mapping == KVX_MAP_BULK) {
        sh.fn = dir == KVX_DIR_GATHER
                    ? reinterpret_cast<const void *>(kvx_bulk_kernel<KVX_DIR_GATHER>)
                    : reinterpret_cast<const void *>(kvx_bulk_kernel<KVX_DIR_SCATTER>);
        sh.threads = 32 * (1 + kBulkLanes);
        sh.bulk = 1;
        sh.stage_bytes = cfg.stage_bytes;
        sh.stages = cfg.unroll;
        sh.smem = size_t(kBulkLanes) * cfg.unroll * cfg.stage_bytes;
    } else if (cfg.mapping == KVX_MAP_CTA) {
        sh.fn = reinterpret_cast<const void *>(pick_cta(cfg.unroll, dir, cfg.store_hint));
        sh.threads = cfg.threads;
    }
    sh.overlap = cfg.overlap == 1 && cfg.mapping == KVX_MAP_WARP_SEGMENT;
    if (cfg.mapping == KVX_MAP_WARP_SEGMENT && split) {
        sh.fn = reinterpret_cast<const void *>(
            pick_split(cfg.unroll, dir, cfg.store_hint, sh.overlap));
        sh.threads = cfg.threads;
    } else if (cfg.mapping == KVX_MAP_WARP_SEGMENT) {
        sh.fn = reinterpret_cast<const void *>(
            pick_kernel(cfg.unroll, dir, cfg.store_hint, plan.batch, w32, sh.overlap, rows));
        sh.threads = cfg.threads;
    }
    return sh;
}

cudaError_t launch_kernel(const LaunchShape &sh, Plan plan, cudaStream_t s)
{
    if (sh.bulk) {
        cudaError_t e = cudaFuncSetAttribute(sh.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(sh.smem));
        if (e != cudaSuccess)
            return e;
        int stage_bytes = sh.stage_bytes, stages = sh.stages;
        void *args[] = {&plan, &stage_bytes, &stages};
        return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(unsigned(sh.threads)), args,
                                sh.smem, s);
    }
    void *args[] = {&plan};
    if (!sh.overlap)
        return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(unsigned(sh.threads)), args,
                                0, s);
    // May start once every CTA of the previous kernel on s has started; the kernel waits for
    // that kernel's completion before it exits.
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(unsigned(sh.ctas));
    lc.blockDim = dim3(unsigned(sh.threads));
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelExC(&lc, sh.fn, args);
}

// Every call starts with an empty last-launch record, so a call that fails or moves
// nothing reports zeros.
void begin_call(kvx_ctx *ctx)
{
    ctx->last_items = 0;
    ctx->last_ctas = 0;
    ctx->last_threads = 0;
    ctx->last_desc_bytes = 0;
}

// The context's next descriptor slot, once the launch that last used it has finished.
kvx_status acquire_slot(kvx_ctx *ctx, size_t bytes, Slot **out)
{
    if (bytes > ctx->slot_bytes)
        return set_err(ctx, KVX_ERR_CAPACITY,
                       "descriptors need %zu bytes, the context holds %zu per call; create it "
                       "with a larger max_descriptor_bytes", bytes, ctx->slot_bytes);
    Slot &slot = ctx->slots[ctx->next];
    if (slot.used) {
        cudaError_t e = cudaEventSynchronize(slot.done);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "waiting for a descriptor buffer");
    }
    *out = &slot;
    return KVX_OK;
}

// After a launch: the slot stays busy until `s` passes this point; record the launch.
kvx_status finish_call(kvx_ctx *ctx, Slot &slot, cudaStream_t s, int64_t items, int64_t ctas,
                       int threads, size_t desc_bytes)
{
    cudaError_t e = cudaEventRecord(slot.done, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "event record");
    slot.used = true;
    ctx->next = (ctx->next + 1) % kSlots;
    ctx->last_items = items;
    ctx->last_ctas = int32_t(ctas);
    ctx->last_threads = threads;
    ctx->last_desc_bytes = int64_t(desc_bytes);
    return KVX_OK;
}

// Launch configuration of an exchange or round trip: warp-segment mapping only.
kvx_status resolve_pair_cfg(kvx_ctx *ctx, int op, const kvx_launch_cfg *user, kvx_launch_cfg *cfg)
{
    kvx_status st = resolve_cfg(ctx, op, user, cfg);
    if (st == KVX_OK && cfg->mapping != KVX_MAP_WARP_SEGMENT)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "%s runs the warp-segment mapping only",
                       op == KVX_OP_EXCHANGE ? "exchange" : "round trip");
    return st;
}

// Segments a warp resolves at once: the configured batch, else the packed default (about
// 32 KiB of segments), with two long segments per warp for the HBM transform (their
// lookups then overlap).  Round trips take theirs from kvx::roundtrip_rule.
void apply_batch(int op, const kvx_launch_cfg &cfg, Plan *plan)
{
    if (cfg.batch > 0)
        plan->batch = cfg.batch;
    else if ((op == KVX_OP_GATHER_HBM || op == KVX_OP_SCATTER_HBM) && plan->batch == 1)
        plan->batch = 2;
}

// With no configuration given, a store or load of page segments shorter than
// kShortSegmentBytes runs on 32 SMs instead of the default 8 or 16, as the round trip does for
// its short segments: a warp then moves one short segment per pass and the link needs more
// warps to keep enough host accesses in flight.  Call after validation (the pool is sound).
void short_segment_grid(int op, const kvx_launch_cfg *user, const kvx_pool *pool,
                        kvx_launch_cfg *cfg)
{
    if (!user && (op == KVX_OP_STORE || op == KVX_OP_LOAD) &&
        int64_t(pool->page_size) * pool->token_bytes < kShortSegmentBytes)
        cfg->sm_cap = kShortSegmentSms;
}

int op_dir(int op)
{
    return (op == KVX_OP_LOAD || op == KVX_OP_SCATTER_HBM) ? KVX_DIR_SCATTER : KVX_DIR_GATHER;
}

kvx_status launch(kvx_ctx *ctx, int op, const kvx_pool *pool, const kvx_request *reqs, int n_req,
                  const kvx_chunk *chunks, int n_chunks, int layer_begin, int layer_end,
                  const kvx_launch_cfg *user_cfg, kvx_stream_t stream)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    begin_call(ctx);
    kvx_launch_cfg cfg;
    kvx_status st = resolve_cfg(ctx, op, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, op,
                       ctx->validation, true, ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    short_segment_grid(op, user_cfg, pool, &cfg);
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    Slot *slot = nullptr;
    if ((st = acquire_slot(ctx, lay.total, &slot)) != KVX_OK)
        return st;
    const int dir = op_dir(op);
    Plan plan = kvx::pack(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, dir, lay,
                          slot->host, slot->dev);
    plan.status = ctx->status_dev;
    apply_batch(op, cfg, &plan);
    choose_split(ctx, cfg, &plan);
    if (plan.total_items == 0)
        return KVX_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool w32 = use_w32(op, cfg, pool, chunks, n_chunks);
    const LaunchShape shape = launch_shape(ctx, cfg, plan, dir, w32,
                                           use_rows(cfg, pool, chunks, n_chunks, w32));
    cudaError_t e = stage(ctx, *slot, lay.total, 0, 0, s, shape.overlap);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "descriptor copy");
    e = launch_kernel(shape, plan, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "kernel launch");
    return finish_call(ctx, *slot, s, plan.total_items, shape.ctas, shape.threads, lay.total);
}

// An exchange whose batches differ in size by more than this factor (in segments) shares its
// units between all warps (kvx_duplex_kernel): with the role split the smaller batch's half
// of the grid would finish early and leave the larger batch on half the CTAs.  Batches of
// similar size keep the role split, which measured 2-5 % faster for them, unless their page
// segments are shorter than kShortSegmentBytes: then every warp mixing both directions
// keeps more of each in flight (one-token MLA pages: 335 GB/s shared, 305 split).
constexpr double kExchangeShareRatio = 1.5;

bool exchange_shared(const Plan &ps, const Plan &pl)
{
    const double a = double(ps.total_items), b = double(pl.total_items);
    if (a > kExchangeShareRatio * b || b > kExchangeShareRatio * a)
        return true;
    return int64_t(ps.page_size) * ps.token_bytes < kShortSegmentBytes && ps.batch == pl.batch;
}

// Work counters and grid of a shared exchange; `next` is a zeroed 256-byte device word.
bool duplex_setup(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &ps, const Plan &pl,
                  unsigned *next, DuplexSync *sy, LaunchShape *sh, bool rows)
{
    sy->unit_items = ps.batch;
    sy->units_s = (ps.total_items + sy->unit_items - 1) / sy->unit_items;
    sy->units_l = (pl.total_items + sy->unit_items - 1) / sy->unit_items;
    sy->next = next;
    if (ps.batch != pl.batch || sy->units_s >= (int64_t(1) << 31) ||
        sy->units_l >= (int64_t(1) << 31))
        return false;
    const int64_t warps_per_cta = cfg.threads / 32;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    int64_t ctas = int64_t(sms) * cfg.ctas_per_sm;
    const int64_t needed = (sy->units_s + sy->units_l + warps_per_cta - 1) / warps_per_cta;
    if (ctas > needed)
        ctas = needed;
    sh->ctas = ctas;
    sh->threads = cfg.threads;
    sh->fn = reinterpret_cast<const void *>(pick_duplex(cfg.unroll, ps.batch > 1, rows));
    return true;
}

cudaError_t launch_duplex_kernel(const LaunchShape &sh, Plan ps, Plan pl, DuplexSync sy,
                                 cudaStream_t s)
{
    void *args[] = {&ps, &pl, &sy};
    return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(unsigned(sh.threads)), args, 0,
                            s);
}

// Exchange grid: sm_cap covers both directions, half of the CTAs per direction.
LaunchShape exchange_shape(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &ps,
                           const Plan &pl, bool rows)
{
    LaunchShape sh;
    const int64_t warps_per_cta = cfg.threads / 32;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    const int64_t per_dir = (int64_t(sms) * cfg.ctas_per_sm + 1) / 2;
    auto needed = [&](const Plan &p) {
        const int64_t per_cta = warps_per_cta * p.batch;
        return (p.total_items + per_cta - 1) / per_cta;
    };
    int64_t role = std::max(needed(ps), needed(pl));
    if (role > per_dir)
        role = per_dir;
    sh.ctas = 2 * role;
    sh.threads = cfg.threads;
    sh.fn = reinterpret_cast<const void *>(pick_exchange(cfg.unroll, ps.batch, pl.batch, rows));
    return sh;
}

cudaError_t launch_exchange_kernel(const LaunchShape &sh, Plan ps, Plan pl, cudaStream_t s)
{
    void *args[] = {&ps, &pl};
    return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(unsigned(sh.threads)), args, 0,
                            s);
}

kvx_status launch_exchange(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *sreqs,
                           int n_sreq, const kvx_chunk *schunks, int n_schunks,
                           const kvx_request *lreqs, int n_lreq, const kvx_chunk *lchunks,
                           int n_lchunks, int layer_begin, int layer_end,
                           const kvx_launch_cfg *user_cfg, kvx_stream_t stream)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    begin_call(ctx);
    kvx_launch_cfg cfg;
    kvx_status st = resolve_pair_cfg(ctx, KVX_OP_EXCHANGE, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate_exchange(pool, sreqs, n_sreq, schunks, n_schunks, lreqs, n_lreq, lchunks,
                                n_lchunks, layer_begin, layer_end, ctx->validation, true,
                                ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const kvx::PackedLayout ls = kvx::packed_layout(pool, n_sreq, n_schunks);
    const kvx::PackedLayout ll = kvx::packed_layout(pool, n_lreq, n_lchunks);
    const size_t total = ls.total + ll.total;  // then 256 bytes of work counters
    Slot *slot = nullptr;
    if ((st = acquire_slot(ctx, total + 256, &slot)) != KVX_OK)
        return st;
    Plan ps = kvx::pack(pool, sreqs, n_sreq, schunks, n_schunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, ls, slot->host, slot->dev);
    Plan pl = kvx::pack(pool, lreqs, n_lreq, lchunks, n_lchunks, layer_begin, layer_end,
                        KVX_DIR_SCATTER, ll, slot->host + ls.total, slot->dev + ls.total);
    ps.status = pl.status = ctx->status_dev;
    apply_batch(KVX_OP_EXCHANGE, cfg, &ps);
    apply_batch(KVX_OP_EXCHANGE, cfg, &pl);
    if (ps.total_items + pl.total_items == 0)
        return KVX_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    LaunchShape shape;
    const bool rows =
        strided_rows(pool, schunks, n_schunks) || strided_rows(pool, lchunks, n_lchunks);
    if (exchange_shared(ps, pl)) {
        DuplexSync sy;
        if (!duplex_setup(ctx, cfg, ps, pl, reinterpret_cast<unsigned *>(slot->dev + total), &sy,
                          &shape, rows))
            return set_err(ctx, KVX_ERR_CAPACITY, "exchange batches of %lld and %lld segments "
                           "(%d and %d per warp) do not fit one shared launch",
                           (long long)ps.total_items, (long long)pl.total_items, ps.batch,
                           pl.batch);
        e = stage(ctx, *slot, total, total, 256, s);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "descriptor copy");
        e = launch_duplex_kernel(shape, ps, pl, sy, s);
    } else {
        e = stage(ctx, *slot, total, 0, 0, s);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "descriptor copy");
        shape = exchange_shape(ctx, cfg, ps, pl, rows);
        e = launch_exchange_kernel(shape, ps, pl, s);
    }
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "kernel launch");
    return finish_call(ctx, *slot, s, ps.total_items + pl.total_items, shape.ctas, shape.threads,
                       total);
}

int64_t roundtrip_units(const Plan &ps, int slices)
{
    return slices > 1 ? ps.total_items * slices : (ps.total_items + ps.batch - 1) / ps.batch;
}

// Units, lag and grid of a round trip whose work counters and completion words start at
// `sync` (sync_bytes(), zeroed before each launch).  False when the units do not fit the
// kernel's 32-bit unit indices.
bool roundtrip_setup(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &ps, int slices,
                     char *sync, RoundTripSync *sy, LaunchShape *sh, bool rows)
{
    sy->slices = slices;
    sy->unit_items = sy->slices > 1 ? 1 : ps.batch;
    sy->units = roundtrip_units(ps, sy->slices);
    if (sy->units >= (int64_t(1) << 31))
        return false;
    sy->next = reinterpret_cast<unsigned *>(sync);
    sy->done = reinterpret_cast<unsigned *>(sync + 256);
    const int64_t warps_per_cta = cfg.threads / 32;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    int64_t ctas = int64_t(sms) * cfg.ctas_per_sm;
    const int64_t needed = (2 * sy->units + warps_per_cta - 1) / warps_per_cta;
    if (ctas > needed)
        ctas = needed;
    sy->lag = unsigned(ctas * warps_per_cta);  // one unit per warp of the grid
    sy->wait_ns = kWaitLimitNs;
    sh->ctas = ctas;
    sh->threads = cfg.threads;
    sh->fn = reinterpret_cast<const void *>(pick_roundtrip(cfg.unroll, ps.batch > 1, rows));
    return true;
}

size_t roundtrip_sync_bytes(const Plan &ps, int slices)
{
    return 256 + sizeof(unsigned) * size_t(roundtrip_units(ps, slices));
}

// The round trip's units and SM cap (kvx::roundtrip_rule) for a validated pool; sets the
// SM cap in cfg and returns the rule.
kvx::RoundTripRule roundtrip_rule_for(const kvx_ctx *ctx, const kvx_pool *pool,
                                      const kvx_launch_cfg *user_cfg, kvx_launch_cfg *cfg)
{
    const kvx::RoundTripRule r = kvx::roundtrip_rule(pool->page_size, pool->token_bytes,
                                                     user_cfg != nullptr, cfg->sm_cap,
                                                     cfg->batch, ctx->num_sms);
    cfg->sm_cap = r.sm_cap;
    return r;
}

// sync_bytes > 0: zero the counters and completion words on `s` first (plans; calls zero
// them with their descriptor copy).
cudaError_t launch_roundtrip_kernel(const LaunchShape &sh, Plan ps, Plan pl, RoundTripSync sy,
                                    size_t sync_bytes, cudaStream_t s)
{
    if (sync_bytes) {
        cudaError_t e = cudaMemsetAsync(sy.next, 0, sync_bytes, s);
        if (e != cudaSuccess)
            return e;
    }
    void *args[] = {&ps, &pl, &sy};
    return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(unsigned(sh.threads)), args, 0,
                            s);
}

// Descriptor slot of a round trip: the store plan, the load plan (same chunks, other page
// tables), then the work counters and one completion word per unit, zeroed per launch.
// test_wait_ns > 0 (kvx_test_roundtrip_timeout): the store counter starts at the unit count,
// so every store counts as handed out and none is done, and each load unit's wait ends
// after test_wait_ns without its store.
kvx_status launch_roundtrip(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *src_reqs,
                            const kvx_request *dst_reqs, int n_req, const kvx_chunk *chunks,
                            int n_chunks, int layer_begin, int layer_end,
                            const kvx_launch_cfg *user_cfg, kvx_stream_t stream,
                            uint64_t test_wait_ns = 0)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    begin_call(ctx);
    kvx_launch_cfg cfg;
    kvx_status st = resolve_pair_cfg(ctx, KVX_OP_ROUNDTRIP, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate_exchange(pool, src_reqs, n_req, chunks, n_chunks, dst_reqs, n_req, chunks,
                                n_chunks, layer_begin, layer_end, ctx->validation, true,
                                ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    const kvx::RoundTripRule rule = roundtrip_rule_for(ctx, pool, user_cfg, &cfg);
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    const size_t sync_off = 2 * lay.total;
    Slot *slot = nullptr;
    if ((st = acquire_slot(ctx, sync_off + 256, &slot)) != KVX_OK)
        return st;
    Plan ps = kvx::pack(pool, src_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, lay, slot->host, slot->dev);
    Plan pl = kvx::pack(pool, dst_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_SCATTER, lay, slot->host + lay.total, slot->dev + lay.total);
    ps.status = pl.status = ctx->status_dev;
    ps.batch = pl.batch = rule.batch;
    if (ps.total_items == 0)
        return KVX_OK;
    // The completion words (4 bytes per unit) are known only now that the plan is packed.
    const size_t sync_bytes = roundtrip_sync_bytes(ps, rule.slices);
    if (sync_off + sync_bytes > ctx->slot_bytes)
        return set_err(ctx, KVX_ERR_CAPACITY,
                       "round trip of %lld segments needs %zu bytes of descriptors and "
                       "completion words, the context holds %zu per call",
                       (long long)ps.total_items, sync_off + sync_bytes, ctx->slot_bytes);
    RoundTripSync sy;
    LaunchShape shape;
    if (!roundtrip_setup(ctx, cfg, ps, rule.slices, slot->dev + sync_off, &sy, &shape,
                         strided_rows(pool, chunks, n_chunks)))
        return set_err(ctx, KVX_ERR_CAPACITY, "round trip of %lld segments (%d per unit) has "
                       "2^31 units or more", (long long)ps.total_items, ps.batch);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = stage(ctx, *slot, sync_off, sync_off, sync_bytes, s);
    if (e == cudaSuccess && test_wait_ns) {
        sy.wait_ns = test_wait_ns;
        const unsigned all_stores = unsigned(sy.units);
        std::memcpy(slot->host + sync_off, &all_stores, sizeof all_stores);
        e = cudaMemcpyAsync(sy.next, slot->host + sync_off, sizeof all_stores,
                            cudaMemcpyHostToDevice, s);
    }
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "descriptor copy");
    e = launch_roundtrip_kernel(shape, ps, pl, sy, 0, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "kernel launch");
    return finish_call(ctx, *slot, s, 2 * ps.total_items, shape.ctas, shape.threads, sync_off);
}

}  // namespace

// A transfer validated and packed once, its descriptors in device memory of its own.
struct kvx_plan {
    kvx_ctx *ctx = nullptr;
    char *dev = nullptr;
    Plan plan;       // the transfer; the store half of an exchange
    Plan load;       // the load half of an exchange
    bool exchange = false;
    bool shared = false;     // shared-work exchange: its counters are zeroed before each launch
    bool roundtrip = false;  // round trip: counters and completion words zeroed per launch
    DuplexSync sync;
    RoundTripSync rsync;
    size_t sync_bytes = 0;
    LaunchShape shape;
};

extern "C" {

kvx_status kvx_plan_create(kvx_ctx *ctx, int op, const kvx_pool *pool, const kvx_request *reqs,
                           int n_req, const kvx_chunk *chunks, int n_chunks, int layer_begin,
                           int layer_end, const kvx_launch_cfg *user_cfg, kvx_stream_t stream,
                           kvx_plan **out)
{
    if (!ctx || !out)
        return KVX_ERR_INVALID_ARG;
    *out = nullptr;
    if (op < KVX_OP_STORE || op > KVX_OP_SCATTER_HBM)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "plans take store, load or transform ops");
    kvx_launch_cfg cfg;
    kvx_status st = resolve_cfg(ctx, op, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, op,
                       ctx->validation, true, ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    short_segment_grid(op, user_cfg, pool, &cfg);
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const int dir = op_dir(op);
    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    kvx_plan *p = new kvx_plan();
    p->ctx = ctx;
    std::vector<char> host(lay.total);
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&p->dev), lay.total);
    if (e != cudaSuccess) {
        delete p;
        return cuda_err(ctx, e, "plan descriptor buffer");
    }
    p->plan = kvx::pack(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, dir, lay,
                        host.data(), p->dev);
    p->plan.status = ctx->status_dev;
    apply_batch(op, cfg, &p->plan);
    choose_split(ctx, cfg, &p->plan);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(p->dev, host.data(), lay.total, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);  // the host image dies with this call
    if (e != cudaSuccess) {
        cudaFree(p->dev);
        delete p;
        return cuda_err(ctx, e, "plan descriptor copy");
    }
    const bool w32 = use_w32(op, cfg, pool, chunks, n_chunks);
    p->shape = launch_shape(ctx, cfg, p->plan, dir, w32,
                            use_rows(cfg, pool, chunks, n_chunks, w32));
    *out = p;
    return KVX_OK;
}

kvx_status kvx_plan_create_exchange(kvx_ctx *ctx, const kvx_pool *pool,
                                    const kvx_request *sreqs, int n_sreq,
                                    const kvx_chunk *schunks, int n_schunks,
                                    const kvx_request *lreqs, int n_lreq,
                                    const kvx_chunk *lchunks, int n_lchunks, int layer_begin,
                                    int layer_end, const kvx_launch_cfg *user_cfg,
                                    kvx_stream_t stream, kvx_plan **out)
{
    if (!ctx || !out)
        return KVX_ERR_INVALID_ARG;
    *out = nullptr;
    kvx_launch_cfg cfg;
    kvx_status st = resolve_pair_cfg(ctx, KVX_OP_EXCHANGE, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate_exchange(pool, sreqs, n_sreq, schunks, n_schunks, lreqs, n_lreq, lchunks,
                                n_lchunks, layer_begin, layer_end, ctx->validation, true,
                                ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const kvx::PackedLayout ls = kvx::packed_layout(pool, n_sreq, n_schunks);
    const kvx::PackedLayout ll = kvx::packed_layout(pool, n_lreq, n_lchunks);
    const size_t total = ls.total + ll.total;
    kvx_plan *p = new kvx_plan();
    p->ctx = ctx;
    p->exchange = true;
    std::vector<char> host(total);
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&p->dev), total + 256);
    if (e != cudaSuccess) {
        delete p;
        return cuda_err(ctx, e, "plan descriptor buffer");
    }
    p->plan = kvx::pack(pool, sreqs, n_sreq, schunks, n_schunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, ls, host.data(), p->dev);
    p->load = kvx::pack(pool, lreqs, n_lreq, lchunks, n_lchunks, layer_begin, layer_end,
                        KVX_DIR_SCATTER, ll, host.data() + ls.total, p->dev + ls.total);
    p->plan.status = p->load.status = ctx->status_dev;
    apply_batch(KVX_OP_EXCHANGE, cfg, &p->plan);
    apply_batch(KVX_OP_EXCHANGE, cfg, &p->load);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(p->dev, host.data(), total, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);  // the host image dies with this call
    if (e != cudaSuccess) {
        cudaFree(p->dev);
        delete p;
        return cuda_err(ctx, e, "plan descriptor copy");
    }
    p->shared = exchange_shared(p->plan, p->load);
    const bool rows =
        strided_rows(pool, schunks, n_schunks) || strided_rows(pool, lchunks, n_lchunks);
    if (!p->shared) {
        p->shape = exchange_shape(ctx, cfg, p->plan, p->load, rows);
    } else if (!duplex_setup(ctx, cfg, p->plan, p->load,
                             reinterpret_cast<unsigned *>(p->dev + total), &p->sync, &p->shape,
                             rows)) {
        cudaFree(p->dev);
        delete p;
        return set_err(ctx, KVX_ERR_CAPACITY, "exchange batches do not fit one shared launch");
    }
    *out = p;
    return KVX_OK;
}

kvx_status kvx_plan_create_roundtrip(kvx_ctx *ctx, const kvx_pool *pool,
                                     const kvx_request *src_reqs, const kvx_request *dst_reqs,
                                     int n_req, const kvx_chunk *chunks, int n_chunks,
                                     int layer_begin, int layer_end,
                                     const kvx_launch_cfg *user_cfg, kvx_stream_t stream,
                                     kvx_plan **out)
{
    if (!ctx || !out)
        return KVX_ERR_INVALID_ARG;
    *out = nullptr;
    kvx_launch_cfg cfg;
    kvx_status st = resolve_pair_cfg(ctx, KVX_OP_ROUNDTRIP, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate_exchange(pool, src_reqs, n_req, chunks, n_chunks, dst_reqs, n_req, chunks,
                                n_chunks, layer_begin, layer_end, ctx->validation, true,
                                ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    const kvx::RoundTripRule rule = roundtrip_rule_for(ctx, pool, user_cfg, &cfg);
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    std::vector<char> host(2 * lay.total);
    kvx_plan *p = new kvx_plan();
    p->ctx = ctx;
    p->exchange = true;
    p->roundtrip = true;
    // Pack once to learn the item count (device addresses not final), then size the
    // allocation and pack again.
    p->plan = kvx::pack(pool, src_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, lay, host.data(), host.data());
    p->plan.batch = rule.batch;
    if (roundtrip_units(p->plan, rule.slices) >= (int64_t(1) << 31)) {
        delete p;
        return set_err(ctx, KVX_ERR_CAPACITY, "round trip of %lld segments (%d per unit) has "
                       "2^31 units or more", (long long)p->plan.total_items, p->plan.batch);
    }
    p->sync_bytes = roundtrip_sync_bytes(p->plan, rule.slices);
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&p->dev), 2 * lay.total + p->sync_bytes);
    if (e != cudaSuccess) {
        delete p;
        return cuda_err(ctx, e, "plan descriptor buffer");
    }
    p->plan = kvx::pack(pool, src_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, lay, host.data(), p->dev);
    p->load = kvx::pack(pool, dst_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_SCATTER, lay, host.data() + lay.total, p->dev + lay.total);
    p->plan.status = p->load.status = ctx->status_dev;
    p->plan.batch = p->load.batch = rule.batch;
    // The unit count was checked above, so the setup cannot fail here.
    roundtrip_setup(ctx, cfg, p->plan, rule.slices, p->dev + 2 * lay.total, &p->rsync,
                    &p->shape, strided_rows(pool, chunks, n_chunks));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(p->dev, host.data(), 2 * lay.total, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);  // the host image dies with this call
    if (e != cudaSuccess) {
        cudaFree(p->dev);
        delete p;
        return cuda_err(ctx, e, "plan descriptor copy");
    }
    *out = p;
    return KVX_OK;
}

kvx_status kvx_plan_launch(const kvx_plan *p, kvx_stream_t stream)
{
    if (!p)
        return KVX_ERR_INVALID_ARG;
    if (p->plan.total_items + (p->exchange && !p->roundtrip ? p->load.total_items : 0) == 0)
        return KVX_OK;
    DeviceGuard guard(p->ctx->device);  // the plan's memory lives on its context's GPU
    if (!guard.ok)
        return set_err(p->ctx, KVX_ERR_CUDA, "cannot make device %d current", p->ctx->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p->roundtrip) {
        e = launch_roundtrip_kernel(p->shape, p->plan, p->load, p->rsync, p->sync_bytes, s);
    } else if (p->shared) {
        e = cudaMemsetAsync(p->sync.next, 0, 256, s);
        if (e == cudaSuccess)
            e = launch_duplex_kernel(p->shape, p->plan, p->load, p->sync, s);
    } else {
        e = p->exchange ? launch_exchange_kernel(p->shape, p->plan, p->load, s)
                        : launch_kernel(p->shape, p->plan, s);
    }
    if (e != cudaSuccess)
        return cuda_err(p->ctx, e, "plan launch");
    return KVX_OK;
}

void kvx_plan_destroy(kvx_plan *p)
{
    if (!p)
        return;
    if (p->dev) {
        DeviceGuard guard(p->ctx->device);
        cudaDeviceSynchronize();
        cudaFree(p->dev);
    }
    delete p;
}

kvx_status kvx_create(kvx_ctx **out, int device, size_t max_descriptor_bytes)
{
    if (!out)
        return KVX_ERR_INVALID_ARG;
    *out = nullptr;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) {
        cudaGetLastError();
        return KVX_ERR_CUDA;
    }
    kvx_ctx *ctx = new kvx_ctx();
    ctx->device = device;
    ctx->slot_bytes = max_descriptor_bytes ? max_descriptor_bytes : kDefaultDescriptorBytes;
    DeviceGuard guard(device);
    cudaError_t e = guard.ok ? cudaSuccess : cudaErrorInvalidDevice;
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i) {
        e = cudaHostAlloc(reinterpret_cast<void **>(&ctx->slots[i].host), ctx->slot_bytes,
                          cudaHostAllocDefault);
        if (e == cudaSuccess)
            e = cudaMalloc(reinterpret_cast<void **>(&ctx->slots[i].dev), ctx->slot_bytes);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&ctx->slots[i].done, cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&ctx->slots[i].staged, cudaEventDisableTiming);
    }
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&ctx->status_dev), 256);
    if (e == cudaSuccess)
        e = cudaMemset(ctx->status_dev, 0, 256);
    if (e == cudaSuccess)
        e = cudaHostAlloc(reinterpret_cast<void **>(&ctx->status_host), 64, cudaHostAllocDefault);
    if (e != cudaSuccess) {
        kvx_destroy(ctx);
        return KVX_ERR_CUDA;
    }
    *out = ctx;
    return KVX_OK;
}

void kvx_destroy(kvx_ctx *ctx)
{
    if (!ctx)
        return;
    {
        DeviceGuard guard(ctx->device);
        for (int i = 0; i < kSlots; ++i) {
            Slot &s = ctx->slots[i];
            if (s.done) {
                if (s.used)
                    cudaEventSynchronize(s.done);
                cudaEventDestroy(s.done);
            }
            if (s.staged)
                cudaEventDestroy(s.staged);
            if (s.dev)
                cudaFree(s.dev);
            if (s.host)
                cudaFreeHost(s.host);
        }
        if (ctx->copy_stream) {
            cudaStreamSynchronize(ctx->copy_stream);
            cudaStreamDestroy(ctx->copy_stream);
        }
        if (ctx->status_dev)
            cudaFree(ctx->status_dev);
        if (ctx->status_host)
            cudaFreeHost(ctx->status_host);
    }
    delete ctx;
}

kvx_status kvx_set_validation(kvx_ctx *ctx, int level)
{
    if (!ctx || level < 0 || level > 2)
        return KVX_ERR_INVALID_ARG;
    ctx->validation = level;
    return KVX_OK;
}

kvx_status kvx_default_launch_cfg(const kvx_ctx *ctx, int op, kvx_launch_cfg *cfg)
{
    if (!ctx || !cfg || op < KVX_OP_STORE || op > KVX_OP_ROUNDTRIP)
        return KVX_ERR_INVALID_ARG;
    defaults_for(ctx, op, cfg);
    return KVX_OK;
}

kvx_status kvx_store_chunks(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *reqs,
                            int n_req, const kvx_chunk *chunks, int n_chunks, int layer_begin,
                            int layer_end, const kvx_launch_cfg *cfg, kvx_stream_t stream)
{
    return launch(ctx, KVX_OP_STORE, pool, reqs, n_req, chunks, n_chunks, layer_begin,
                  layer_end, cfg, stream);
}

kvx_status kvx_load_chunks(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *reqs,
                           int n_req, const kvx_chunk *chunks, int n_chunks, int layer_begin,
                           int layer_end, const kvx_launch_cfg *cfg, kvx_stream_t stream)
{
    return launch(ctx, KVX_OP_LOAD, pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                  cfg, stream);
}

kvx_status kvx_exchange_chunks(kvx_ctx *ctx, const kvx_pool *pool,
                               const kvx_request *store_reqs, int n_store_req,
                               const kvx_chunk *store_chunks, int n_store_chunks,
                               const kvx_request *load_reqs, int n_load_req,
                               const kvx_chunk *load_chunks, int n_load_chunks,
                               int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                               kvx_stream_t stream)
{
    return launch_exchange(ctx, pool, store_reqs, n_store_req, store_chunks, n_store_chunks,
                           load_reqs, n_load_req, load_chunks, n_load_chunks, layer_begin,
                           layer_end, cfg, stream);
}

kvx_status kvx_roundtrip_chunks(kvx_ctx *ctx, const kvx_pool *pool,
                                const kvx_request *src_reqs, const kvx_request *dst_reqs,
                                int n_req, const kvx_chunk *chunks, int n_chunks,
                                int layer_begin, int layer_end, const kvx_launch_cfg *cfg,
                                kvx_stream_t stream)
{
    return launch_roundtrip(ctx, pool, src_reqs, dst_reqs, n_req, chunks, n_chunks, layer_begin,
                            layer_end, cfg, stream);
}

kvx_status kvx_test_roundtrip_timeout(kvx_ctx *ctx, const kvx_pool *pool,
                                      const kvx_request *src_reqs, const kvx_request *dst_reqs,
                                      int n_req, const kvx_chunk *chunks, int n_chunks,
                                      uint64_t wait_ns, kvx_stream_t stream)
{
    if (!ctx || !pool)
        return KVX_ERR_INVALID_ARG;
    if (wait_ns < 1000000ull || wait_ns > kWaitLimitNs)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "wait_ns %llu outside [1 ms, 1 s]",
                       (unsigned long long)wait_ns);
    return launch_roundtrip(ctx, pool, src_reqs, dst_reqs, n_req, chunks, n_chunks, 0,
                            pool->num_layers, nullptr, stream, wait_ns);
}

kvx_status kvx_transform_hbm(kvx_ctx *ctx, int dir, const kvx_pool *pool,
                             const kvx_request *reqs, int n_req, const kvx_chunk *chunks,
                             int n_chunks, int layer_begin, int layer_end,
                             const kvx_launch_cfg *cfg, kvx_stream_t stream)
{
    if (dir != KVX_DIR_GATHER && dir != KVX_DIR_SCATTER)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "transform direction %d", dir);
    return launch(ctx, dir == KVX_DIR_GATHER ? KVX_OP_GATHER_HBM : KVX_OP_SCATTER_HBM, pool,
                  reqs, n_req, chunks, n_chunks, layer_begin, layer_end, cfg, stream);
}

kvx_status kvx_dma_baseline(kvx_ctx *ctx, int dir, const kvx_pool *pool,
                            const kvx_request *reqs, int n_req, const kvx_chunk *chunks,
                            int n_chunks, int layer_begin, int layer_end, kvx_stream_t stream,
                            int64_t *n_copies)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    if (n_copies)
        *n_copies = 0;
    if (dir != KVX_DIR_GATHER && dir != KVX_DIR_SCATTER)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "baseline direction %d", dir);
    // Chunks may sit in host or device memory here, so the pointer-type checks of level 2
    // do not apply; sizes, ranges and alignment are checked as for the kernels.
    const int level = ctx->validation < 1 ? ctx->validation : 1;
    kvx_status st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                                  dir == KVX_DIR_GATHER ? KVX_OP_STORE : KVX_OP_LOAD, level,
                                  false, ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    for (int r = 0; r < n_req; ++r)
        if (reqs[r].n_tokens > 0 && !reqs[r].page_table_host)
            return set_err(ctx, KVX_ERR_INVALID_ARG,
                           "request %d: the DMA baseline needs page_table_host", r);
    DeviceGuard guard(ctx->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t v = pool->token_bytes;
    const int32_t P = pool->page_size;
    int64_t copies = 0;
    for (int c = 0; c < n_chunks; ++c) {
        const kvx_chunk &ch = chunks[c];
        const int32_t *pt = reqs[ch.request].page_table_host;
        int lo, hi;
        kvx::chunk_layers(ch, layer_begin, layer_end, &lo, &hi);
        if (lo >= hi || ch.n_tokens == 0)
            continue;
        const bool lm = ch.layout != KVX_CHUNK_TOKEN_MAJOR;
        int64_t slab_stride = lm ? int64_t(ch.n_tokens) * v : v;
        if (ch.layout == KVX_CHUNK_STRIPED)
            slab_stride =
                (slab_stride + KVX_STRIPE_ALIGN - 1) / KVX_STRIPE_ALIGN * KVX_STRIPE_ALIGN;
        const int64_t row_stride = lm ? v : int64_t(ch.n_layers) * pool->kv_factor * v;
        const int32_t t_end = ch.token_begin + ch.n_tokens;
        for (int l = lo; l < hi; ++l)
            for (int kv = 0; kv < pool->kv_factor; ++kv) {
                char *base = static_cast<char *>((kv == 0 ? pool->k_pages : pool->v_pages)[l]);
                const int64_t slab = int64_t(l - ch.layer_begin) * pool->kv_factor + kv;
                for (int32_t lp = ch.token_begin / P; lp * P < t_end; ++lp) {
                    const int32_t tb = lp * P > ch.token_begin ? lp * P : ch.token_begin;
                    const int32_t te = (lp + 1) * P < t_end ? (lp + 1) * P : t_end;
                    const int32_t page = pt[lp];
                    if (page < 0 || page >= pool->num_pages)
                        return set_err(ctx, KVX_ERR_PAGE_OUT_OF_RANGE, "page id %d", page);
                    char *pg = base + (int64_t(page) * P + (tb - lp * P)) * v;
                    char *ck = static_cast<char *>(ch.ptr) + slab * slab_stride +
                               int64_t(tb - ch.token_begin) * row_stride;
                    char *dst = dir == KVX_DIR_GATHER ? ck : pg;
                    const char *src = dir == KVX_DIR_GATHER ? pg : ck;
                    cudaError_t e;
                    if (row_stride == v)
                        e = cudaMemcpyAsync(dst, src, size_t(te - tb) * v, cudaMemcpyDefault, s);
                    else
                        e = cudaMemcpy2DAsync(dst, dir == KVX_DIR_GATHER ? row_stride : v, src,
                                              dir == KVX_DIR_GATHER ? v : row_stride, v,
                                              size_t(te - tb), cudaMemcpyDefault, s);
                    if (e != cudaSuccess)
                        return cuda_err(ctx, e, "baseline copy");
                    ++copies;
                }
            }
    }
    if (n_copies)
        *n_copies = copies;
    return KVX_OK;
}

kvx_status kvx_get_status(kvx_ctx *ctx, kvx_stream_t stream, uint32_t *flags)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    DeviceGuard guard(ctx->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(ctx->status_host, ctx->status_dev, sizeof(unsigned int),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(ctx->status_dev, 0, sizeof(unsigned int), s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "reading the device status");
    const uint32_t f = *ctx->status_host;
    if (flags)
        *flags = f;
    if (f)
        return set_err(ctx, KVX_ERR_DEVICE_STATUS, "device status 0x%x", f);
    return KVX_OK;
}

const char *kvx_last_error(const kvx_ctx *ctx) { return ctx ? ctx->err : ""; }

kvx_status kvx_last_launch(const kvx_ctx *ctx, int64_t *items, int32_t *ctas, int32_t *threads,
                           int64_t *descriptor_bytes)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    if (descriptor_bytes)
        *descriptor_bytes = ctx->last_desc_bytes;
    if (items)
        *items = ctx->last_items;
    if (ctas)
        *ctas = ctx->last_ctas;
    if (threads)
        *threads = ctx->last_threads;
    return KVX_OK;
}

kvx_status kvx_host_alloc(void **ptr, size_t bytes)
{
    if (!ptr || bytes == 0)
        return KVX_ERR_INVALID_ARG;
    cudaError_t e = cudaHostAlloc(ptr, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *ptr = nullptr;
        return KVX_ERR_CUDA;
    }
    return KVX_OK;
}

kvx_status kvx_host_free(void *ptr)
{
    if (!ptr)
        return KVX_OK;
    return cudaFreeHost(ptr) == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}

kvx_status kvx_host_register(void *ptr, size_t bytes)
{
    if (!ptr || bytes == 0)
        return KVX_ERR_INVALID_ARG;
    cudaError_t e =
        cudaHostRegister(ptr, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KVX_ERR_CUDA;
    }
    return KVX_OK;
}

kvx_status kvx_host_unregister(void *ptr)
{
    if (!ptr)
        return KVX_ERR_INVALID_ARG;
    return cudaHostUnregister(ptr) == cudaSuccess ? KVX_OK : KVX_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free load
//
// kvx_load_chunks_noalloc is kvx_load_chunks for callers that may not allocate device
// memory: a serving engine that hands nearly all of HBM to its KV page pool at start-up
// (a later cudaMalloc fails, or eats into pages the engine already promised), or a
// plug-in the engine calls with no place to keep a kvx_ctx between calls.  Its scratch
// -- the status word and the packed descriptors that kvx_create would otherwise allocate
// -- is the fixed array below.  Every GPU that loads this library holds that array until
// the process exits.

namespace {

const size_t kNoallocScratchBytes = KVX_NOALLOC_SCRATCH_BYTES;
const size_t kNoallocHeader = 256;  // status word, then zero padding
const int kNoallocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVX_NOALLOC_SCRATCH_BYTES];

// Host image of the scratch, filled under the mutex and copied from pageable memory:
// cudaMemcpyAsync returns only after it has consumed a pageable source, so the image can
// be refilled as soon as the copy call returns.
unsigned char g_noalloc_stage[KVX_NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kNoallocMaxDevices];  // device address of the array, per device

}  // namespace

extern "C" kvx_status kvx_load_chunks_noalloc(const kvx_pool *pool, const kvx_request *reqs,
                                              int n_req, const kvx_chunk *chunks, int n_chunks,
                                              int layer_begin, int layer_end,
                                              const kvx_launch_cfg *cfg, kvx_stream_t stream,
                                              uint32_t *device_flags)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The descriptor copy below reads a static host image that the next call overwrites; a
    // capturing stream would record that copy and replay whatever the image then holds.
    // Refuse it before doing anything.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) {
        cudaGetLastError();
        return KVX_ERR_CUDA;
    }
    if (capture != cudaStreamCaptureStatusNone)
        return KVX_ERR_INVALID_ARG;
    kvx_launch_cfg c;
    kvx_status st = resolve_cfg(nullptr, KVX_OP_LOAD, cfg, &c);
    if (st != KVX_OK)
        return st;
    if (c.mapping != KVX_MAP_WARP_SEGMENT || c.overlap)
        return KVX_ERR_INVALID_ARG;
    st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, KVX_OP_LOAD,
                       1, false, nullptr, 0);
    if (st != KVX_OK)
        return st;
    short_segment_grid(KVX_OP_LOAD, cfg, pool, &c);
    if (device_flags && (reinterpret_cast<uintptr_t>(device_flags) & 3u))
        return KVX_ERR_ALIGNMENT;
    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    if (kNoallocHeader + lay.total > kNoallocScratchBytes)
        return KVX_ERR_CAPACITY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) {
        cudaGetLastError();
        return KVX_ERR_CUDA;
    }
    // Launch-shape input only (no buffers, no stream): the device's SM count, so that the
    // same cfg gives the same launch as kvx_load_chunks.
    kvx_ctx shape_ctx;
    shape_ctx.device = dev;
    if (cudaDeviceGetAttribute(&shape_ctx.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
        return KVX_ERR_CUDA;

    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        // First call on this device, with it current: look up the array's device address.
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) {
            cudaGetLastError();
            return KVX_ERR_CUDA;
        }
        g_noalloc_addr[dev] = addr;
    }
    char *dev_block = static_cast<char *>(g_noalloc_addr[dev]);
    std::memset(g_noalloc_stage, 0, kNoallocHeader);  // the status word starts each call at 0
    Plan plan = kvx::pack(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                          KVX_DIR_SCATTER, lay,
                          reinterpret_cast<char *>(g_noalloc_stage) + kNoallocHeader,
                          dev_block + kNoallocHeader);
    plan.status = device_flags ? device_flags : reinterpret_cast<unsigned int *>(dev_block);
    apply_batch(KVX_OP_LOAD, c, &plan);
    choose_split(&shape_ctx, c, &plan);
    if (plan.total_items == 0)
        return KVX_OK;
    if (cudaMemcpyAsync(dev_block, g_noalloc_stage, kNoallocHeader + lay.total,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KVX_ERR_CUDA;
    if (launch_kernel(launch_shape(&shape_ctx, c, plan, KVX_DIR_SCATTER, false,
                                   use_rows(c, pool, chunks, n_chunks, false)),
                      plan, s) != cudaSuccess)
        return KVX_ERR_CUDA;
    return KVX_OK;
}
