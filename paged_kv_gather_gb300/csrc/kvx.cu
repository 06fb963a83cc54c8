// kvx.cu -- GB300 (sm_103a) kernels and C-ABI entry points of the paged KV gather/scatter
// library.
//
// One kernel family moves every byte.  A persistent grid of warps walks the batch's work
// items; an item is one (chunk, layer, kv, page) segment, contiguous on the page side
// ("Strata Guide: Hierarchical Context Caching for Long LLMs", section "Two-Dimensional
// Memory Layout Decoupling": the layout change is address arithmetic done by the moving
// thread, not a separate pass).  Each lane moves 16-byte units ("Step 1:
// High-Performance GPU-Assisted I/O CUDA Kernel": 128-bit vector accesses, a page-table
// lookup per unit of work, streaming stores into HBM), with `unroll` independent loads in
// flight per lane before its stores, because host-link reads need many bytes in flight
// (section "The Physics of I/O Bandwidth and Little's Law": X = C * S / L).  The grid is
// capped to a few SMs for host transfers so a concurrent compute stream keeps the rest
// (section "Non-Intrusive Resource Sizing"); the HBM-only transform uses every SM.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <vector>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kvx_internal.h"

using kvx::DevChunk;
using kvx::Plan;

// ------------------------------------------------------------------------------- device

namespace {

__device__ __forceinline__ uint4 ld_nc_v4(const uint4 *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Coherent 16-byte load, cached in L2 only: for bytes another warp of the same launch wrote
// (the read-only .nc path is valid only for data no thread writes during the launch).
__device__ __forceinline__ uint4 ld_cg_v4(const uint4 *p)
{
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

template <bool NC>
__device__ __forceinline__ uint4 ld_v4(const uint4 *p)
{
    return NC ? ld_nc_v4(p) : ld_cg_v4(p);
}

template <int HINT>
__device__ __forceinline__ void st_v4(uint4 *p, const uint4 &v)
{
    if (HINT == KVX_HINT_STREAMING)
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
    else
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
}

// Chunk owning `item`: the largest c with item_begin[c] <= item.  A 32-way search: each
// step the warp probes 32 evenly spaced entries and keeps the last one not above `item`,
// so 18k chunks take three coalesced probes.
__device__ __forceinline__ int find_chunk(const int64_t *__restrict__ begin, int n, int64_t item,
                                          int lane)
{
    int lo = 0, hi = n;  // begin[lo] <= item < begin[hi]
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int idx = lo + lane * step;
        const bool ok = idx < hi && __ldg(begin + idx) <= item;
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        lo += (31 - __clz(m)) * step;
        hi = min(hi, lo + step);
    }
    return lo;
}

// Contiguous copy of n16 16-byte units.  Lane i owns units i, i + 32, i + 64, ...; each
// pass issues U independent loads before its U stores.  NC = false reads through the
// coherent path.
template <int U, int HINT, bool NC = true>
__device__ __forceinline__ void copy_contig(const uint4 *__restrict__ s, uint4 *__restrict__ d,
                                            int n16, int lane)
{
    s += lane;
    d += lane;
    int rem = n16 - lane;  // units of this lane's stride left, scaled by 32
    for (; rem > 32 * (U - 1); rem -= 32 * U, s += 32 * U, d += 32 * U) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            r[u] = ld_v4<NC>(s + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            st_v4<HINT>(d + 32 * u, r[u]);
    }
    if (rem > 0) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (32 * u < rem)
                r[u] = ld_v4<NC>(s + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (32 * u < rem)
                st_v4<HINT>(d + 32 * u, r[u]);
    }
}

// One work item resolved to addresses: `rows` rows of row_bytes, contiguous on the page side
// (pitch = token_bytes) and contiguous or strided on the chunk side.
struct Segment {
    const char *src;
    char *dst;
    int64_t s_pitch;
    int64_t d_pitch;
    int32_t rows;
    bool contiguous;  // rows back to back on both sides: one run of rows * token_bytes
};

// Chunk owning `item` for one lane alone (plain binary search): used when every lane
// resolves a different item.
__device__ __forceinline__ int find_chunk_lane(const int64_t *__restrict__ begin, int n,
                                               int64_t item)
{
    int lo = 0, hi = n;  // begin[lo] <= item < begin[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(begin + mid) <= item)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Addresses of item `item` of chunk `c`.  Returns false, after flagging the device status
// when `flag` is set, if the page id is outside the pool; the segment is then skipped.
template <int DIR>
__device__ __forceinline__ bool segment_of(const Plan &p, int c, int64_t item, bool flag,
                                           Segment &sg)
{
    const int64_t v = p.token_bytes;
    const DevChunk &ch = p.chunks[c];
    const int64_t i = item - p.item_begin[c];
    const int32_t np = ch.np;
    const int32_t slab = int32_t(i / np);
    const int32_t j = int32_t(i - int64_t(slab) * np);
    const int32_t kv = p.kv_factor == 2 ? (slab & 1) : 0;
    const int32_t layer = ch.la + (p.kv_factor == 2 ? (slab >> 1) : slab);
    const int32_t lpage = ch.pf + j;
    const int32_t pt0 = lpage * p.page_size;
    const int32_t tb = max(ch.t0, pt0);
    const int32_t te = min(ch.t_end, pt0 + p.page_size);
    const int32_t page = p.reqs[ch.request].page_table[lpage];
    if (unsigned(page) >= unsigned(p.num_pages)) {
        if (flag)
            atomicOr(p.status, KVX_DEV_PAGE_OUT_OF_RANGE);
        return false;
    }
    char *pg = p.pools[kv * p.num_layers + layer] + (int64_t(page) * p.page_size + (tb - pt0)) * v;
    char *ck = ch.ptr + int64_t(ch.slab0 + slab) * ch.slab_stride +
               int64_t(tb - ch.t0) * ch.row_stride;
    sg.src = DIR == KVX_DIR_GATHER ? pg : ck;
    sg.dst = DIR == KVX_DIR_GATHER ? ck : pg;
    sg.s_pitch = DIR == KVX_DIR_GATHER ? v : ch.row_stride;
    sg.d_pitch = DIR == KVX_DIR_GATHER ? ch.row_stride : v;
    sg.rows = te - tb;
    sg.contiguous = ch.row_stride == v;
    return true;
}

// Resolve item -> segment (warp-collective: every lane of the warp calls it with the same
// item).
template <int DIR>
__device__ __forceinline__ bool resolve_segment(const Plan &p, int64_t item, int lane,
                                                Segment &sg)
{
    const int c = find_chunk(p.item_begin, p.n_chunks, item, lane);
    return segment_of<DIR>(p, c, item, lane == 0, sg);
}

__device__ __forceinline__ Segment shfl_segment(const Segment &s, int src_lane)
{
    Segment r;
    r.src = reinterpret_cast<const char *>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(s.src), src_lane));
    r.dst = reinterpret_cast<char *>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(s.dst), src_lane));
    r.s_pitch = __shfl_sync(0xffffffffu, s.s_pitch, src_lane);
    r.d_pitch = __shfl_sync(0xffffffffu, s.d_pitch, src_lane);
    r.rows = __shfl_sync(0xffffffffu, s.rows, src_lane);
    r.contiguous = __shfl_sync(0xffffffffu, int(s.contiguous), src_lane) != 0;
    return r;
}

template <int U, int HINT, bool NC = true>
__device__ __forceinline__ void copy_segment(const Segment &sg, int64_t v, int lane)
{
    if (sg.contiguous) {
        copy_contig<U, HINT, NC>(reinterpret_cast<const uint4 *>(sg.src),
                                 reinterpret_cast<uint4 *>(sg.dst),
                                 int((int64_t(sg.rows) * v) >> 4), lane);
    } else {
        // Token-major chunk: each token is its own run on the chunk side.
        for (int r = 0; r < sg.rows; ++r)
            copy_contig<1, HINT, NC>(reinterpret_cast<const uint4 *>(sg.src + r * sg.s_pitch),
                                     reinterpret_cast<uint4 *>(sg.dst + r * sg.d_pitch),
                                     int(v >> 4), lane);
    }
}

// Warp per page segment.  DIR = KVX_DIR_GATHER copies page -> chunk, KVX_DIR_SCATTER the
// reverse.  BATCHED = false: a warp resolves one segment at a time (32-way search), for
// page segments of 16 KiB and more.  BATCHED = true (short segments): each lane resolves
// one of p.batch consecutive segments in parallel and the warp then copies them back to
// back, so the lookup latency of short segments overlaps instead of adding up.
template <int U, int DIR, int HINT, bool BATCHED>
__device__ __forceinline__ void run_segments(const Plan &p, int64_t warp, int64_t n_warps,
                                             int lane)
{
    const int64_t v = p.token_bytes;
    if (!BATCHED) {
        for (int64_t item = warp; item < p.total_items; item += n_warps) {
            Segment sg;
            if (resolve_segment<DIR>(p, item, lane, sg))
                copy_segment<U, HINT>(sg, v, lane);
        }
    } else {
        const int B = p.batch;
        for (int64_t base = warp * B; base < p.total_items; base += n_warps * B) {
            const int64_t mine = base + lane;
            Segment sg;
            sg.src = nullptr;
            sg.dst = nullptr;
            sg.s_pitch = sg.d_pitch = 0;
            sg.rows = 0;
            sg.contiguous = true;
            bool ok = false;
            if (lane < B && mine < p.total_items)
                ok = segment_of<DIR>(p, find_chunk_lane(p.item_begin, p.n_chunks, mine), mine,
                                     true, sg);
            const unsigned valid = __ballot_sync(0xffffffffu, ok);
            for (int k = 0; k < B; ++k) {
                const Segment s = shfl_segment(sg, k);
                if (valid & (1u << k))
                    copy_segment<U, HINT>(s, v, lane);
            }
        }
    }
}

template <int U, int DIR, int HINT, bool BATCHED>
__global__ void __launch_bounds__(1024, 1) kvx_segment_kernel(const Plan p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    run_segments<U, DIR, HINT, BATCHED>(p, warp, n_warps, lane);
}

// Exchange: one launch moves a store batch (pages -> host chunks) and a load batch (host
// chunks -> pages) at once.  Even CTAs run the store plan, odd CTAs the load plan, so the
// block scheduler spreads both directions evenly over the SMs the launch gets instead of
// giving each direction its own contiguous block of SMs (two separate kernels), which
// lets the two directions of the host link run at full rate together.
template <int U, bool BATCHED_S, bool BATCHED_L>
__global__ void __launch_bounds__(1024, 1) kvx_exchange_kernel(const Plan ps, const Plan pl)
{
    const int lane = threadIdx.x & 31;
    const int64_t wpc = blockDim.x >> 5;
    const int64_t role_cta = blockIdx.x >> 1;
    const int64_t warp = role_cta * wpc + (threadIdx.x >> 5);
    if ((blockIdx.x & 1) == 0) {
        const int64_t ctas = (int64_t(gridDim.x) + 1) >> 1;
        run_segments<U, KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED_S>(ps, warp, ctas * wpc, lane);
    } else {
        const int64_t ctas = int64_t(gridDim.x) >> 1;
        run_segments<U, KVX_DIR_SCATTER, KVX_HINT_STREAMING, BATCHED_L>(pl, warp, ctas * wpc,
                                                                        lane);
    }
}

// ------------------------------------------------------------------ bulk-copy (TMA) mapping
//
// One warp per CTA streams its items through a ring of shared-memory stages with the
// Blackwell bulk-copy engine: cp.async.bulk global -> shared completes on an mbarrier
// (transaction bytes), then cp.async.bulk shared -> global (bulk group) writes the stage
// out.  Up to n_stages - 1 loads are in flight per CTA without holding them in registers,
// and the SM's load/store pipes stay free for other work.  Every wait is bounded: past
// about one second the kernel flags KVX_DEV_WAIT_TIMEOUT, drains what it issued and exits.

constexpr int kBulkMaxStages = 8;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Warp-uniform bounded wait for the completion of phase `parity` of an mbarrier.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int lane)
{
    const uint32_t addr = smem_u32(bar);
    const uint64_t deadline = global_ns() + kWaitLimitNs;
    while (true) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(addr), "r"(parity)
                     : "memory");
        if (__any_sync(0xffffffffu, done))
            return true;
        const int late = lane == 0 ? int(global_ns() > deadline) : 0;
        if (__shfl_sync(0xffffffffu, late, 0))
            return false;
    }
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                 "[%0], [%1], %2, [%3];" ::"r"(smem_u32(smem_dst)),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int DIR>
__global__ void __launch_bounds__(32) kvx_bulk_kernel(const Plan p, int stage_bytes,
                                                     int n_stages)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kBulkMaxStages];
    __shared__ char *stage_dst[kBulkMaxStages];
    __shared__ uint32_t stage_len[kBulkMaxStages];
    const int lane = threadIdx.x;
    const int64_t v = p.token_bytes;
    if (lane == 0) {
        for (int st = 0; st < n_stages; ++st)
            mbar_init(&full[st], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // Piece stream: items of this CTA, cut into runs of at most stage_bytes.
    int64_t item = blockIdx.x;
    Segment sg;
    bool have = false;
    int32_t row = 0, n_rows = 0;
    int64_t off = 0, row_bytes = 0;
    auto next = [&](const char *&src, char *&dst, uint32_t &bytes) -> bool {
        while (true) {
            if (have) {
                if (off < row_bytes) {
                    const int64_t b = min(int64_t(stage_bytes), row_bytes - off);
                    src = sg.src + row * sg.s_pitch + off;
                    dst = sg.dst + row * sg.d_pitch + off;
                    bytes = uint32_t(b);
                    off += b;
                    return true;
                }
                off = 0;
                if (++row < n_rows)
                    continue;
                have = false;
            }
            if (item >= p.total_items)
                return false;
            if (resolve_segment<DIR>(p, item, lane, sg)) {
                have = true;
                row = 0;
                off = 0;
                n_rows = sg.contiguous ? 1 : sg.rows;
                row_bytes = sg.contiguous ? int64_t(sg.rows) * v : v;
            }
            item += gridDim.x;
        }
    };

    uint32_t issued = 0, retired = 0;
    bool more = true, timed_out = false;
    const char *src = nullptr;
    char *dst = nullptr;
    uint32_t bytes = 0;
    auto issue = [&]() {
        const uint32_t st = issued % n_stages;
        if (lane == 0) {
            stage_dst[st] = dst;
            stage_len[st] = bytes;
            mbar_expect_tx(&full[st], bytes);
            bulk_load(ring + size_t(st) * stage_bytes, src, bytes, &full[st]);
        }
        ++issued;
    };
    while (issued + 1 < uint32_t(n_stages)) {
        if (!next(src, dst, bytes)) {
            more = false;
            break;
        }
        issue();
    }
    while (retired < issued) {
        const uint32_t st = retired % n_stages;
        if (!mbar_wait(&full[st], (retired / n_stages) & 1u, lane)) {
            timed_out = true;
            break;
        }
        if (lane == 0)
            bulk_store(stage_dst[st], ring + size_t(st) * stage_bytes, stage_len[st]);
        ++retired;
        if (more) {
            if (!next(src, dst, bytes)) {
                more = false;
            } else {
                // The stage about to be refilled was last written out by the store issued
                // one iteration ago: wait until at most the newest store still reads.
                if (lane == 0)
                    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                __syncwarp();
                issue();
            }
        }
    }
    if (timed_out) {
        if (lane == 0)
            atomicOr(p.status, KVX_DEV_WAIT_TIMEOUT);
        for (uint32_t r = retired; r < issued; ++r)  // drain the loads still in flight
            mbar_wait(&full[r % n_stages], (r / n_stages) & 1u, lane);
    }
    if (lane == 0)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

// ------------------------------------------------------------------------- round trip
//
// Store a batch to host chunks and load the same chunks into other pages in one launch
// (a swap-out followed by a swap-in elsewhere).  The store and load plans enumerate the
// same items, so load unit u reads exactly the host bytes store unit u writes.  Units
// (unit_items consecutive items) are handed out by two fetch-and-add counters, one per
// direction.  A warp takes a store unit while the loads handed out are within `lag`
// units (one per warp of the grid by default) of the stores handed out, and a load unit
// otherwise,
// so each load usually starts well after its store finished.  A warp that holds a load
// unit whose store has not been handed out yet hands out (and does) store units until it
// has; only then does it wait for that store.  Every wait is therefore on a unit held by a
// running warp that waits on nothing, whatever the residency of the grid, so the waits
// end; each is still bounded (about one second, then KVX_DEV_WAIT_TIMEOUT and the unit is
// skipped).  Both directions of the host link run from the first completed store to the
// last load, in a single launch.

struct RoundTripSync {
    unsigned int *next;  // [0] next store unit, [1] next load unit; zero at launch
    unsigned int *done;  // [units]: 1 once the store unit's bytes are in host memory
    int64_t units;
    int unit_items;
    unsigned lag;        // loads handed out may trail stores handed out by this many units
};

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Lane 0: bounded wait for a store unit to finish.
__device__ __forceinline__ bool wait_unit(const RoundTripSync &sy, int64_t unit)
{
    const uint64_t deadline = global_ns() + kWaitLimitNs;
    while (ld_acquire_u32(sy.done + unit) == 0u) {
        if (global_ns() > deadline)
            return false;
        __nanosleep(200);
    }
    return true;
}

enum : int { kUnitStore = 1, kUnitLoad = 2, kUnitSkip = 3 };

// Lane 0: the warp's next unit (-1: nothing left for this warp) and what to do with it.
// `pending` carries a load unit taken before its store was handed out.
__device__ __forceinline__ long long next_unit(const RoundTripSync &sy, unsigned lag,
                                               long long &pending, int &what)
{
    const unsigned n = unsigned(sy.units);
    if (pending < 0) {
        const unsigned si = ld_relaxed_u32(sy.next);
        const unsigned li = ld_relaxed_u32(sy.next + 1);
        if (si < n && li + lag >= si) {
            const unsigned s = atomicAdd(sy.next, 1u);
            if (s < n) {
                what = kUnitStore;
                return s;
            }
        }
        const unsigned t = atomicAdd(sy.next + 1, 1u);
        if (t >= n)
            return -1;  // every load is handed out; their holders finish the stores
        pending = t;
    }
    if (ld_relaxed_u32(sy.next) <= unsigned(pending)) {
        // The store this load needs is not handed out yet: hand out the next one.
        const unsigned s = atomicAdd(sy.next, 1u);
        if (s < n) {
            what = kUnitStore;
            return s;
        }
    }
    const long long u = pending;
    pending = -1;
    what = wait_unit(sy, u) ? kUnitLoad : kUnitSkip;
    return u;
}

// Items [first, first + count) of plan p, warp-collective (count is 1 unless BATCHED).
// NC = false for bytes written earlier in the same launch.
template <int U, int DIR, int HINT, bool BATCHED, bool NC>
__device__ __forceinline__ void copy_items(const Plan &p, int64_t first, int count, int lane)
{
    const int64_t v = p.token_bytes;
    if (!BATCHED) {  // one item per unit
        Segment sg;
        if (resolve_segment<DIR>(p, first, lane, sg))
            copy_segment<U, HINT, NC>(sg, v, lane);
        return;
    }
    Segment sg;
    sg.src = nullptr;
    sg.dst = nullptr;
    sg.s_pitch = sg.d_pitch = 0;
    sg.rows = 0;
    sg.contiguous = true;
    bool ok = false;
    if (lane < count) {
        const int64_t mine = first + lane;
        ok = segment_of<DIR>(p, find_chunk_lane(p.item_begin, p.n_chunks, mine), mine, true,
                             sg);
    }
    const unsigned valid = __ballot_sync(0xffffffffu, ok);
    for (int k = 0; k < count; ++k) {
        const Segment sk = shfl_segment(sg, k);
        if (valid & (1u << k))
            copy_segment<U, HINT, NC>(sk, v, lane);
    }
}

template <int U, bool BATCHED>
__global__ void __launch_bounds__(1024, 1)
    kvx_roundtrip_kernel(const Plan ps, const Plan pl, const RoundTripSync sy)
{
    const int lane = threadIdx.x & 31;
    long long pending = -1;  // lane 0's
    for (;;) {
        long long unit = -1;
        int what = 0;
        if (lane == 0) {
            unit = next_unit(sy, sy.lag, pending, what);
            if (what == kUnitSkip)
                atomicOr(ps.status, KVX_DEV_WAIT_TIMEOUT);
        }
        unit = __shfl_sync(0xffffffffu, unit, 0);
        what = __shfl_sync(0xffffffffu, what, 0);
        if (unit < 0)
            break;
        if (what == kUnitSkip)
            continue;  // its store never finished: leave the unit alone
        __syncwarp();  // lane 0's acquire orders every lane's loads below
        const int64_t first = unit * sy.unit_items;
        const int count = int(min(int64_t(sy.unit_items), ps.total_items - first));
        if (what == kUnitLoad) {
            copy_items<U, KVX_DIR_SCATTER, KVX_HINT_STREAMING, BATCHED, false>(pl, first, count,
                                                                             lane);
        } else {
            // HBM reads need fewer bytes in flight than host reads: four loads per lane.
            copy_items<(U > 4 ? 4 : U), KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED, true>(
                ps, first, count, lane);
            __syncwarp();  // every lane's writes happen before lane 0's release
            if (lane == 0)
                st_release_u32(sy.done + unit, 1u);
        }
    }
}

// Exchange with shared work: a store batch and an independent load batch, each warp taking
// its next unit from whichever direction is further behind in proportion to its size, so
// both directions finish together and every warp works until the last unit, whatever the
// ratio of the two batches.  No unit waits on another.
struct DuplexSync {
    unsigned int *next;  // [0] next store unit, [1] next load unit; zero at launch
    int64_t units_s;
    int64_t units_l;
    int unit_items;
};

// Lane 0: the next unit (-1: none left) and its direction.
__device__ __forceinline__ long long next_duplex_unit(const DuplexSync &sy, int &what)
{
    const unsigned ns = unsigned(sy.units_s), nl = unsigned(sy.units_l);
    const unsigned si = ld_relaxed_u32(sy.next);
    const unsigned li = ld_relaxed_u32(sy.next + 1);
    // store progress si / ns against load progress li / nl
    const bool store_first = si < ns && (li >= nl || uint64_t(si) * nl <= uint64_t(li) * ns);
    for (int attempt = 0; attempt < 2; ++attempt) {
        const bool store = (attempt == 0) == store_first;
        const unsigned u = atomicAdd(sy.next + (store ? 0 : 1), 1u);
        if (u < (store ? ns : nl)) {
            what = store ? kUnitStore : kUnitLoad;
            return u;
        }
    }
    return -1;
}

template <int U, bool BATCHED>
__global__ void __launch_bounds__(1024, 1)
    kvx_duplex_kernel(const Plan ps, const Plan pl, const DuplexSync sy)
{
    const int lane = threadIdx.x & 31;
    for (;;) {
        long long unit = -1;
        int what = 0;
        if (lane == 0)
            unit = next_duplex_unit(sy, what);
        unit = __shfl_sync(0xffffffffu, unit, 0);
        what = __shfl_sync(0xffffffffu, what, 0);
        if (unit < 0)
            break;
        const int64_t first = unit * sy.unit_items;
        if (what == kUnitLoad) {
            const int count = int(min(int64_t(sy.unit_items), pl.total_items - first));
            copy_items<U, KVX_DIR_SCATTER, KVX_HINT_STREAMING, BATCHED, true>(pl, first, count,
                                                                            lane);
        } else {
            const int count = int(min(int64_t(sy.unit_items), ps.total_items - first));
            copy_items<(U > 4 ? 4 : U), KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED, true>(
                ps, first, count, lane);
        }
    }
}

typedef void (*DuplexFn)(Plan, Plan, DuplexSync);

DuplexFn pick_duplex(int unroll, bool batched)
{
    switch (unroll) {
    case 1: return batched ? kvx_duplex_kernel<1, true> : kvx_duplex_kernel<1, false>;
    case 2: return batched ? kvx_duplex_kernel<2, true> : kvx_duplex_kernel<2, false>;
    case 4: return batched ? kvx_duplex_kernel<4, true> : kvx_duplex_kernel<4, false>;
    case 8: return batched ? kvx_duplex_kernel<8, true> : kvx_duplex_kernel<8, false>;
    }
    return nullptr;
}

typedef void (*RoundTripFn)(Plan, Plan, RoundTripSync);

RoundTripFn pick_roundtrip(int unroll, bool batched)
{
    switch (unroll) {
    case 1: return batched ? kvx_roundtrip_kernel<1, true> : kvx_roundtrip_kernel<1, false>;
    case 2: return batched ? kvx_roundtrip_kernel<2, true> : kvx_roundtrip_kernel<2, false>;
    case 4: return batched ? kvx_roundtrip_kernel<4, true> : kvx_roundtrip_kernel<4, false>;
    case 8: return batched ? kvx_roundtrip_kernel<8, true> : kvx_roundtrip_kernel<8, false>;
    }
    return nullptr;
}

typedef void (*KernelFn)(Plan);

template <int U, bool BATCHED>
KernelFn pick_hint_dir(int dir, int hint)
{
    if (dir == KVX_DIR_GATHER)
        return hint == KVX_HINT_STREAMING ? kvx_segment_kernel<U, KVX_DIR_GATHER, 1, BATCHED>
                                          : kvx_segment_kernel<U, KVX_DIR_GATHER, 0, BATCHED>;
    return hint == KVX_HINT_STREAMING ? kvx_segment_kernel<U, KVX_DIR_SCATTER, 1, BATCHED>
                                      : kvx_segment_kernel<U, KVX_DIR_SCATTER, 0, BATCHED>;
}

template <bool BATCHED>
KernelFn pick_unroll(int unroll, int dir, int hint)
{
    switch (unroll) {
    case 1: return pick_hint_dir<1, BATCHED>(dir, hint);
    case 2: return pick_hint_dir<2, BATCHED>(dir, hint);
    case 4: return pick_hint_dir<4, BATCHED>(dir, hint);
    case 8: return pick_hint_dir<8, BATCHED>(dir, hint);
    }
    return nullptr;
}

// The warp-segment kernel for (unroll, direction, hint), batched when more than one
// segment is resolved per warp at once.
KernelFn pick_kernel(int unroll, int dir, int hint, int batch = 1)
{
    return batch > 1 ? pick_unroll<true>(unroll, dir, hint)
                     : pick_unroll<false>(unroll, dir, hint);
}

typedef void (*ExchangeFn)(Plan, Plan);

template <int U>
ExchangeFn pick_exchange_u(bool bs, bool bl)
{
    if (bs)
        return bl ? kvx_exchange_kernel<U, true, true> : kvx_exchange_kernel<U, true, false>;
    return bl ? kvx_exchange_kernel<U, false, true> : kvx_exchange_kernel<U, false, false>;
}

ExchangeFn pick_exchange(int unroll, int batch_s, int batch_l)
{
    switch (unroll) {
    case 1: return pick_exchange_u<1>(batch_s > 1, batch_l > 1);
    case 2: return pick_exchange_u<2>(batch_s > 1, batch_l > 1);
    case 4: return pick_exchange_u<4>(batch_s > 1, batch_l > 1);
    case 8: return pick_exchange_u<8>(batch_s > 1, batch_l > 1);
    }
    return nullptr;
}

}  // namespace

// --------------------------------------------------------------------------------- host

namespace {

const int kSlots = 4;
const size_t kDefaultDescriptorBytes = 8u << 20;
const int kDefaultStageBytes = 32 << 10;
const int kDefaultStages = 6;
const int64_t kMaxBulkSmem = 220 << 10;

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
cudaError_t stage(kvx_ctx *ctx, Slot &slot, size_t bytes, size_t zero_off, size_t zero_bytes,
                  cudaStream_t s)
{
    cudaError_t e = cudaMemcpyAsync(slot.dev, slot.host, bytes, cudaMemcpyHostToDevice,
                                    ctx->copy_stream);
    if (e == cudaSuccess && zero_bytes)
        e = cudaMemsetAsync(slot.dev + zero_off, 0, zero_bytes, ctx->copy_stream);
    if (e == cudaSuccess)
        e = cudaEventRecord(slot.staged, ctx->copy_stream);
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
    switch (op) {
    case KVX_OP_STORE:
        c->sm_cap = 16;
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
    default:  // HBM transform: the whole GPU, two 256-thread CTAs per SM, 8 loads in flight
        c->sm_cap = 0;
        c->ctas_per_sm = 2;
        c->threads = 256;
        c->unroll = 8;
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
    bool ok = out->sm_cap >= 0 && out->ctas_per_sm >= 1 && out->ctas_per_sm <= 32 &&
              out->batch >= 0 && out->batch <= 32 &&
              (out->store_hint == KVX_HINT_DEFAULT || out->store_hint == KVX_HINT_STREAMING);
    if (out->mapping == KVX_MAP_WARP_SEGMENT) {
        ok = ok && out->threads >= 32 && out->threads <= 1024 && out->threads % 32 == 0 &&
             pick_kernel(out->unroll, 0, 0);
    } else if (out->mapping == KVX_MAP_BULK) {
        // One warp per CTA; `unroll` counts shared-memory stages.
        if (!user->unroll)
            out->unroll = kDefaultStages;
        out->threads = 32;
        ok = ok && out->unroll >= 2 && out->unroll <= kBulkMaxStages &&
             out->stage_bytes >= 16 && out->stage_bytes % 16 == 0 &&
             int64_t(out->unroll) * out->stage_bytes <= kMaxBulkSmem;
    } else {
        ok = false;
    }
    if (!ok)
        return set_err(ctx, KVX_ERR_INVALID_ARG,
                       "launch cfg: sm_cap %d ctas_per_sm %d threads %d unroll %d hint %d "
                       "mapping %d stage_bytes %d batch %d", user->sm_cap, user->ctas_per_sm,
                       user->threads, user->unroll, user->store_hint, user->mapping,
                       user->stage_bytes, user->batch);
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
};

LaunchShape launch_shape(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &plan, int dir)
{
    LaunchShape sh;
    const int64_t warps_per_cta = cfg.threads / 32;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    int64_t ctas = int64_t(sms) * cfg.ctas_per_sm;
    const int64_t per_cta = warps_per_cta * (cfg.mapping == KVX_MAP_BULK ? 1 : plan.batch);
    const int64_t needed = (plan.total_items + per_cta - 1) / per_cta;
    if (ctas > needed)
        ctas = needed;
    sh.ctas = ctas;
    if (cfg.mapping == KVX_MAP_BULK) {
        sh.fn = dir == KVX_DIR_GATHER
                    ? reinterpret_cast<const void *>(kvx_bulk_kernel<KVX_DIR_GATHER>)
                    : reinterpret_cast<const void *>(kvx_bulk_kernel<KVX_DIR_SCATTER>);
        sh.threads = 32;
        sh.bulk = 1;
        sh.stage_bytes = cfg.stage_bytes;
        sh.stages = cfg.unroll;
        sh.smem = size_t(cfg.unroll) * cfg.stage_bytes;
    } else {
        sh.fn = reinterpret_cast<const void *>(pick_kernel(cfg.unroll, dir, cfg.store_hint,
                                                           plan.batch));
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
        return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(32u), args, sh.smem, s);
    }
    void *args[] = {&plan};
    return cudaLaunchKernel(sh.fn, dim3(unsigned(sh.ctas)), dim3(unsigned(sh.threads)), args, 0,
                            s);
}

kvx_status launch(kvx_ctx *ctx, int op, const kvx_pool *pool, const kvx_request *reqs, int n_req,
                  const kvx_chunk *chunks, int n_chunks, int layer_begin, int layer_end,
                  const kvx_launch_cfg *user_cfg, kvx_stream_t stream)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    ctx->last_items = 0;
    ctx->last_ctas = 0;
    ctx->last_threads = 0;
    ctx->last_desc_bytes = 0;
    kvx_launch_cfg cfg;
    kvx_status st = resolve_cfg(ctx, op, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, op,
                       ctx->validation, true, ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);

    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    if (lay.total > ctx->slot_bytes)
        return set_err(ctx, KVX_ERR_CAPACITY,
                       "descriptors need %zu bytes, the context holds %zu per call; create it "
                       "with a larger max_descriptor_bytes", lay.total, ctx->slot_bytes);
    Slot &slot = ctx->slots[ctx->next];
    if (slot.used) {
        cudaError_t e = cudaEventSynchronize(slot.done);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "waiting for a descriptor buffer");
    }
    const int dir = (op == KVX_OP_LOAD || op == KVX_OP_SCATTER_HBM) ? KVX_DIR_SCATTER
                                                                    : KVX_DIR_GATHER;
    Plan plan = kvx::pack(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, dir, lay,
                          slot.host, slot.dev);
    plan.status = ctx->status_dev;
    if (cfg.batch > 0)
        plan.batch = cfg.batch;
    else if ((op == KVX_OP_GATHER_HBM || op == KVX_OP_SCATTER_HBM) && plan.batch == 1)
        plan.batch = 2;  // HBM transform: overlap the lookup of two long segments per warp
    if (plan.total_items == 0)
        return KVX_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = stage(ctx, slot, lay.total, 0, 0, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "descriptor copy");
    const LaunchShape shape = launch_shape(ctx, cfg, plan, dir);
    e = launch_kernel(shape, plan, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "kernel launch");
    const int64_t ctas = shape.ctas;
    e = cudaEventRecord(slot.done, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "event record");
    slot.used = true;
    ctx->next = (ctx->next + 1) % kSlots;
    ctx->last_items = plan.total_items;
    ctx->last_ctas = int32_t(ctas);
    ctx->last_threads = cfg.threads;
    ctx->last_desc_bytes = int64_t(lay.total);
    return KVX_OK;
}

// An exchange whose batches differ in size by more than this factor (in segments) shares its
// units between all warps (kvx_duplex_kernel): with the role split the smaller batch's half
// of the grid would finish early and leave the larger batch on half the CTAs.  Batches of
// similar size keep the role split, which measured 2-5 % faster for them.
constexpr double kExchangeShareRatio = 1.5;

bool exchange_shared(const Plan &ps, const Plan &pl)
{
    const double a = double(ps.total_items), b = double(pl.total_items);
    return a > kExchangeShareRatio * b || b > kExchangeShareRatio * a;
}

// Work counters and grid of a shared exchange; `next` is a zeroed 256-byte device word.
bool duplex_setup(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &ps, const Plan &pl,
                  unsigned *next, DuplexSync *sy, LaunchShape *sh)
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
    sh->fn = reinterpret_cast<const void *>(pick_duplex(cfg.unroll, ps.batch > 1));
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
                           const Plan &pl)
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
    sh.fn = reinterpret_cast<const void *>(pick_exchange(cfg.unroll, ps.batch, pl.batch));
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
    ctx->last_items = 0;
    ctx->last_ctas = 0;
    ctx->last_threads = 0;
    ctx->last_desc_bytes = 0;
    kvx_launch_cfg cfg;
    kvx_status st = resolve_cfg(ctx, KVX_OP_EXCHANGE, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    if (cfg.mapping != KVX_MAP_WARP_SEGMENT)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "exchange runs the warp-segment mapping only");
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
    if (total > ctx->slot_bytes)
        return set_err(ctx, KVX_ERR_CAPACITY,
                       "descriptors need %zu bytes, the context holds %zu per call; create it "
                       "with a larger max_descriptor_bytes", total, ctx->slot_bytes);
    Slot &slot = ctx->slots[ctx->next];
    if (slot.used) {
        cudaError_t e = cudaEventSynchronize(slot.done);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "waiting for a descriptor buffer");
    }
    Plan ps = kvx::pack(pool, sreqs, n_sreq, schunks, n_schunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, ls, slot.host, slot.dev);
    Plan pl = kvx::pack(pool, lreqs, n_lreq, lchunks, n_lchunks, layer_begin, layer_end,
                        KVX_DIR_SCATTER, ll, slot.host + ls.total, slot.dev + ls.total);
    ps.status = pl.status = ctx->status_dev;
    if (cfg.batch > 0)
        ps.batch = pl.batch = cfg.batch;
    if (ps.total_items + pl.total_items == 0)
        return KVX_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    int64_t ctas;
    if (exchange_shared(ps, pl)) {
        if (total + 256 > ctx->slot_bytes)
            return set_err(ctx, KVX_ERR_CAPACITY, "descriptors need %zu bytes, the context "
                           "holds %zu per call", total + 256, ctx->slot_bytes);
        DuplexSync sy;
        LaunchShape shape;
        if (!duplex_setup(ctx, cfg, ps, pl, reinterpret_cast<unsigned *>(slot.dev + total), &sy,
                          &shape))
            return set_err(ctx, KVX_ERR_CAPACITY, "exchange batches of %lld and %lld segments "
                           "(%d and %d per warp) do not fit one shared launch",
                           (long long)ps.total_items, (long long)pl.total_items, ps.batch,
                           pl.batch);
        e = stage(ctx, slot, total, total, 256, s);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "descriptor copy");
        e = launch_duplex_kernel(shape, ps, pl, sy, s);
        ctas = shape.ctas;
    } else {
        e = stage(ctx, slot, total, 0, 0, s);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "descriptor copy");
        const LaunchShape shape = exchange_shape(ctx, cfg, ps, pl);
        e = launch_exchange_kernel(shape, ps, pl, s);
        ctas = shape.ctas;
    }
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "kernel launch");
    e = cudaEventRecord(slot.done, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "event record");
    slot.used = true;
    ctx->next = (ctx->next + 1) % kSlots;
    ctx->last_items = ps.total_items + pl.total_items;
    ctx->last_ctas = int32_t(ctas);
    ctx->last_threads = cfg.threads;
    ctx->last_desc_bytes = int64_t(total);
    return KVX_OK;
}

// Units, lag and grid of a round trip whose work counters and completion words start at
// `sync` (sync_bytes(), zeroed before each launch).
void roundtrip_setup(const kvx_ctx *ctx, const kvx_launch_cfg &cfg, const Plan &ps, char *sync,
                     RoundTripSync *sy, LaunchShape *sh)
{
    sy->unit_items = ps.batch;
    sy->units = (ps.total_items + sy->unit_items - 1) / sy->unit_items;
    sy->next = reinterpret_cast<unsigned *>(sync);
    sy->done = reinterpret_cast<unsigned *>(sync + 256);
    const int64_t warps_per_cta = cfg.threads / 32;
    const int sms = cfg.sm_cap > 0 ? cfg.sm_cap : ctx->num_sms;
    int64_t ctas = int64_t(sms) * cfg.ctas_per_sm;
    const int64_t needed = (2 * sy->units + warps_per_cta - 1) / warps_per_cta;
    if (ctas > needed)
        ctas = needed;
    sy->lag = unsigned(ctas * warps_per_cta);  // one unit per warp of the grid
    sh->ctas = ctas;
    sh->threads = cfg.threads;
    sh->fn = reinterpret_cast<const void *>(pick_roundtrip(cfg.unroll, ps.batch > 1));
}

size_t roundtrip_sync_bytes(const Plan &ps)
{
    const int64_t units = (ps.total_items + ps.batch - 1) / ps.batch;
    return 256 + sizeof(unsigned) * size_t(units);
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
kvx_status launch_roundtrip(kvx_ctx *ctx, const kvx_pool *pool, const kvx_request *src_reqs,
                            const kvx_request *dst_reqs, int n_req, const kvx_chunk *chunks,
                            int n_chunks, int layer_begin, int layer_end,
                            const kvx_launch_cfg *user_cfg, kvx_stream_t stream)
{
    if (!ctx)
        return KVX_ERR_INVALID_ARG;
    ctx->last_items = 0;
    ctx->last_ctas = 0;
    ctx->last_threads = 0;
    ctx->last_desc_bytes = 0;
    kvx_launch_cfg cfg;
    kvx_status st = resolve_cfg(ctx, KVX_OP_ROUNDTRIP, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    if (cfg.mapping != KVX_MAP_WARP_SEGMENT)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "round trip runs the warp-segment mapping only");
    st = kvx::validate_exchange(pool, src_reqs, n_req, chunks, n_chunks, dst_reqs, n_req, chunks,
                                n_chunks, layer_begin, layer_end, ctx->validation, true,
                                ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const kvx::PackedLayout lay = kvx::packed_layout(pool, n_req, n_chunks);
    // Units from the packed item count (known after packing); bound the sync area first by
    // the largest count the slot could describe.
    Slot &slot = ctx->slots[ctx->next];
    if (2 * lay.total + 256 > ctx->slot_bytes)
        return set_err(ctx, KVX_ERR_CAPACITY,
                       "descriptors need %zu bytes, the context holds %zu per call; create it "
                       "with a larger max_descriptor_bytes", 2 * lay.total + 256,
                       ctx->slot_bytes);
    if (slot.used) {
        cudaError_t e = cudaEventSynchronize(slot.done);
        if (e != cudaSuccess)
            return cuda_err(ctx, e, "waiting for a descriptor buffer");
    }
    Plan ps = kvx::pack(pool, src_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_GATHER, lay, slot.host, slot.dev);
    Plan pl = kvx::pack(pool, dst_reqs, n_req, chunks, n_chunks, layer_begin, layer_end,
                        KVX_DIR_SCATTER, lay, slot.host + lay.total, slot.dev + lay.total);
    ps.status = pl.status = ctx->status_dev;
    if (cfg.batch > 0)
        ps.batch = pl.batch = cfg.batch;
    if (ps.total_items == 0)
        return KVX_OK;
    const size_t sync_off = 2 * lay.total;
    const size_t sync_bytes = roundtrip_sync_bytes(ps);
    if (sync_bytes > (size_t(1) << 33) || sync_off + sync_bytes > ctx->slot_bytes)
        return set_err(ctx, KVX_ERR_CAPACITY,
                       "round trip of %lld segments needs %zu bytes of descriptors and "
                       "completion words, the context holds %zu per call",
                       (long long)ps.total_items, sync_off + sync_bytes, ctx->slot_bytes);
    RoundTripSync sy;
    LaunchShape shape;
    roundtrip_setup(ctx, cfg, ps, slot.dev + sync_off, &sy, &shape);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = stage(ctx, slot, sync_off, sync_off, sync_bytes, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "descriptor copy");
    e = launch_roundtrip_kernel(shape, ps, pl, sy, 0, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "kernel launch");
    const int64_t ctas = shape.ctas;
    e = cudaEventRecord(slot.done, s);
    if (e != cudaSuccess)
        return cuda_err(ctx, e, "event record");
    slot.used = true;
    ctx->next = (ctx->next + 1) % kSlots;
    ctx->last_items = 2 * ps.total_items;
    ctx->last_ctas = int32_t(ctas);
    ctx->last_threads = cfg.threads;
    ctx->last_desc_bytes = int64_t(sync_off);
    return KVX_OK;
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
    DeviceGuard guard(ctx->device);
    if (!guard.ok)
        return set_err(ctx, KVX_ERR_CUDA, "cannot make device %d current", ctx->device);
    const int dir = (op == KVX_OP_LOAD || op == KVX_OP_SCATTER_HBM) ? KVX_DIR_SCATTER
                                                                    : KVX_DIR_GATHER;
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
    if (cfg.batch > 0)
        p->plan.batch = cfg.batch;
    else if ((op == KVX_OP_GATHER_HBM || op == KVX_OP_SCATTER_HBM) && p->plan.batch == 1)
        p->plan.batch = 2;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(p->dev, host.data(), lay.total, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);  // the host image dies with this call
    if (e != cudaSuccess) {
        cudaFree(p->dev);
        delete p;
        return cuda_err(ctx, e, "plan descriptor copy");
    }
    p->shape = launch_shape(ctx, cfg, p->plan, dir);
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
    kvx_status st = resolve_cfg(ctx, KVX_OP_EXCHANGE, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    if (cfg.mapping != KVX_MAP_WARP_SEGMENT)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "exchange runs the warp-segment mapping only");
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
    if (cfg.batch > 0)
        p->plan.batch = p->load.batch = cfg.batch;
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
    if (!p->shared) {
        p->shape = exchange_shape(ctx, cfg, p->plan, p->load);
    } else if (!duplex_setup(ctx, cfg, p->plan, p->load,
                             reinterpret_cast<unsigned *>(p->dev + total), &p->sync, &p->shape)) {
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
    kvx_status st = resolve_cfg(ctx, KVX_OP_ROUNDTRIP, user_cfg, &cfg);
    if (st != KVX_OK)
        return st;
    if (cfg.mapping != KVX_MAP_WARP_SEGMENT)
        return set_err(ctx, KVX_ERR_INVALID_ARG, "round trip runs the warp-segment mapping only");
    st = kvx::validate_exchange(pool, src_reqs, n_req, chunks, n_chunks, dst_reqs, n_req, chunks,
                                n_chunks, layer_begin, layer_end, ctx->validation, true,
                                ctx->err, sizeof ctx->err);
    if (st != KVX_OK)
        return st;
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
    if (cfg.batch > 0)
        p->plan.batch = cfg.batch;
    p->sync_bytes = roundtrip_sync_bytes(p->plan);
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
    if (cfg.batch > 0)
        p->plan.batch = p->load.batch = cfg.batch;
    roundtrip_setup(ctx, cfg, p->plan, p->dev + 2 * lay.total, &p->rsync, &p->shape);
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
            slab_stride = (slab_stride + KVX_STRIPE_ALIGN - 1) / KVX_STRIPE_ALIGN * KVX_STRIPE_ALIGN;
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
    kvx_launch_cfg c;
    kvx_status st = resolve_cfg(nullptr, KVX_OP_LOAD, cfg, &c);
    if (st != KVX_OK)
        return st;
    if (c.mapping != KVX_MAP_WARP_SEGMENT)
        return KVX_ERR_INVALID_ARG;
    st = kvx::validate(pool, reqs, n_req, chunks, n_chunks, layer_begin, layer_end, KVX_OP_LOAD,
                       1, false, nullptr, 0);
    if (st != KVX_OK)
        return st;
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
    int sms = 0;
    if (c.sm_cap == 0 &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVX_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

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
    if (plan.total_items == 0)
        return KVX_OK;
    if (cudaMemcpyAsync(dev_block, g_noalloc_stage, kNoallocHeader + lay.total,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KVX_ERR_CUDA;
    const int64_t warps_per_cta = c.threads / 32;
    int64_t ctas = int64_t(c.sm_cap > 0 ? c.sm_cap : sms) * c.ctas_per_sm;
    const int64_t needed = (plan.total_items + warps_per_cta - 1) / warps_per_cta;
    if (ctas > needed)
        ctas = needed;
    void *args[] = {&plan};
    if (cudaLaunchKernel(reinterpret_cast<const void *>(pick_kernel(c.unroll, KVX_DIR_SCATTER,
                                                                    c.store_hint, plan.batch)),
                         dim3(unsigned(ctas)), dim3(unsigned(c.threads)), args, 0, s) !=
        cudaSuccess)
        return KVX_ERR_CUDA;
    return KVX_OK;
}
