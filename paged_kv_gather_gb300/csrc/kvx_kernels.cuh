// kvx_kernels.cuh -- the sm_103a kernels of the paged KV gather/scatter library, and the
// functions that pick a kernel instantiation for a launch.  Included by kvx.cu only.
//
// By default a persistent grid of warps walks the batch's work items; an item is one
// (chunk, layer, kv, page) segment, contiguous on the page side
// ("Strata Guide: Hierarchical Context Caching for Long LLMs", section "Two-Dimensional
// Memory Layout Decoupling": the layout change is address arithmetic done by the moving
// thread, not a separate pass).  Each lane moves 16-byte units ("Step 1:
// High-Performance GPU-Assisted I/O CUDA Kernel": 128-bit vector accesses, a page-table
// lookup per unit of work, streaming stores into HBM), with `unroll` independent loads in
// flight per lane before its stores, because host-link reads need many bytes in flight
// (section "The Physics of I/O Bandwidth and Little's Law": X = C * S / L).  The grid is
// capped to a few SMs for host transfers so a concurrent compute stream keeps the rest
// (section "Non-Intrusive Resource Sizing"); the HBM-only transform uses every SM.
//
// Kernels: kvx_segment_kernel (store, load, HBM gather/scatter; the default mapping),
// kvx_rows_kernel (the same for chunks whose page segments are strided rows),
// kvx_split_kernel (the same for batches with fewer segments than warps, in row slices),
// their overlapped variants kvx_segment_overlap_kernel, kvx_rows_overlap_kernel and
// kvx_split_overlap_kernel,
// kvx_exchange_kernel and kvx_duplex_kernel (a store batch and a load batch in one launch),
// kvx_roundtrip_kernel (store, then load the same chunks elsewhere, ordered per unit inside
// the launch), and two alternative mappings of a single transfer: kvx_cta_kernel (a whole
// CTA per segment) and kvx_bulk_kernel (bulk-copy staging through shared memory).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

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

// Coherent 16-byte load, cached in L2 only (ld.global.cg through the compiler's own
// intrinsic, so it stays ordered after fences and warp barriers like any load): for bytes
// another warp of the same launch wrote (the read-only .nc path is valid only for data no
// thread writes during the launch).
__device__ __forceinline__ uint4 ld_cg_v4(const uint4 *p)
{
    return __ldcg(p);
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

// 32-byte accesses (sm_100 and later): one vector of eight 32-bit words per lane, so each
// warp instruction moves 1 KiB.  Used by the HBM transform when every address it touches
// is 32-byte aligned (the host checks the pool, the chunks and token_bytes).
struct V8 {
    unsigned a, b, c, d, e, f, g, h;
};

__device__ __forceinline__ V8 ld_nc_v8(const V8 *p)
{
    V8 r;
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r.a), "=r"(r.b), "=r"(r.c), "=r"(r.d), "=r"(r.e), "=r"(r.f), "=r"(r.g), "=r"(r.h)
        : "l"(p));
    return r;
}

template <int HINT>
__device__ __forceinline__ void st_v8(V8 *p, const V8 &v)
{
    if (HINT == KVX_HINT_STREAMING)
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                     "r"(v.a), "r"(v.b), "r"(v.c), "r"(v.d), "r"(v.e), "r"(v.f), "r"(v.g),
                     "r"(v.h)
                     : "memory");
    else
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                     "r"(v.a), "r"(v.b), "r"(v.c), "r"(v.d), "r"(v.e), "r"(v.f), "r"(v.g),
                     "r"(v.h)
                     : "memory");
}

// Contiguous copy of n32 32-byte units: lane i owns units i, i + 32, ...; U loads in flight.
template <int U, int HINT>
__device__ __forceinline__ void copy_contig32(const V8 *__restrict__ s, V8 *__restrict__ d,
                                              int n32, int lane)
{
    s += lane;
    d += lane;
    int rem = n32 - lane;
    for (; rem > 32 * (U - 1); rem -= 32 * U, s += 32 * U, d += 32 * U) {
        V8 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            r[u] = ld_nc_v8(s + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            st_v8<HINT>(d + 32 * u, r[u]);
    }
    if (rem > 0) {
        V8 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (32 * u < rem)
                r[u] = ld_nc_v8(s + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (32 * u < rem)
                st_v8<HINT>(d + 32 * u, r[u]);
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
    sg.contiguous = ch.row_stride == v || te - tb == 1;  // one row is one run
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

// W32: 32-byte accesses, U / 2 of them in flight per lane (the same bytes as U 16-byte ones);
// only for segments whose addresses and sizes are all multiples of 32 bytes.
template <int U, int HINT, bool NC = true, bool W32 = false>
__device__ __forceinline__ void copy_segment(const Segment &sg, int64_t v, int lane)
{
    if (W32) {
        constexpr int U32 = U > 1 ? U / 2 : 1;
        if (sg.contiguous) {
            copy_contig32<U32, HINT>(reinterpret_cast<const V8 *>(sg.src),
                                     reinterpret_cast<V8 *>(sg.dst),
                                     int((int64_t(sg.rows) * v) >> 5), lane);
        } else {
            for (int r = 0; r < sg.rows; ++r)
                copy_contig32<1, HINT>(reinterpret_cast<const V8 *>(sg.src + r * sg.s_pitch),
                                       reinterpret_cast<V8 *>(sg.dst + r * sg.d_pitch),
                                       int(v >> 5), lane);
        }
        return;
    }
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
template <int U, int DIR, int HINT, bool BATCHED, bool W32 = false>
__device__ __forceinline__ void run_segments(const Plan &p, int64_t warp, int64_t n_warps,
                                             int lane)
{
    const int64_t v = p.token_bytes;
    if (!BATCHED) {
        for (int64_t item = warp; item < p.total_items; item += n_warps) {
            Segment sg;
            if (resolve_segment<DIR>(p, item, lane, sg))
                copy_segment<U, HINT, true, W32>(sg, v, lane);
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
                    copy_segment<U, HINT, true, W32>(s, v, lane);
            }
        }
    }
}

template <int U, int DIR, int HINT, bool BATCHED, bool W32 = false>
__global__ void __launch_bounds__(1024, 1) kvx_segment_kernel(const Plan p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    run_segments<U, DIR, HINT, BATCHED, W32>(p, warp, n_warps, lane);
}

// Programmatic dependent launch (kvx_launch_cfg.overlap).  An overlapped transfer kernel
// lets the next kernel on its stream launch as soon as all its CTAs have started (when that
// kernel is launched to overlap too), and before it exits waits until the kernel before it
// on the stream has completed, so kernels on a stream still complete in order.  These
// instructions live only in the overlapped kernels: their mere presence adds about a third
// to the warp instructions of the copy loop (the durations are the same).
__device__ __forceinline__ void allow_next_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void wait_previous_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int U, int DIR, int HINT, bool BATCHED, bool W32 = false>
__global__ void __launch_bounds__(1024, 1) kvx_segment_overlap_kernel(const Plan p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    allow_next_launch();
    run_segments<U, DIR, HINT, BATCHED, W32>(p, warp, n_warps, lane);
    wait_previous_grid();
}

// Strided rows: `rows` rows of n16_row 16-byte units, row r at src + r * s_pitch and
// dst + r * d_pitch.  The units of all rows form one sequence that the warp walks as it
// walks a contiguous run (lane i owns units i, i + 32, ...), with U loads in flight per lane
// across row boundaries, so a page of short rows costs a host round trip per pass of 32 U
// units rather than one (or more) per row.  A lane's position advances 32 units at a time:
// dr rows and dc units, plus one row when the unit index within the row wraps.
template <int U, int HINT, bool NC>
__device__ __forceinline__ void copy_rows(const char *src, char *dst, int64_t s_pitch,
                                          int64_t d_pitch, int rows, int n16_row, int lane)
{
    const int total = rows * n16_row;
    const int dr = 32 / n16_row, dc = 32 - dr * n16_row;
    const int64_t s_step = dr * s_pitch + dc * 16, d_step = dr * d_pitch + dc * 16;
    const int64_t s_wrap = s_pitch - int64_t(n16_row) * 16;
    const int64_t d_wrap = d_pitch - int64_t(n16_row) * 16;
    const int row0 = lane / n16_row;
    int col = lane - row0 * n16_row;
    int64_t s_off = row0 * s_pitch + col * 16, d_off = row0 * d_pitch + col * 16;
    for (int j = lane; j < total; j += 32 * U) {
        uint4 r[U];
        int c = col;
        int64_t o = s_off;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (j + 32 * u < total)
                r[u] = ld_v4<NC>(reinterpret_cast<const uint4 *>(src + o));
            o += s_step;
            c += dc;
            if (c >= n16_row) {
                c -= n16_row;
                o += s_wrap;
            }
        }
        s_off = o;
        c = col;
        o = d_off;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (j + 32 * u < total)
                st_v4<HINT>(reinterpret_cast<uint4 *>(dst + o), r[u]);
            o += d_step;
            c += dc;
            if (c >= n16_row) {
                c -= n16_row;
                o += d_wrap;
            }
        }
        d_off = o;
        col = c;
    }
}

// A segment of a launch with token-major chunks: strided rows walked as one sequence, and a
// contiguous segment as one row (one code path, so the kernel holds one copy loop).
template <int U, int HINT, bool NC = true>
__device__ __forceinline__ void copy_segment_rows(const Segment &sg, int64_t v, int lane)
{
    if (sg.contiguous)
        copy_rows<U, HINT, NC>(sg.src, sg.dst, 0, 0, 1, int((int64_t(sg.rows) * v) >> 4), lane);
    else
        copy_rows<U, HINT, NC>(sg.src, sg.dst, sg.s_pitch, sg.d_pitch, sg.rows, int(v >> 4),
                               lane);
}

// The row walk as a call of its own, for the kernels that move both directions (the round
// trip and the exchange): inlined there twice, beside their other state, it spilled, and
// the spills cost the token-major exchange a quarter of its bandwidth.
template <int U, int HINT, bool NC>
__device__ __noinline__ void copy_segment_rows_call(const Segment sg, int64_t v, int lane)
{
    copy_segment_rows<U, HINT, NC>(sg, v, lane);
}

// One segment of a round trip: the row walk (out of line) in the variants for token-major
// chunks, the plain copy otherwise.
template <int U, int HINT, bool NC, bool ROWS>
__device__ __forceinline__ void copy_any_segment(const Segment &sg, int64_t v, int lane)
{
    if (ROWS)
        copy_segment_rows_call<U, HINT, NC>(sg, v, lane);
    else
        copy_segment<U, HINT, NC>(sg, v, lane);
}

// One segment of run_row_segments: the row walk inline, or out of line when CALL.
template <int U, int HINT, bool CALL>
__device__ __forceinline__ void copy_row_segment(const Segment &sg, int64_t v, int lane)
{
    if (CALL)
        copy_segment_rows_call<U, HINT, true>(sg, v, lane);
    else
        copy_segment_rows<U, HINT>(sg, v, lane);
}

// The warp-segment walk of run_segments for launches whose chunks include token-major ones
// of more than one (layer, kv) slab: their page segments are strided on the chunk side, and
// the plain copy moves such a segment one row and one unit per lane at a time.  CALL: the
// walk out of line (copy_segment_rows_call).
template <int U, int DIR, int HINT, bool BATCHED, bool CALL = false>
__device__ __forceinline__ void run_row_segments(const Plan &p, int64_t warp, int64_t n_warps,
                                                 int lane)
{
    const int64_t v = p.token_bytes;
    if (!BATCHED) {
        for (int64_t item = warp; item < p.total_items; item += n_warps) {
            Segment sg;
            if (resolve_segment<DIR>(p, item, lane, sg))
                copy_row_segment<U, HINT, CALL>(sg, v, lane);
        }
        return;
    }
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
            ok = segment_of<DIR>(p, find_chunk_lane(p.item_begin, p.n_chunks, mine), mine, true,
                                 sg);
        const unsigned valid = __ballot_sync(0xffffffffu, ok);
        for (int k = 0; k < B; ++k) {
            const Segment s = shfl_segment(sg, k);
            if (valid & (1u << k))
                copy_row_segment<U, HINT, CALL>(s, v, lane);
        }
    }
}

template <int U, int DIR, int HINT, bool BATCHED>
__global__ void __launch_bounds__(1024, 1) kvx_rows_kernel(const Plan p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    run_row_segments<U, DIR, HINT, BATCHED>(p, warp, n_warps, lane);
}

template <int U, int DIR, int HINT, bool BATCHED>
__global__ void __launch_bounds__(1024, 1) kvx_rows_overlap_kernel(const Plan p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    allow_next_launch();
    run_row_segments<U, DIR, HINT, BATCHED>(p, warp, n_warps, lane);
    wait_previous_grid();
}

// Few segments, many warps: each segment is cut into p.split slices of its rows, one warp
// per slice, so a small transfer still puts the whole grid's bytes in flight.  Slice k of
// a segment of r rows holds rows [k r / split, (k + 1) r / split); a slice may be empty
// when a partial page has fewer rows than split.
template <int U, int DIR, int HINT>
__device__ __forceinline__ void split_segments(const Plan &p)
{
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int S = p.split;
    const int64_t v = p.token_bytes;
    for (int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         w < p.total_items * S; w += n_warps) {
        const int64_t item = w / S;
        const int k = int(w - item * S);
        Segment sg;
        if (!resolve_segment<DIR>(p, item, lane, sg))
            continue;
        const int r0 = k * sg.rows / S, r1 = (k + 1) * sg.rows / S;
        if (r1 <= r0)
            continue;
        sg.src += int64_t(r0) * sg.s_pitch;
        sg.dst += int64_t(r0) * sg.d_pitch;
        sg.rows = r1 - r0;
        copy_segment<U, HINT>(sg, v, lane);
    }
}

template <int U, int DIR, int HINT>
__global__ void __launch_bounds__(1024, 1) kvx_split_kernel(const Plan p)
{
    split_segments<U, DIR, HINT>(p);
}

template <int U, int DIR, int HINT>
__global__ void __launch_bounds__(1024, 1) kvx_split_overlap_kernel(const Plan p)
{
    allow_next_launch();
    split_segments<U, DIR, HINT>(p);
    wait_previous_grid();
}

// Exchange: one launch moves a store batch (pages -> host chunks) and a load batch (host
// chunks -> pages) at once.  Even CTAs run the store plan, odd CTAs the load plan, so the
// block scheduler spreads both directions evenly over the SMs the launch gets instead of
// giving each direction its own contiguous block of SMs (two separate kernels), which
// lets the two directions of the host link run at full rate together.
// ROWS: the row walk of run_row_segments, out of line (chunks include token-major ones of
// several slabs).
template <int U, bool BATCHED_S, bool BATCHED_L, bool ROWS = false>
__global__ void __launch_bounds__(1024, 1) kvx_exchange_kernel(const Plan ps, const Plan pl)
{
    const int lane = threadIdx.x & 31;
    const int64_t wpc = blockDim.x >> 5;
    const int64_t role_cta = blockIdx.x >> 1;
    const int64_t warp = role_cta * wpc + (threadIdx.x >> 5);
    if ((blockIdx.x & 1) == 0) {
        const int64_t ctas = (int64_t(gridDim.x) + 1) >> 1;
        if (ROWS)
            run_row_segments<U, KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED_S, true>(
                ps, warp, ctas * wpc, lane);
        else
            run_segments<U, KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED_S>(ps, warp, ctas * wpc,
                                                                        lane);
    } else {
        const int64_t ctas = int64_t(gridDim.x) >> 1;
        if (ROWS)
            run_row_segments<U, KVX_DIR_SCATTER, KVX_HINT_STREAMING, BATCHED_L, true>(
                pl, warp, ctas * wpc, lane);
        else
            run_segments<U, KVX_DIR_SCATTER, KVX_HINT_STREAMING, BATCHED_L>(pl, warp,
                                                                            ctas * wpc, lane);
    }
}

// ------------------------------------------------------------------ CTA-per-segment mapping
//
// Every thread of a CTA moves part of the same segment: thread t takes 16-byte units t,
// t + T, t + 2T, ... (T threads), U of them in flight before their stores.  Warp 0
// resolves 32 consecutive segments at once, one per lane, into shared memory; the CTA then
// walks them without further synchronisation.  Per SM this keeps the bytes in flight of
// many warps while touching only a few segments (DRAM streams) at a time.

// Units [0, n16) of one segment, strided over the CTA.
template <int U, int HINT>
__device__ __forceinline__ void copy_contig_cta(const uint4 *__restrict__ s,
                                                uint4 *__restrict__ d, int n16, int tid, int T)
{
    int i = tid;
    for (; i + (U - 1) * T < n16; i += U * T) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            r[u] = ld_nc_v4(s + i + u * T);
#pragma unroll
        for (int u = 0; u < U; ++u)
            st_v4<HINT>(d + i + u * T, r[u]);
    }
    if (i < n16) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i + u * T < n16)
                r[u] = ld_nc_v4(s + i + u * T);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i + u * T < n16)
                st_v4<HINT>(d + i + u * T, r[u]);
    }
}

template <int U, int DIR, int HINT>
__global__ void __launch_bounds__(1024, 1) kvx_cta_kernel(const Plan p)
{
    __shared__ Segment segs[32];
    __shared__ unsigned valid;
    const int tid = threadIdx.x;
    const int T = blockDim.x;
    const int64_t v = p.token_bytes;
    const int units_per_row = int(v >> 4);
    for (int64_t base = int64_t(blockIdx.x) * 32; base < p.total_items;
         base += int64_t(gridDim.x) * 32) {
        __syncthreads();  // the previous batch's segments are no longer read
        if (tid < 32) {
            Segment sg;
            sg.src = nullptr;
            sg.dst = nullptr;
            sg.s_pitch = sg.d_pitch = 0;
            sg.rows = 0;
            sg.contiguous = true;
            const int64_t mine = base + tid;
            bool ok = false;
            if (mine < p.total_items)
                ok = segment_of<DIR>(p, find_chunk_lane(p.item_begin, p.n_chunks, mine), mine,
                                     true, sg);
            segs[tid] = sg;
            const unsigned m = __ballot_sync(0xffffffffu, ok);
            if (tid == 0)
                valid = m;
        }
        __syncthreads();
        const unsigned m = valid;
        const int n = int(min(int64_t(32), p.total_items - base));
        for (int k = 0; k < n; ++k) {
            if (!((m >> k) & 1u))
                continue;
            const Segment sg = segs[k];
            if (sg.contiguous) {
                copy_contig_cta<U, HINT>(reinterpret_cast<const uint4 *>(sg.src),
                                         reinterpret_cast<uint4 *>(sg.dst),
                                         int((int64_t(sg.rows) * v) >> 4), tid, T);
            } else {
                // Token-major chunk: unit j of the segment is unit j % units_per_row of row
                // j / units_per_row, each row at its own pitch on the chunk side.
                const int total = sg.rows * units_per_row;
                for (int j = tid; j < total; j += T) {
                    const int r = j / units_per_row, u = j - r * units_per_row;
                    const uint4 x = ld_nc_v4(reinterpret_cast<const uint4 *>(
                                                 sg.src + r * sg.s_pitch) + u);
                    st_v4<HINT>(reinterpret_cast<uint4 *>(sg.dst + r * sg.d_pitch) + u, x);
                }
            }
        }
    }
}

typedef void (*CtaFn)(Plan);

template <int U>
CtaFn pick_cta_u(int dir, int hint)
{
    if (dir == KVX_DIR_GATHER)
        return hint == KVX_HINT_STREAMING ? kvx_cta_kernel<U, KVX_DIR_GATHER, 1>
                                          : kvx_cta_kernel<U, KVX_DIR_GATHER, 0>;
    return hint == KVX_HINT_STREAMING ? kvx_cta_kernel<U, KVX_DIR_SCATTER, 1>
                                      : kvx_cta_kernel<U, KVX_DIR_SCATTER, 0>;
}

// The CTA-per-segment kernel for (unroll, direction, hint); nullptr for another unroll.
CtaFn pick_cta(int unroll, int dir, int hint)
{
    switch (unroll) {
    case 1: return pick_cta_u<1>(dir, hint);
    case 2: return pick_cta_u<2>(dir, hint);
    case 4: return pick_cta_u<4>(dir, hint);
    case 8: return pick_cta_u<8>(dir, hint);
    }
    return nullptr;
}

// ------------------------------------------------------------------ bulk-copy (TMA) mapping
//
// Host-link bandwidth per SM is capped on GB300 at about 50 GB/s however the bytes in
// flight are held (registers, cp.async into shared memory or bulk copies), and host reads
// reach that cap only with about 128 KiB in flight per SM: less is latency-bound, more
// queues up and runs slower.  So the fewest SMs that reach the link's peak are the ones
// that keep exactly that much in flight without stalls between copies.  Each CTA here is
// three warps.  Warp 0 resolves the CTA's segments 32 at a time, one per lane (chunk search
// and page-table read in parallel), into a queue of kBulkQueue batches in shared memory.
// Lane 0 of warps 1 and 2 (the copy lanes) take alternate batches and each drives the
// Blackwell bulk-copy engine on its own ring of n_stages shared-memory stages: it packs
// segments into stages back to back, cutting a segment where a stage ends, loads each full
// stage (cp.async.bulk global -> shared, completing on the stage's mbarrier with transaction
// bytes) and writes it out (cp.async.bulk shared -> global, one bulk group per stage), with
// one copy per run of pieces that lie back to back on that side: a stage's host side is
// then usually one copy, and only its page side needs one copy per page segment.  Each
// lane keeps n_stages - 1 stages loading while the next fills; two lanes keep their issue
// costs (a bulk copy occupies its issuing thread for a few hundred cycles) from adding up.
// Every wait is bounded (about one second): on expiry the kernel flags
// KVX_DEV_WAIT_TIMEOUT, issues nothing more, waits (again bounded) for the copies it issued
// and exits.

constexpr int kBulkLanes = 2;         // copy lanes per CTA, each with its own ring
constexpr int kBulkMaxStages = 8;     // stages per ring
constexpr int kBulkQueue = 4;         // resolved batches of 32 segments between the warps
constexpr int kBulkStagePieces = 32;  // pieces per stage at most
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

// One arrival (release at CTA scope: the caller's earlier shared-memory writes are visible
// to whoever waits on the completed phase).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}

// One thread: bounded wait for the completion of phase `parity` of an mbarrier.
__device__ __forceinline__ bool mbar_wait1(uint64_t *bar, uint32_t parity)
{
    if (mbar_test(bar, parity))
        return true;
    const uint64_t deadline = global_ns() + kWaitLimitNs;
    while (!mbar_test(bar, parity))
        if (global_ns() > deadline)
            return false;
    return true;
}

// Warp-uniform bounded wait (every lane returns the same answer); sleeps between polls so
// that a waiting warp leaves the shared-memory pipe to the copy lanes.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, int lane)
{
    const uint64_t deadline = global_ns() + kWaitLimitNs;
    while (true) {
        if (__any_sync(0xffffffffu, mbar_test(bar, parity)))
            return true;
        const int late = lane == 0 ? int(global_ns() > deadline) : 0;
        if (__shfl_sync(0xffffffffu, late, 0))
            return false;
        __nanosleep(500);
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
}

// One copy lane's ring bookkeeping.
struct BulkLaneState {
    uint64_t full[kBulkMaxStages];  // stage loaded: one arrival + its bytes
    const char *psrc[kBulkMaxStages][kBulkStagePieces];
    char *pdst[kBulkMaxStages][kBulkStagePieces];
    uint32_t poff[kBulkMaxStages][kBulkStagePieces];
    uint32_t plen[kBulkMaxStages][kBulkStagePieces];
    uint32_t npieces[kBulkMaxStages];
};

// Shared state of one bulk CTA (the rings of stages are the dynamic shared memory).
struct BulkShared {
    uint64_t qfull[kBulkQueue];   // batch resolved: 32 arrivals (every lane of warp 0)
    uint64_t qempty[kBulkQueue];  // batch consumed: one arrival (its copy lane)
    Segment seg[kBulkQueue][32];
    unsigned valid[kBulkQueue];
    BulkLaneState lane[kBulkLanes];
};

// A copy lane's ring: stages [retired, issued) are loading (their loads issued, their
// stores not yet), and stage `issued` is being filled when `open`.
struct BulkRing {
    BulkLaneState &ls;
    unsigned char *ring;
    uint32_t stage_bytes;
    uint32_t n_stages;
    uint32_t issued = 0, retired = 0;
    uint32_t fill = 0, np = 0;
    bool open = false;

    __device__ BulkRing(BulkLaneState &s, unsigned char *r, uint32_t sb, uint32_t ns)
        : ls(s), ring(r), stage_bytes(sb), n_stages(ns)
    {
    }

    __device__ unsigned char *stage(uint32_t st) { return ring + size_t(st) * stage_bytes; }

    // Oldest loading stage: wait for its bytes, then write it out (one bulk group), one bulk
    // copy per run of pieces that are back to back at their destination.
    __device__ bool retire_one()
    {
        const uint32_t st = retired % n_stages;
        if (!mbar_wait1(&ls.full[st], (retired / n_stages) & 1u))
            return false;
        const uint32_t n = ls.npieces[st];
        for (uint32_t i = 0; i < n;) {
            char *d = ls.pdst[st][i];
            uint32_t bytes = ls.plen[st][i];
            uint32_t j = i + 1;
            for (; j < n && ls.pdst[st][j] == d + bytes; ++j)
                bytes += ls.plen[st][j];
            bulk_store(d, stage(st) + ls.poff[st][i], bytes);
            i = j;
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        ++retired;
        return true;
    }

    // The open stage is complete: expect its bytes (with the stage's one arrival), then load
    // it, one bulk copy per run of pieces that are back to back at their source.
    __device__ void close_stage()
    {
        const uint32_t st = issued % n_stages;
        ls.npieces[st] = np;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                         smem_u32(&ls.full[st])),
                     "r"(fill)
                     : "memory");
        for (uint32_t i = 0; i < np;) {
            const char *s = ls.psrc[st][i];
            uint32_t bytes = ls.plen[st][i];
            uint32_t j = i + 1;
            for (; j < np && ls.psrc[st][j] == s + bytes; ++j)
                bytes += ls.plen[st][j];
            bulk_load(stage(st) + ls.poff[st][i], s, bytes, &ls.full[st]);
            i = j;
        }
        ++issued;
        open = false;
    }

    __device__ bool open_stage()
    {
        if (issued - retired == n_stages - 1 && !retire_one())
            return false;
        // The stage about to be filled was last written out n_stages stages ago; at most one
        // newer store group may still be reading shared memory.
        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        open = true;
        fill = 0;
        np = 0;
        return true;
    }

    // A contiguous run of `bytes` (a multiple of 16): recorded as pieces cut at stage
    // boundaries, so every stage but the last is filled completely whatever the segment size.
    __device__ bool add_run(const char *src, char *dst, int64_t bytes)
    {
        while (bytes > 0) {
            if (!open && !open_stage())
                return false;
            const uint32_t st = issued % n_stages;
            const uint32_t take = uint32_t(min(bytes, int64_t(stage_bytes - fill)));
            ls.psrc[st][np] = src;
            ls.pdst[st][np] = dst;
            ls.poff[st][np] = fill;
            ls.plen[st][np] = take;
            ++np;
            fill += take;
            src += take;
            dst += take;
            bytes -= take;
            if (fill == stage_bytes || np == kBulkStagePieces)
                close_stage();
        }
        return true;
    }

    // After a timeout: issue no more stores, but wait (bounded) until the loads already
    // issued have landed, so that no bulk copy still targets this CTA's shared memory when
    // it exits.  False if one of them did not land within its limit either.
    __device__ bool drain_loads()
    {
        open = false;  // the open stage's loads are issued only when it closes: none yet
        bool ok = true;
        for (; retired < issued; ++retired)
            ok = mbar_wait1(&ls.full[retired % n_stages], (retired / n_stages) & 1u) && ok;
        return ok;
    }
};

// The CTA's items are first, first + 1, ..., first + n_mine - 1 (a contiguous block, so
// that consecutive segments of a chunk stay back to back on its side); batch k holds items
// first + 32 k .. first + 32 k + 31.
template <int DIR>
__device__ __forceinline__ void bulk_resolver(const Plan &p, BulkShared &sh, int64_t first,
                                              int64_t n_mine, int64_t n_batches, int lane)
{
    for (int64_t k = 0; k < n_batches; ++k) {
        const int q = int(k % kBulkQueue);
        if (k >= kBulkQueue &&
            !mbar_wait_warp(&sh.qempty[q], uint32_t((k / kBulkQueue - 1) & 1), lane)) {
            if (lane == 0)
                atomicOr(p.status, KVX_DEV_WAIT_TIMEOUT);
            return;  // the copy lane's wait for this batch then runs out too
        }
        Segment sg;
        sg.src = nullptr;
        sg.dst = nullptr;
        sg.s_pitch = sg.d_pitch = 0;
        sg.rows = 0;
        sg.contiguous = true;
        bool ok = false;
        const int64_t idx = k * 32 + lane;
        if (idx < n_mine) {
            const int64_t item = first + idx;
            ok = segment_of<DIR>(p, find_chunk_lane(p.item_begin, p.n_chunks, item), item, true,
                                 sg);
        }
        sh.seg[q][lane] = sg;
        const unsigned m = __ballot_sync(0xffffffffu, ok);
        if (lane == 0)
            sh.valid[q] = m;
        mbar_arrive(&sh.qfull[q]);  // each lane releases its own entry (and lane 0 the mask)
    }
}

// Copy lane `which`: batches which, which + kBulkLanes, ...
template <int DIR>
__device__ __forceinline__ void bulk_copier(const Plan &p, BulkShared &sh, unsigned char *ring,
                                            int stage_bytes, int n_stages, int64_t n_batches,
                                            int which)
{
    BulkRing r(sh.lane[which], ring + size_t(which) * n_stages * stage_bytes,
               uint32_t(stage_bytes), uint32_t(n_stages));
    const int64_t v = p.token_bytes;
    bool ok = true;
    for (int64_t k = which; k < n_batches && ok; k += kBulkLanes) {
        const int q = int(k % kBulkQueue);
        if (!mbar_wait1(&sh.qfull[q], uint32_t((k / kBulkQueue) & 1))) {
            ok = false;
            break;
        }
        const unsigned m = sh.valid[q];
        for (int i = 0; i < 32 && ok; ++i) {
            if (!((m >> i) & 1u))
                continue;
            const Segment sg = sh.seg[q][i];
            const int n_runs = sg.contiguous ? 1 : sg.rows;
            const int64_t run = sg.contiguous ? int64_t(sg.rows) * v : v;
            for (int rr = 0; rr < n_runs && ok; ++rr)
                ok = r.add_run(sg.src + rr * sg.s_pitch, sg.dst + rr * sg.d_pitch, run);
        }
        mbar_arrive(&sh.qempty[q]);  // the batch's entries are no longer read
    }
    if (ok) {
        if (r.open)
            r.close_stage();
        while (ok && r.retired < r.issued)
            ok = r.retire_one();
    }
    if (!ok) {
        atomicOr(p.status, KVX_DEV_WAIT_TIMEOUT);
        r.drain_loads();
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// n_stages stages of stage_bytes per copy lane: dynamic shared memory of
// kBulkLanes x n_stages x stage_bytes.
template <int DIR>
__global__ void __launch_bounds__(32 * (1 + kBulkLanes), 1)
    kvx_bulk_kernel(const Plan p, int stage_bytes, int n_stages)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ BulkShared sh;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t per_cta = (p.total_items + gridDim.x - 1) / gridDim.x;
    const int64_t first = min(p.total_items, int64_t(blockIdx.x) * per_cta);
    const int64_t n_mine = min(p.total_items - first, per_cta);
    const int64_t n_batches = (n_mine + 31) / 32;
    if (threadIdx.x == 0) {
        for (int j = 0; j < kBulkLanes; ++j)
            for (int st = 0; st < n_stages; ++st)
                mbar_init(&sh.lane[j].full[st], 1);
        for (int q = 0; q < kBulkQueue; ++q) {
            mbar_init(&sh.qfull[q], 32);
            mbar_init(&sh.qempty[q], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0)
        bulk_resolver<DIR>(p, sh, first, n_mine, n_batches, lane);
    else if (lane == 0)
        bulk_copier<DIR>(p, sh, ring, stage_bytes, n_stages, n_batches, warp - 1);
}

// ------------------------------------------------------------------------- round trip
//
// Store a batch to host chunks and load the same chunks into other pages in one launch
// (a swap-out followed by a swap-in elsewhere).  The store and load plans enumerate the
// same items, so load unit u reads exactly the host bytes store unit u writes.  A unit is
// unit_items consecutive items, or one row slice of a long item (slices > 1); units are
// handed out by two fetch-and-add counters, one per direction.  A warp takes a store unit
// while the loads handed out are within `lag` units (one per warp of the grid by default)
// of the stores handed out, and a load unit otherwise, so each load usually starts well
// after its store finished.  A warp that holds a load unit whose store has not been
// handed out yet hands out (and does) store units until it has; only then does it wait
// for that store.  Every wait is therefore on a unit held by a
// running warp that waits on nothing, whatever the residency of the grid, so the waits
// end; each is still bounded (about one second, then KVX_DEV_WAIT_TIMEOUT and the unit is
// skipped).  Both directions of the host link run from the first completed store to the
// last load, in a single launch.

struct RoundTripSync {
    unsigned int *next;  // [0] next store unit, [1] next load unit; zero at launch
    unsigned int *done;  // [units]: 1 once the store unit's bytes are in host memory
    int64_t units;
    int unit_items;
    int slices;          // > 1: unit u is row slice u % slices of item u / slices
    unsigned lag;        // loads handed out may trail stores handed out by this many units
    uint64_t wait_ns;    // limit of one wait for a store unit (about one second)
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
    const uint64_t deadline = global_ns() + sy.wait_ns;
    while (ld_acquire_u32(sy.done + unit) == 0u) {
        if (global_ns() > deadline)
            return false;
        __nanosleep(200);
    }
    return true;
}

enum : int { kUnitStore = 1, kUnitLoad = 2, kUnitSkip = 3 };

// Lane 0: the warp's next unit (-1: nothing left for this warp) and what to do with it.
// `pending` carries a load unit taken before its store was handed out.  Units stay below
// 2^31 (the host checks), so 32-bit indices hold them.
__device__ __forceinline__ int next_unit(const RoundTripSync &sy, unsigned lag, int &pending,
                                         int &what)
{
    const unsigned n = unsigned(sy.units);
    if (pending < 0) {
        const unsigned si = ld_relaxed_u32(sy.next);
        const unsigned li = ld_relaxed_u32(sy.next + 1);
        if (si < n && li + lag >= si) {
            const unsigned s = atomicAdd(sy.next, 1u);
            if (s < n) {
                what = kUnitStore;
                return int(s);
            }
        }
        const unsigned t = atomicAdd(sy.next + 1, 1u);
        if (t >= n)
            return -1;  // every load is handed out; their holders finish the stores
        pending = int(t);
    }
    if (ld_relaxed_u32(sy.next) <= unsigned(pending)) {
        // The store this load needs is not handed out yet: hand out the next one.
        const unsigned s = atomicAdd(sy.next, 1u);
        if (s < n) {
            what = kUnitStore;
            return int(s);
        }
    }
    const int u = pending;
    pending = -1;
    what = wait_unit(sy, u) ? kUnitLoad : kUnitSkip;
    return u;
}

// Items [first, first + count) of plan p, warp-collective (count is 1 unless BATCHED).
// With slices > 1 (not BATCHED), only rows [k r / slices, (k + 1) r / slices) of the one
// item's r rows, k = slice.  NC = false for bytes written earlier in the same launch.  ROWS:
// strided rows walked as one sequence (chunks include token-major ones of several slabs).
template <int U, int DIR, int HINT, bool BATCHED, bool NC, bool ROWS = false>
__device__ __forceinline__ void copy_items(const Plan &p, int64_t first, int count, int lane,
                                           int slices = 1, int slice = 0)
{
    const int64_t v = p.token_bytes;
    if (!BATCHED) {  // one item per unit
        Segment sg;
        if (resolve_segment<DIR>(p, first, lane, sg)) {
            if (slices > 1) {
                const int r0 = int(int64_t(slice) * sg.rows / slices);
                const int r1 = int(int64_t(slice + 1) * sg.rows / slices);
                sg.src += int64_t(r0) * sg.s_pitch;
                sg.dst += int64_t(r0) * sg.d_pitch;
                sg.rows = r1 - r0;
            }
            if (sg.rows > 0)
                copy_any_segment<U, HINT, NC, ROWS>(sg, v, lane);
        }
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
            copy_any_segment<U, HINT, NC, ROWS>(sk, v, lane);
    }
}

template <int U, bool BATCHED, bool ROWS>
__global__ void __launch_bounds__(1024, 1)
    kvx_roundtrip_kernel(const Plan ps, const Plan pl, const RoundTripSync sy)
{
    const int lane = threadIdx.x & 31;
    int pending = -1;  // lane 0's
    for (;;) {
        int unit = -1;
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
        int64_t first;
        int count, slice = 0;
        if (sy.slices > 1) {  // a row slice of one long segment
            first = unit / sy.slices;
            slice = int(unit - first * sy.slices);
            count = 1;
        } else {
            first = int64_t(unit) * sy.unit_items;
            count = int(min(int64_t(sy.unit_items), ps.total_items - first));
        }
        if (what == kUnitLoad) {
            // Short (batched) segments fill at most a few loads per lane: four are enough.
            copy_items<((BATCHED || ROWS) && U > 4 ? 4 : U), KVX_DIR_SCATTER,
                       KVX_HINT_STREAMING, BATCHED, false, ROWS>(pl, first, count, lane,
                                                                 sy.slices, slice);
        } else {
            // HBM reads need fewer bytes in flight than host reads: four loads per lane.
            copy_items<(U > 4 ? 4 : U), KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED, true, ROWS>(
                ps, first, count, lane, sy.slices, slice);
            // Each lane's host writes are performed at GPU scope, then lane 0 publishes the
            // unit with a release (the fence costs nothing measurable, and it keeps the
            // publication correct without leaning on the warp barrier's ordering).
            __threadfence();
            __syncwarp();
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

template <int U, bool BATCHED, bool ROWS = false>
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
            // Short (batched) segments fill at most a few loads per lane: four are enough.
            copy_items<((BATCHED || ROWS) && U > 4 ? 4 : U), KVX_DIR_SCATTER,
                       KVX_HINT_STREAMING, BATCHED, true, ROWS>(pl, first, count, lane);
        } else {
            const int count = int(min(int64_t(sy.unit_items), ps.total_items - first));
            copy_items<(U > 4 ? 4 : U), KVX_DIR_GATHER, KVX_HINT_DEFAULT, BATCHED, true, ROWS>(
                ps, first, count, lane);
        }
    }
}

typedef void (*DuplexFn)(Plan, Plan, DuplexSync);

// The shared-work exchange kernel for (unroll, batched); rows: strided token-major rows
// walked as one sequence, out of line and at most 4 loads deep, for segments of one unit
// each (batched ones keep the plain copy, as in the round trip).
DuplexFn pick_duplex(int unroll, bool batched, bool rows = false)
{
    if (rows && !batched) {
        switch (unroll) {
        case 1: return kvx_duplex_kernel<1, false, true>;
        case 2: return kvx_duplex_kernel<2, false, true>;
        case 4:
        case 8: return kvx_duplex_kernel<4, false, true>;
        }
        return nullptr;
    }
    switch (unroll) {
    case 1: return batched ? kvx_duplex_kernel<1, true> : kvx_duplex_kernel<1, false>;
    case 2: return batched ? kvx_duplex_kernel<2, true> : kvx_duplex_kernel<2, false>;
    case 4: return batched ? kvx_duplex_kernel<4, true> : kvx_duplex_kernel<4, false>;
    case 8: return batched ? kvx_duplex_kernel<8, true> : kvx_duplex_kernel<8, false>;
    }
    return nullptr;
}

typedef void (*RoundTripFn)(Plan, Plan, RoundTripSync);

// The round-trip kernel for (unroll, batched), walking strided rows as one sequence when rows
// (chunks include a token-major one of several slabs).  The row walk holds at most 4 loads
// in flight per lane.  Its batched variants spill around the out-of-line walk, and still
// beat the plain copy's row at a time by 13 % on pages of 2 and 4 MLA tokens.
RoundTripFn pick_roundtrip(int unroll, bool batched, bool rows = false)
{
    if (rows) {
        switch (unroll) {
        case 1:
            return batched ? kvx_roundtrip_kernel<1, true, true>
                           : kvx_roundtrip_kernel<1, false, true>;
        case 2:
            return batched ? kvx_roundtrip_kernel<2, true, true>
                           : kvx_roundtrip_kernel<2, false, true>;
        case 4:
        case 8:
            return batched ? kvx_roundtrip_kernel<4, true, true>
                           : kvx_roundtrip_kernel<4, false, true>;
        }
        return nullptr;
    }
    switch (unroll) {
    case 1:
        return batched ? kvx_roundtrip_kernel<1, true, false>
                       : kvx_roundtrip_kernel<1, false, false>;
    case 2:
        return batched ? kvx_roundtrip_kernel<2, true, false>
                       : kvx_roundtrip_kernel<2, false, false>;
    case 4:
        return batched ? kvx_roundtrip_kernel<4, true, false>
                       : kvx_roundtrip_kernel<4, false, false>;
    case 8:
        return batched ? kvx_roundtrip_kernel<8, true, false>
                       : kvx_roundtrip_kernel<8, false, false>;
    }
    return nullptr;
}

typedef void (*KernelFn)(Plan);

template <int U, int DIR, int HINT, bool BATCHED, bool W32>
KernelFn segment_fn(bool overlap)
{
    return overlap ? kvx_segment_overlap_kernel<U, DIR, HINT, BATCHED, W32>
                   : kvx_segment_kernel<U, DIR, HINT, BATCHED, W32>;
}

template <int U, bool BATCHED, bool W32>
KernelFn pick_hint_dir(int dir, int hint, bool overlap)
{
    if (dir == KVX_DIR_GATHER)
        return hint == KVX_HINT_STREAMING
                   ? segment_fn<U, KVX_DIR_GATHER, 1, BATCHED, W32>(overlap)
                   : segment_fn<U, KVX_DIR_GATHER, 0, BATCHED, W32>(overlap);
    return hint == KVX_HINT_STREAMING ? segment_fn<U, KVX_DIR_SCATTER, 1, BATCHED, W32>(overlap)
                                      : segment_fn<U, KVX_DIR_SCATTER, 0, BATCHED, W32>(overlap);
}

template <bool BATCHED, bool W32>
KernelFn pick_unroll(int unroll, int dir, int hint, bool overlap)
{
    switch (unroll) {
    case 1: return pick_hint_dir<1, BATCHED, W32>(dir, hint, overlap);
    case 2: return pick_hint_dir<2, BATCHED, W32>(dir, hint, overlap);
    case 4: return pick_hint_dir<4, BATCHED, W32>(dir, hint, overlap);
    case 8: return pick_hint_dir<8, BATCHED, W32>(dir, hint, overlap);
    }
    return nullptr;
}

template <int U, int DIR, int HINT, bool BATCHED>
KernelFn rows_fn(bool overlap)
{
    return overlap ? kvx_rows_overlap_kernel<U, DIR, HINT, BATCHED>
                   : kvx_rows_kernel<U, DIR, HINT, BATCHED>;
}

template <int U, bool BATCHED>
KernelFn pick_rows_hint_dir(int dir, int hint, bool overlap)
{
    if (dir == KVX_DIR_GATHER)
        return hint == KVX_HINT_STREAMING ? rows_fn<U, KVX_DIR_GATHER, 1, BATCHED>(overlap)
                                          : rows_fn<U, KVX_DIR_GATHER, 0, BATCHED>(overlap);
    return hint == KVX_HINT_STREAMING ? rows_fn<U, KVX_DIR_SCATTER, 1, BATCHED>(overlap)
                                      : rows_fn<U, KVX_DIR_SCATTER, 0, BATCHED>(overlap);
}

// The row-walking kernel holds at most 4 loads in flight per lane: its position arithmetic
// leaves no registers for 8 at 1024 threads per CTA.
template <bool BATCHED>
KernelFn pick_rows(int unroll, int dir, int hint, bool overlap)
{
    switch (unroll) {
    case 1: return pick_rows_hint_dir<1, BATCHED>(dir, hint, overlap);
    case 2: return pick_rows_hint_dir<2, BATCHED>(dir, hint, overlap);
    case 4:
    case 8: return pick_rows_hint_dir<4, BATCHED>(dir, hint, overlap);
    }
    return nullptr;
}

// The warp-segment kernel for (unroll, direction, hint), batched when more than one
// segment is resolved per warp at once, with 32-byte accesses when w32, walking strided
// rows as one sequence when rows (launches with token-major chunks; not with w32), and the
// overlapped variant when overlap.
KernelFn pick_kernel(int unroll, int dir, int hint, int batch = 1, bool w32 = false,
                     bool overlap = false, bool rows = false)
{
    if (rows && !w32)
        return batch > 1 ? pick_rows<true>(unroll, dir, hint, overlap)
                         : pick_rows<false>(unroll, dir, hint, overlap);
    if (w32)
        return batch > 1 ? pick_unroll<true, true>(unroll, dir, hint, overlap)
                         : pick_unroll<false, true>(unroll, dir, hint, overlap);
    return batch > 1 ? pick_unroll<true, false>(unroll, dir, hint, overlap)
                     : pick_unroll<false, false>(unroll, dir, hint, overlap);
}

template <int U, int DIR, int HINT>
KernelFn split_fn(bool overlap)
{
    return overlap ? kvx_split_overlap_kernel<U, DIR, HINT> : kvx_split_kernel<U, DIR, HINT>;
}

template <int U>
KernelFn pick_split_u(int dir, int hint, bool overlap)
{
    if (dir == KVX_DIR_GATHER)
        return hint == KVX_HINT_STREAMING ? split_fn<U, KVX_DIR_GATHER, 1>(overlap)
                                          : split_fn<U, KVX_DIR_GATHER, 0>(overlap);
    return hint == KVX_HINT_STREAMING ? split_fn<U, KVX_DIR_SCATTER, 1>(overlap)
                                      : split_fn<U, KVX_DIR_SCATTER, 0>(overlap);
}

// The row-slice kernel for (unroll, direction, hint), overlapped when overlap.
KernelFn pick_split(int unroll, int dir, int hint, bool overlap = false)
{
    switch (unroll) {
    case 1: return pick_split_u<1>(dir, hint, overlap);
    case 2: return pick_split_u<2>(dir, hint, overlap);
    case 4: return pick_split_u<4>(dir, hint, overlap);
    case 8: return pick_split_u<8>(dir, hint, overlap);
    }
    return nullptr;
}

typedef void (*ExchangeFn)(Plan, Plan);

template <int U, bool ROWS>
ExchangeFn pick_exchange_u(bool bs, bool bl)
{
    if (bs)
        return bl ? kvx_exchange_kernel<U, true, true, ROWS>
                  : kvx_exchange_kernel<U, true, false, ROWS>;
    return bl ? kvx_exchange_kernel<U, false, true, ROWS>
              : kvx_exchange_kernel<U, false, false, ROWS>;
}

// The role-split exchange kernel; rows: the row-walking variant (at most 4 loads in flight
// per lane), for chunks that include a token-major one of several slabs.
ExchangeFn pick_exchange(int unroll, int batch_s, int batch_l, bool rows = false)
{
    const bool bs = batch_s > 1, bl = batch_l > 1;
    if (rows) {
        switch (unroll) {
        case 1: return pick_exchange_u<1, true>(bs, bl);
        case 2: return pick_exchange_u<2, true>(bs, bl);
        case 4:
        case 8: return pick_exchange_u<4, true>(bs, bl);
        }
        return nullptr;
    }
    switch (unroll) {
    case 1: return pick_exchange_u<1, false>(bs, bl);
    case 2: return pick_exchange_u<2, false>(bs, bl);
    case 4: return pick_exchange_u<4, false>(bs, bl);
    case 8: return pick_exchange_u<8, false>(bs, bl);
    }
    return nullptr;
}

}  // namespace

