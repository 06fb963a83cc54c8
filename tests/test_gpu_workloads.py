"""GPU parity at the full sizes of the five workloads, in the launch configurations the bench
times (the library defaults, and the few-SM and partition legs), every output byte checked
against the CPU oracle.

Verification copies device tensors into pinned host memory and runs the oracle on them:
  llama8b       store, load, HBM gather/scatter and the per-page DMA baseline, all layers;
                the headline round trip in one launch, and the exchange pipeline;
  llama8b       also the store and load on 4 SMs, bulk and register mappings;
  llama70b      80 layer-streamed loads, 1 MiB and 2 MiB per-layer chunks, every layer, and
                with the bulk mapping on 5 SMs;
  qwen7b_batch  one batched load and one batched store concurrently on two streams (plain,
                or two I/O partitions), and both in one exchange launch;
  mla_sweep     every page size x chunk size cell, store and load, kernel and DMA baseline;
  mla_blocks    per-block STRIPED objects: one store, then per-layer loads.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_gather_gb300.build import build  # noqa: E402

build()
import oracle  # noqa: E402
from paged_kv_gather_gb300 import kvx  # noqa: E402
from paged_kv_gather_gb300 import workloads as wl  # noqa: E402
from tests.gpu_common import (CANARY, HostPool, Requests, assert_bytes_equal,  # noqa: E402
                              oracle_chunks, pinned_copy)


@pytest.fixture(scope="module")
def ctx():
    c = kvx.kvx_create(0, 64 << 20)
    yield c
    kvx.kvx_destroy(c)


def _pools(shape, seed, fill=None):
    t = torch.empty((shape.kv_factor, shape.num_layers, shape.num_pages, shape.page_size,
                     shape.token_bytes), dtype=torch.uint8, device="cuda")
    if fill is None:
        wl.fill_values(t, shape.dtype, wl.values_generator(seed, "cuda"))
    else:
        t.fill_(fill)
    return t


def _fill_host(hb_array, nbytes, shape, seed, stream_id):
    """Seeded K/V values for host chunks: drawn on the GPU, copied into the host arena."""
    g = wl.values_generator(seed, "cuda", stream=stream_id)
    step = 1 << 30
    for s in range(0, nbytes, step):
        e = min(nbytes, s + step)
        tmp = torch.empty(e - s, dtype=torch.uint8, device="cuda")
        wl.fill_values(tmp, shape.dtype, g)
        torch.from_numpy(hb_array[s:e]).copy_(tmp)


def _compare_pool(t, exp_pool, what, layers=None):
    KV, L = t.shape[:2]
    buf = torch.empty(t.shape[2:], dtype=torch.uint8, pin_memory=True)
    for k in range(KV):
        for l in (range(L) if layers is None else layers):
            got = pinned_copy(t[k, l], buf)
            if not np.array_equal(got, exp_pool.pools[k][l]):
                bad = np.argwhere(got != exp_pool.pools[k][l])
                raise AssertionError(f"{what}: kv {k} layer {l}: {len(bad)} bytes differ, "
                                     f"first at {bad[0].tolist()}")


def _requests(reqs):
    return Requests([r.page_table for r in reqs], [r.n_tokens for r in reqs])


# ----------------------------------------------------------------------------- llama8b

def test_llama8b_full_size_all_paths(ctx):
    w = wl.llama8b()
    s = w.shape
    N = w.store_bytes()
    assert N == 4 << 30
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)  # pre-transfer state, pinned
    host_pool = hp.pool
    src, dst = _requests(w.store_requests), _requests(w.load_requests)
    nbytes = w.store_arena_bytes
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream

    # store (pages -> mapped pinned host chunks)
    arena = kvx.HostBuffer(nbytes + 4096)
    arena.array[:] = CANARY
    kvx.kvx_store_chunks(ctx, kvx.Pool.from_tensor(pools, s.page_size), src.array,
                         kvx.chunks_array(w.store_chunks, arena.ptr), stream=sh)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    expect = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(host_pool, src.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(arena.array, expect, "llama8b store")

    # HBM gather into device chunks
    dchunk = torch.full((nbytes + 4096,), CANARY, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()  # filled on the current stream; the transform runs on another
    kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, kvx.Pool.from_tensor(pools, s.page_size),
                          src.array, kvx.chunks_array(w.store_chunks, dchunk.data_ptr()),
                          stream=sh)
    stream.synchronize()
    assert_bytes_equal(pinned_copy(dchunk), expect, "llama8b HBM gather")

    # DMA baseline store into a second host arena
    arena2 = kvx.HostBuffer(nbytes + 4096)
    arena2.array[:] = CANARY
    n = kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_GATHER, kvx.Pool.from_tensor(pools, s.page_size),
                             src.array, kvx.chunks_array(w.store_chunks, arena2.ptr), stream=sh)
    stream.synchronize()
    assert n == 131072
    assert_bytes_equal(arena2.array, expect, "llama8b DMA store")
    arena2.close()

    # load (host chunks -> the disjoint fresh page set)
    kvx.kvx_load_chunks(ctx, kvx.Pool.from_tensor(pools, s.page_size), dst.array,
                        kvx.chunks_array(w.load_chunks, arena.ptr), stream=sh)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    oracle.load(host_pool, dst.oracle(), oracle_chunks(w.load_chunks, arena.array), threads=16)
    _compare_pool(pools, host_pool, "llama8b load")

    # HBM scatter and DMA load into two further disjoint page sets
    used = np.concatenate([src.host[0], dst.host[0]])
    free = np.setdiff1d(np.arange(s.num_pages, dtype=np.int32), used)
    free = np.random.default_rng(w.seed).permutation(free).astype(np.int32)
    third = Requests([free[:2048]], [32768])
    fourth = Requests([free[2048:4096]], [32768])
    kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, kvx.Pool.from_tensor(pools, s.page_size),
                          third.array, kvx.chunks_array(w.load_chunks, dchunk.data_ptr()),
                          stream=sh)
    n = kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_SCATTER, kvx.Pool.from_tensor(pools, s.page_size),
                             fourth.array, kvx.chunks_array(w.load_chunks, arena.ptr), stream=sh)
    stream.synchronize()
    assert n == 131072
    assert kvx.kvx_get_status(ctx, sh) == 0
    oracle.load(host_pool, third.oracle(), oracle_chunks(w.load_chunks, expect), threads=16)
    oracle.load(host_pool, fourth.oracle(), oracle_chunks(w.load_chunks, arena.array), threads=16)
    _compare_pool(pools, host_pool, "llama8b HBM scatter + DMA load")
    arena.close()
    hp.close()


def test_llama8b_pipelined_round_trip_as_benchmarked(ctx):
    """The headline step exactly as bench.py runs it: exchange launches that each store one
    chunk group and load the previous one, two steps back to back (the pipeline carries over
    the step boundary), then the flush of the last load."""
    import bench
    w = wl.llama8b()
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    src, dst = _requests(w.store_requests), _requests(w.load_requests)
    arena = kvx.HostBuffer(w.store_arena_bytes + 4096)
    arena.array[:] = CANARY
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    rt = bench.RoundTrip(kvx, ctx, pool, src.array, dst.array,
                         kvx.chunks_array(w.store_chunks, arena.ptr), s.num_layers,
                         kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_EXCHANGE), 8,
                         torch.device("cuda", 0))
    rt.step()
    rt.step()
    rt.flush()
    torch.cuda.synchronize()
    assert kvx.kvx_get_status(ctx, rt.stream.cuda_stream) == 0
    expect = np.full(w.store_arena_bytes + 4096, CANARY, np.uint8)
    oracle.store(hp.pool, src.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(arena.array, expect, "llama8b pipelined store")
    oracle.load(hp.pool, dst.oracle(), oracle_chunks(w.load_chunks, expect), threads=16)
    _compare_pool(pools, hp.pool, "llama8b pipelined load")
    arena.close()
    hp.close()


def test_llama8b_roundtrip_in_one_launch_as_benchmarked(ctx):
    """The headline step exactly as bench.py runs it: one kvx_roundtrip_chunks launch that
    stores every chunk and loads it into the fresh page set, twice in a row, in the
    library's default launch configuration."""
    w = wl.llama8b()
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    src, dst = _requests(w.store_requests), _requests(w.load_requests)
    arena = kvx.HostBuffer(w.store_arena_bytes + 4096)
    arena.array[:] = CANARY
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    chunks = kvx.chunks_array(w.store_chunks, arena.ptr)
    stream = torch.cuda.Stream()
    for _ in range(2):
        kvx.kvx_roundtrip_chunks(ctx, pool, src.array, dst.array, chunks,
                                 stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    expect = np.full(w.store_arena_bytes + 4096, CANARY, np.uint8)
    oracle.store(hp.pool, src.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(arena.array, expect, "llama8b round-trip store")
    oracle.load(hp.pool, dst.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    _compare_pool(pools, hp.pool, "llama8b round-trip load")
    arena.close()
    hp.close()


# ----------------------------------------------------------------------------- llama70b

def _io_cfg(ctx, op, cap, mapping=None, stages=0, stage_bytes=0):
    c = kvx.kvx_default_launch_cfg(ctx, op)
    c.sm_cap = cap
    if mapping is not None:
        c.mapping, c.threads, c.unroll, c.stage_bytes = mapping, 0, stages, stage_bytes
    return c


@pytest.mark.parametrize("mapping", ["bulk", "segment"])
def test_llama8b_store_and_load_on_4_sms_as_benchmarked(ctx, mapping):
    """The full request stored and loaded on 4 SMs, in the launch configurations the bench's
    4-SM legs time: the bulk mapping (store: two rings of 6 x 16 KiB, load: 3 x 32 KiB) and
    the register mapping capped to 4 SMs."""
    w = wl.llama8b()
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    src, dst = _requests(w.store_requests), _requests(w.load_requests)
    nbytes = w.store_arena_bytes
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    if mapping == "bulk":
        cs = _io_cfg(ctx, kvx.KVX_OP_STORE, 4, kvx.KVX_MAP_BULK, 6, 16384)
        cl = _io_cfg(ctx, kvx.KVX_OP_LOAD, 4, kvx.KVX_MAP_BULK, 3, 32768)
    else:
        cs = _io_cfg(ctx, kvx.KVX_OP_STORE, 4)
        cl = _io_cfg(ctx, kvx.KVX_OP_LOAD, 4)
    arena = kvx.HostBuffer(nbytes + 4096)
    arena.array[:] = CANARY
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    torch.cuda.synchronize()
    kvx.kvx_store_chunks(ctx, pool, src.array, kvx.chunks_array(w.store_chunks, arena.ptr), 0,
                         s.num_layers, cs, sh)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    expect = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(hp.pool, src.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(arena.array, expect, f"llama8b store, {mapping}, 4 SMs")
    kvx.kvx_load_chunks(ctx, pool, dst.array, kvx.chunks_array(w.load_chunks, arena.ptr), 0,
                        s.num_layers, cl, sh)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    oracle.load(hp.pool, dst.oracle(), oracle_chunks(w.load_chunks, arena.array), threads=16)
    _compare_pool(pools, hp.pool, f"llama8b load, {mapping}, 4 SMs")
    arena.close()
    hp.close()


@pytest.mark.parametrize("tokens_per_chunk,mapping", [(256, None), (512, None),
                                                      (256, "bulk")])
def test_llama70b_layer_streamed_load_full_size(ctx, tokens_per_chunk, mapping):
    """80 per-layer loads on a high-priority stream, as the streamed prefill issues them;
    per-layer chunks of 256 tokens (1 MiB, the closed form) and of 512 tokens (2 MiB); and
    the bulk mapping on 5 SMs that the bench streams beside GEMMs."""
    w = wl.llama70b(tokens_per_chunk=tokens_per_chunk)
    s = w.shape
    assert w.load_bytes() == 20 << 30
    assert all(c.nbytes(s) == tokens_per_chunk * 4096 for c in w.load_chunks)
    pools = _pools(s, w.seed, fill=CANARY)
    dst = _requests(w.load_requests)
    nbytes = w.load_arena_bytes
    arena = kvx.HostBuffer(nbytes)
    _fill_host(arena.array, nbytes, s, w.seed, stream_id=1)
    per_layer = [[c for c in w.load_chunks if c.layer_begin == l] for l in range(s.num_layers)]
    arrays = [kvx.chunks_array(cs, arena.ptr) for cs in per_layer]
    stream = torch.cuda.Stream(priority=-1)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    cfg = None if mapping is None else _io_cfg(ctx, kvx.KVX_OP_LOAD, 5, kvx.KVX_MAP_BULK)
    torch.cuda.synchronize()
    for l in range(s.num_layers):
        kvx.kvx_load_chunks(ctx, pool, dst.array, arrays[l], l, l + 1, cfg,
                            stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp_layer = [np.empty((s.num_pages, s.page_size, s.token_bytes), np.uint8) for _ in range(2)]
    buf = torch.empty(pools.shape[2:], dtype=torch.uint8, pin_memory=True)
    for l in range(s.num_layers):
        for e in exp_layer:
            e[:] = CANARY
        opool = oracle.Pool([[exp_layer[k] if i == l else None for i in range(s.num_layers)]
                             for k in range(2)], s.page_size)
        oracle.load(opool, dst.oracle(), oracle_chunks(per_layer[l], arena.array), l, l + 1,
                    threads=16)
        for k in range(2):
            got = pinned_copy(pools[k, l], buf)
            assert np.array_equal(got, exp_layer[k]), f"llama70b layer {l} kv {k}"
    arena.close()


# ----------------------------------------------------------------------------- qwen7b_batch

@pytest.mark.parametrize("placement", ["streams", "store_16sm", "store_6sm", "partitions"])
def test_qwen7b_batched_concurrent_load_and_store_full_size(ctx, placement):
    """The batched load and store at once on two plain streams (default grids, or the store
    on 16 or 6 SMs), or on the streams of two 16-SM I/O partitions (green contexts), as the
    bench measures them."""
    w = wl.qwen7b_batch()
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    host_pool = hp.pool
    reqs = _requests(w.load_requests)
    ld = kvx.HostBuffer(w.load_arena_bytes)
    _fill_host(ld.array, w.load_arena_bytes, s, w.seed, stream_id=2)
    st = kvx.HostBuffer(w.store_arena_bytes + 4096)
    st.array[:] = CANARY
    ctx2 = kvx.kvx_create(0, 64 << 20)  # one context per concurrent stream
    part = None
    try:
        cl = cs = None
        if placement == "partitions":
            part = kvx.kvx_partition_create(0, 16, -1, 0, io_groups=2)
            sa = torch.cuda.ExternalStream(part.io_streams[0])
            sb = torch.cuda.ExternalStream(part.io_streams[1])
            cl = _io_cfg(ctx, kvx.KVX_OP_LOAD, 0)  # each partition bounds its kernel's SMs
            cs = _io_cfg(ctx2, kvx.KVX_OP_STORE, 0)
        else:
            sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
            if placement in ("store_16sm", "store_6sm"):
                cs = _io_cfg(ctx2, kvx.KVX_OP_STORE, int(placement[6:-2]))
        pool = kvx.Pool.from_tensor(pools, s.page_size)
        torch.cuda.synchronize()
        kvx.kvx_load_chunks(ctx, pool, reqs.array, kvx.chunks_array(w.load_chunks, ld.ptr),
                            cfg=cl, stream=sa.cuda_stream)
        kvx.kvx_store_chunks(ctx2, pool, reqs.array, kvx.chunks_array(w.store_chunks, st.ptr),
                             cfg=cs, stream=sb.cuda_stream)
        torch.cuda.synchronize()
        assert kvx.kvx_get_status(ctx, sa.cuda_stream) == 0
        assert kvx.kvx_get_status(ctx2, sb.cuda_stream) == 0
    finally:
        kvx.kvx_destroy(ctx2)
        if part is not None:
            torch.cuda.synchronize()
            part.close()
    expect = np.full(w.store_arena_bytes + 4096, CANARY, np.uint8)
    oracle.store(host_pool, reqs.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(st.array, expect, "qwen7b batched store")
    oracle.load(host_pool, reqs.oracle(), oracle_chunks(w.load_chunks, ld.array), threads=16)
    _compare_pool(pools, host_pool, "qwen7b batched load")
    ld.close()
    st.close()
    hp.close()


def test_qwen7b_batched_partial_hits_in_one_exchange_launch(ctx):
    """The batched load and store of the 64 partial-hit requests in one exchange launch."""
    w = wl.qwen7b_batch()
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    reqs = _requests(w.load_requests)
    ld = kvx.HostBuffer(w.load_arena_bytes)
    _fill_host(ld.array, w.load_arena_bytes, s, w.seed, stream_id=2)
    st = kvx.HostBuffer(w.store_arena_bytes + 4096)
    st.array[:] = CANARY
    sh = torch.cuda.current_stream().cuda_stream
    kvx.kvx_exchange_chunks(ctx, kvx.Pool.from_tensor(pools, s.page_size), reqs.array,
                            kvx.chunks_array(w.store_chunks, st.ptr), reqs.array,
                            kvx.chunks_array(w.load_chunks, ld.ptr), stream=sh)
    torch.cuda.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    expect = np.full(w.store_arena_bytes + 4096, CANARY, np.uint8)
    oracle.store(hp.pool, reqs.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(st.array, expect, "qwen7b exchange store")
    oracle.load(hp.pool, reqs.oracle(), oracle_chunks(w.load_chunks, ld.array), threads=16)
    _compare_pool(pools, hp.pool, "qwen7b exchange load")
    ld.close()
    st.close()
    hp.close()


# ----------------------------------------------------------------------------- mla_sweep

@pytest.mark.parametrize("page_size", wl.MLA_PAGE_SIZES)
@pytest.mark.parametrize("chunk_bytes", wl.MLA_CHUNK_BYTES)
def test_mla_sweep_cell_full_size(ctx, page_size, chunk_bytes):
    w = wl.mla_sweep(page_size, chunk_bytes)
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    host_pool = hp.pool
    src, dst = _requests(w.store_requests), _requests(w.load_requests)
    nbytes = w.store_arena_bytes
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    sh = torch.cuda.current_stream().cuda_stream
    expect = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(host_pool, src.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    for how in ("kernel", "dma"):
        arena = kvx.HostBuffer(nbytes + 4096)
        arena.array[:] = CANARY
        ch = kvx.chunks_array(w.store_chunks, arena.ptr)
        if how == "kernel":
            kvx.kvx_store_chunks(ctx, pool, src.array, ch, stream=sh)
        else:
            kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_GATHER, pool, src.array, ch, stream=sh)
        torch.cuda.synchronize()
        assert_bytes_equal(arena.array, expect, f"mla P={page_size} C={chunk_bytes} {how} store")
        arena.close()
    # Loads: the kernel into the disjoint page set, then the DMA baseline back into it
    # after clearing it, each checked against the oracle.
    arena = kvx.HostBuffer(nbytes + 4096)
    arena.array[:] = expect
    ch = kvx.chunks_array(w.load_chunks, arena.ptr)
    oracle.load(host_pool, dst.oracle(), oracle_chunks(w.load_chunks, arena.array), threads=16)
    for how in ("kernel", "dma"):
        idx = torch.from_numpy(dst.host[0]).long().cuda()
        pools[:, :, idx] = CANARY
        if how == "kernel":
            kvx.kvx_load_chunks(ctx, pool, dst.array, ch, stream=sh)
        else:
            kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_SCATTER, pool, dst.array, ch, stream=sh)
        torch.cuda.synchronize()
        assert kvx.kvx_get_status(ctx, sh) == 0
        _compare_pool(pools, host_pool, f"mla P={page_size} C={chunk_bytes} {how} load")
    arena.close()
    hp.close()


# ----------------------------------------------------------------------------- mla_blocks

def test_mla_block_objects_store_and_per_layer_load(ctx):
    """Per-block STRIPED chunks (one 4096-aligned object per layer): one store of every
    layer, then one load call per layer (layer window [l, l+1)), as a per-layer retrieve of
    block objects issues them."""
    w = wl.mla_blocks(16)
    s = w.shape
    pools = _pools(s, w.seed)
    hp = HostPool(pools, s.page_size)
    src, dst = _requests(w.store_requests), _requests(w.load_requests)
    nbytes = w.store_arena_bytes
    arena = kvx.HostBuffer(nbytes + 4096)
    arena.array[:] = CANARY
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    stream = torch.cuda.Stream(priority=-1)
    sh = stream.cuda_stream
    ch = kvx.chunks_array(w.store_chunks, arena.ptr)
    kvx.kvx_store_chunks(ctx, pool, src.array, ch, stream=sh)
    stream.synchronize()
    expect = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(hp.pool, src.oracle(), oracle_chunks(w.store_chunks, expect), threads=16)
    assert_bytes_equal(arena.array, expect, "mla block objects store")
    for l in range(s.num_layers):
        kvx.kvx_load_chunks(ctx, pool, dst.array, ch, l, l + 1, stream=sh)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    oracle.load(hp.pool, dst.oracle(), oracle_chunks(w.load_chunks, arena.array), threads=16)
    _compare_pool(pools, hp.pool, "mla block objects per-layer load")
    arena.close()
    hp.close()
