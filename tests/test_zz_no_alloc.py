"""kvx_load_chunks_noalloc against the CPU oracle and kvx_load_chunks, through the C ABI.

The allocation-free load is for callers that may not allocate device memory (an engine
that gave nearly all of HBM to its KV page pool, or a plug-in with nowhere to keep a
context).  Every call must write exactly the bytes the oracle writes, and the same bytes
the context-based load writes, call after call, although all calls reuse one fixed scratch
array inside the library.  This file is collected last so that a stop at the first failure
has run everything else.
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
from tests.gpu_common import (CANARY, DevicePool, Requests, assert_pool_equal,  # noqa: E402
                              expected_load, oracle_chunks)


def _batch(seed, n_req, max_tokens, L=3, KV=2, P=16, v=512, tpc=96, min_tokens=1, spare=8):
    """Random requests on disjoint pages, layer-major and token-major chunks of host bytes."""
    rng = np.random.default_rng(seed)
    lens = [int(rng.integers(min_tokens, max_tokens)) for _ in range(n_req)]
    pages = [-(-n // P) for n in lens]
    num_pages = sum(pages) + spare
    perm = rng.permutation(num_pages).astype(np.int32)
    tables, at = [], 0
    for npg in pages:
        tables.append(perm[at:at + npg].copy())
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, tpc, 0, L, r % 2)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, num_pages)
    wl.place_chunks(specs, shape)
    return shape, lens, tables, specs, wl._arena_bytes(specs, shape), rng


def _pool(shape, random_seed=None):
    """A device pool of canary bytes, or of random bytes when random_seed is given."""
    p = DevicePool.empty(shape.num_layers, shape.kv_factor, shape.num_pages, shape.page_size,
                         shape.token_bytes)
    if random_seed is not None:
        p.fill_random(random_seed)
    return p


def test_noalloc_load_matches_oracle_and_context_load_two_calls_in_a_row():
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    host_bufs = []
    try:
        # Two different batches back to back on one stream, the second smaller than the
        # first, so descriptors left in the shared array by call 1 would show in call 2.
        # Call 1 writes into canary-filled pools, call 2 into pools of random bytes: every
        # byte outside the destination slots must keep its value.
        for call, (n_req, max_tokens, seed) in enumerate(((3, 900, None), (2, 300, 77))):
            shape, lens, tables, specs, nbytes, rng = _batch(100 + call, n_req, max_tokens)
            ctx_pool = _pool(shape, seed)
            new_pool = _pool(shape, seed)
            pre = new_pool.host_copy()
            host = kvx.HostBuffer(nbytes)
            host_bufs.append(host)
            host.array[:] = rng.integers(0, 256, nbytes, dtype=np.uint8)
            reqs = Requests(tables, lens)
            chunks = kvx.chunks_array(specs, host.ptr)
            torch.cuda.synchronize()  # page tables were copied on the current stream
            kvx.kvx_load_chunks(ctx, ctx_pool.pool, reqs.array, chunks, 0, shape.num_layers,
                                None, stream.cuda_stream)
            kvx.kvx_load_chunks_noalloc(new_pool.pool, reqs.array, chunks, 0, shape.num_layers,
                                        None, stream.cuda_stream, flags.data_ptr())
            stream.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            assert int(flags.item()) == 0
            exp = expected_load(pre, reqs, specs, host.array.copy())
            assert_pool_equal(new_pool, exp)  # the oracle, byte for byte
            assert torch.equal(ctx_pool.tensor, new_pool.tensor), f"call {call + 1}"
            # The load really wrote something: the chunk bytes sit in the pages.
            t0 = torch.from_numpy(tables[0]).long().cuda()
            assert not torch.equal(new_pool.tensor[:, :, t0], _pool(shape, seed).tensor[:, :, t0])
    finally:
        for h in host_bufs:
            h.close()
        kvx.kvx_destroy(ctx)


def test_noalloc_load_without_a_flags_word_skips_a_bad_page_like_the_context_load():
    """device_flags NULL: the kernel reports into the array's own status word; a page id
    past the pool is skipped there exactly as the context load skips it, and every other
    byte matches the oracle (run on a host pool with one extra page that takes the writes
    aimed at the bad id)."""
    shape, lens, tables, specs, nbytes, rng = _batch(400, 2, 500, min_tokens=100, spare=0)
    bad = [t.copy() for t in tables]
    bad[0][1] = shape.num_pages  # outside the pool: skipped by the kernel
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    host = kvx.HostBuffer(nbytes)
    try:
        host.array[:] = rng.integers(0, 256, nbytes, dtype=np.uint8)
        reqs = Requests(bad, lens, host_copy=False)
        chunks = kvx.chunks_array(specs, host.ptr)
        ctx_pool, new_pool = _pool(shape, 401), _pool(shape, 401)
        pre = new_pool.host_copy()
        torch.cuda.synchronize()  # page tables were copied on the current stream
        kvx.kvx_load_chunks(ctx, ctx_pool.pool, reqs.array, chunks, 0, shape.num_layers, None,
                            stream.cuda_stream)
        kvx.kvx_load_chunks_noalloc(new_pool.pool, reqs.array, chunks, 0, shape.num_layers,
                                    None, stream.cuda_stream, 0)
        stream.synchronize()
        # The context load saw the bad page in its own status word.
        assert kvx.kvx_get_status(ctx, stream.cuda_stream) == kvx.KVX_DEV_PAGE_OUT_OF_RANGE
        assert torch.equal(ctx_pool.tensor, new_pool.tensor)
        # Oracle: the same pool plus one spare page that stands for the bad id.
        ext = oracle.Pool([[np.concatenate([a, np.full((1,) + a.shape[1:], CANARY, np.uint8)])
                            for a in row] for row in pre.pools], shape.page_size)
        oracle.load(ext, Requests(bad, lens).oracle(), oracle_chunks(specs, host.array.copy()))
        exp = oracle.Pool([[a[:shape.num_pages] for a in row] for row in ext.pools],
                          shape.page_size)
        assert_pool_equal(new_pool, exp)
        # The valid part moved: the first page of request 0 now holds chunk bytes.
        assert not torch.equal(new_pool.tensor[:, :, int(tables[0][0])],
                               _pool(shape, 401).tensor[:, :, int(tables[0][0])])
    finally:
        host.close()
        kvx.kvx_destroy(ctx)


def test_noalloc_load_reports_bad_pages_and_rejects_oversized_batches():
    shape, lens, tables, specs, nbytes, rng = _batch(300, 1, 200, min_tokens=64)
    assert len(tables[0]) >= 4  # the bad page is one of several
    pool = _pool(shape, 301)
    before = pool.tensor.clone()
    host = kvx.HostBuffer(nbytes)
    try:
        bad = tables[0].copy()
        bad[-1] = shape.num_pages + 7  # the kernel skips this page and flags it
        reqs = Requests([bad], lens, host_copy=False)
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        kvx.kvx_load_chunks_noalloc(pool.pool, reqs.array, kvx.chunks_array(specs, host.ptr), 0,
                                    shape.num_layers, None, 0, flags.data_ptr())
        torch.cuda.synchronize()
        assert int(flags.item()) == kvx.KVX_DEV_PAGE_OUT_OF_RANGE
        # A batch whose descriptors exceed the fixed array is refused before any launch.
        many = [wl.ChunkSpec(0, i % lens[0], 1, 0, 1, 0, 0) for i in range(20000)]
        big = kvx.chunks_array(many, host.ptr)
        assert len(many) * 64 > kvx.KVX_NOALLOC_SCRATCH_BYTES  # 64 bytes per chunk
        snapshot = pool.tensor.clone()
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_load_chunks_noalloc(pool.pool, reqs.array, big, 0, 1, None, 0, 0)
        assert e.value.status == kvx.KVX_ERR_CAPACITY
        torch.cuda.synchronize()
        assert torch.equal(snapshot, pool.tensor)
        assert not torch.equal(before, pool.tensor)
    finally:
        host.close()


def test_noalloc_load_refuses_a_capturing_stream():
    """Its descriptor copy reads a host image that the next call overwrites, so a stream
    under capture is refused before anything is recorded or moved."""
    shape, lens, tables, specs, nbytes, rng = _batch(500, 1, 300, min_tokens=32)
    pool = _pool(shape, 501)
    host = kvx.HostBuffer(nbytes)
    try:
        host.array[:] = rng.integers(0, 256, nbytes, dtype=np.uint8)
        reqs = Requests(tables, lens)
        chunks = kvx.chunks_array(specs, host.ptr)
        snapshot = pool.tensor.clone()
        torch.cuda.synchronize()
        dummy = torch.zeros(1, device="cuda")
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            with pytest.raises(kvx.KvxError) as e:
                kvx.kvx_load_chunks_noalloc(pool.pool, reqs.array, chunks, 0, shape.num_layers,
                                            None, s.cuda_stream, 0)
            dummy.add_(1)  # the capture itself goes on normally
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
        g.replay()
        torch.cuda.synchronize()
        assert float(dummy.item()) == 1.0
        assert torch.equal(snapshot, pool.tensor)
        # Outside capture the same call moves the bytes.
        kvx.kvx_load_chunks_noalloc(pool.pool, reqs.array, chunks, 0, shape.num_layers, None,
                                    0, 0)
        torch.cuda.synchronize()
        assert not torch.equal(snapshot, pool.tensor)
    finally:
        host.close()
