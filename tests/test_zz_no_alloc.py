"""kvx_load_chunks_noalloc against kvx_load_chunks, through the C ABI.

The allocation-free load is for callers that may not allocate device memory (an engine
that gave nearly all of HBM to its KV page pool, or a plug-in with nowhere to keep a
context).  It must write exactly the bytes the context-based load writes, call after
call, although every call reuses the same fixed scratch array inside the library.  This
file is collected last so that a stop at the first failure has run everything else.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_gather_gb300.build import build  # noqa: E402

build()
from paged_kv_gather_gb300 import kvx  # noqa: E402
from paged_kv_gather_gb300 import workloads as wl  # noqa: E402


def _batch(seed, n_req, max_tokens, L=3, KV=2, P=16, v=512, tpc=96, min_tokens=1):
    """Random requests on disjoint pages, layer-major and token-major chunks of host bytes."""
    rng = np.random.default_rng(seed)
    lens = [int(rng.integers(min_tokens, max_tokens)) for _ in range(n_req)]
    pages = [-(-n // P) for n in lens]
    num_pages = sum(pages) + 8
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


def _pools(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    t = torch.randint(0, 256, (shape.kv_factor, shape.num_layers, shape.num_pages,
                               shape.page_size, shape.token_bytes), generator=g,
                      device="cuda", dtype=torch.int16).to(torch.uint8)
    return t, t.clone()


def test_noalloc_load_matches_context_load_two_calls_in_a_row():
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    host_bufs = []
    try:
        # Two different batches back to back on one stream, the second smaller than the
        # first, so descriptors left in the shared array by call 1 would show in call 2.
        for call, (n_req, max_tokens) in enumerate(((3, 900), (2, 300))):
            shape, lens, tables, specs, nbytes, rng = _batch(100 + call, n_req, max_tokens)
            ref_pool, new_pool = _pools(shape, 200 + call)
            host = kvx.HostBuffer(nbytes)
            host_bufs.append(host)
            host.array[:] = rng.integers(0, 256, nbytes, dtype=np.uint8)
            dev_tables = [torch.from_numpy(t).cuda() for t in tables]
            reqs = kvx.requests_array([(d.data_ptr(), t, n)
                                       for d, t, n in zip(dev_tables, tables, lens)])
            chunks = kvx.chunks_array(specs, host.ptr)
            ref = kvx.Pool.from_tensor(ref_pool, shape.page_size)
            new = kvx.Pool.from_tensor(new_pool, shape.page_size)
            torch.cuda.synchronize()  # pools and flags were written on the current stream
            kvx.kvx_load_chunks(ctx, ref, reqs, chunks, 0, shape.num_layers, None,
                                stream.cuda_stream)
            kvx.kvx_load_chunks_noalloc(new, reqs, chunks, 0, shape.num_layers, None,
                                        stream.cuda_stream, flags.data_ptr())
            stream.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            assert int(flags.item()) == 0
            assert torch.equal(ref_pool, new_pool), f"call {call + 1} differs"
            # The load really wrote something: the chunk bytes sit in the pages.
            t0 = torch.from_numpy(tables[0]).long().cuda()
            assert not torch.equal(new_pool[:, :, t0], _pools(shape, 200 + call)[0][:, :, t0])
    finally:
        for h in host_bufs:
            h.close()
        kvx.kvx_destroy(ctx)


def test_noalloc_load_reports_bad_pages_and_rejects_oversized_batches():
    shape, lens, tables, specs, nbytes, rng = _batch(300, 1, 200, min_tokens=64)
    assert len(tables[0]) >= 4  # the bad page is one of several
    pool_t, _ = _pools(shape, 301)
    before = pool_t.clone()
    host = kvx.HostBuffer(nbytes)
    try:
        bad = tables[0].copy()
        bad[-1] = shape.num_pages + 7  # the kernel skips this page and flags it
        dev = torch.from_numpy(bad).cuda()
        reqs = kvx.requests_array([(dev.data_ptr(), None, lens[0])])
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        pool = kvx.Pool.from_tensor(pool_t, shape.page_size)
        kvx.kvx_load_chunks_noalloc(pool, reqs, kvx.chunks_array(specs, host.ptr), 0,
                                    shape.num_layers, None, 0, flags.data_ptr())
        torch.cuda.synchronize()
        assert int(flags.item()) == kvx.KVX_DEV_PAGE_OUT_OF_RANGE
        # A batch whose descriptors exceed the fixed array is refused before any launch.
        many = [wl.ChunkSpec(0, i % lens[0], 1, 0, 1, 0, 0) for i in range(20000)]
        big = kvx.chunks_array(many, host.ptr)
        assert len(many) * 56 > kvx.KVX_NOALLOC_SCRATCH_BYTES  # 56-byte chunk descriptors
        snapshot = pool_t.clone()
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_load_chunks_noalloc(pool, reqs, big, 0, 1, None, 0, 0)
        assert e.value.status == kvx.KVX_ERR_CAPACITY
        torch.cuda.synchronize()
        assert torch.equal(snapshot, pool_t)
        assert not torch.equal(before, pool_t)
    finally:
        host.close()
