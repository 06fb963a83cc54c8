"""GPU parity: every kernel path against the CPU oracle, byte for byte (small and ragged).

All transfers go through the C ABI (libkvx.so) via the ctypes binding; expected bytes come
from the oracle run on host copies of the same seeded inputs.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts too; every test here is gpu-marked
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_gather_gb300.build import build  # noqa: E402

build()
import oracle  # noqa: E402
from paged_kv_gather_gb300 import kvx  # noqa: E402
from paged_kv_gather_gb300 import workloads as wl  # noqa: E402
from tests.gpu_common import (CANARY, Arena, DevicePool, Requests, assert_bytes_equal,  # noqa: E402
                              assert_pool_equal, bulk, cfg, expected_load, expected_store,
                              oracle_chunks, random_case)


@pytest.fixture(scope="module")
def ctx():
    c = kvx.kvx_create(0, 64 << 20)
    yield c
    kvx.kvx_destroy(c)


@pytest.fixture
def stream():
    s = torch.cuda.Stream()
    yield s
    s.synchronize()


def _store(ctx, op, dpool, reqs, specs, arena, lb, le, c, stream):
    ch = kvx.chunks_array(specs, arena.ptr)
    if op == "store":
        kvx.kvx_store_chunks(ctx, dpool.pool, reqs.array, ch, lb, le, c, stream.cuda_stream)
    elif op == "gather":
        kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, dpool.pool, reqs.array, ch, lb, le, c,
                              stream.cuda_stream)
    else:
        kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_GATHER, dpool.pool, reqs.array, ch, lb, le,
                             stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0


def _load(ctx, op, dpool, reqs, specs, arena, lb, le, c, stream):
    ch = kvx.chunks_array(specs, arena.ptr)
    if op == "load":
        kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array, ch, lb, le, c, stream.cuda_stream)
    elif op == "scatter":
        kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, dpool.pool, reqs.array, ch, lb, le, c,
                              stream.cuda_stream)
    else:
        kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_SCATTER, dpool.pool, reqs.array, ch, lb, le,
                             stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0


# ----------------------------------------------------------------------------- tiny workload

@pytest.mark.parametrize("op_store,op_load,where", [("store", "load", "host"),
                                                    ("gather", "scatter", "device"),
                                                    ("dma", "dma", "host")])
def test_tiny_workload_round_trip(ctx, stream, op_store, op_load, where):
    """tiny: token-major chunk; store from one random page set, load into a disjoint one."""
    w = wl.tiny()
    s = w.shape
    dpool = DevicePool.empty(s.num_layers, s.kv_factor, s.num_pages, s.page_size, s.token_bytes)
    g = wl.values_generator(w.seed, "cuda")
    wl.fill_values(dpool.tensor, s.dtype, g)
    src = Requests([r.page_table for r in w.store_requests], [r.n_tokens for r in w.store_requests])
    arena = Arena(w.store_arena_bytes, where)
    _store(ctx, op_store, dpool, src, w.store_chunks, arena, 0, None, cfg(), stream)
    exp = expected_store(dpool, src, w.store_chunks, w.store_arena_bytes)
    assert_bytes_equal(arena.numpy(), exp, f"tiny {op_store}")

    dst = Requests([r.page_table for r in w.load_requests], [r.n_tokens for r in w.load_requests])
    pre = dpool.host_copy()
    _load(ctx, op_load, dpool, dst, w.load_chunks, arena, 0, None, cfg(), stream)
    exp_pool = expected_load(pre, dst, w.load_chunks, arena.numpy())
    assert_pool_equal(dpool, exp_pool)
    # The logical readback through the new page table equals the original.
    for k in range(s.kv_factor):
        for l in range(s.num_layers):
            a = dpool.tensor[k, l][torch.from_numpy(src.host[0]).long().cuda()]
            b = dpool.tensor[k, l][torch.from_numpy(dst.host[0]).long().cuda()]
            assert torch.equal(a, b)
    arena.close()


def cta(sm_cap, ctas_per_sm, threads, unroll, hint):
    """Launch configuration of the CTA-per-segment mapping."""
    return cfg(sm_cap, ctas_per_sm, threads, unroll, hint, kvx.KVX_MAP_CTA)


# ----------------------------------------------------------------------------- random batches

CONFIGS = [cfg(), cfg(1, 1, 32, 1, 0), cfg(2, 1, 64, 2, 1), cfg(3, 2, 256, 4, 0),
           cfg(0, 1, 1024, 8, 1), cfg(1, 1, 1024, 8, 0), cfg(5, 3, 96, 4, 1),
           bulk(), bulk(2, 1, 2, 64), bulk(3, 2, 3, 4096), bulk(0, 1, 8, 1040),
           cfg(3, 1, 256, 8, 0, batch=32), cfg(2, 2, 128, 2, 1, batch=5),
           cfg(0, 1, 64, 4, 0, batch=2),
           cta(2, 1, 256, 8, 1), cta(1, 1, 32, 1, 0), cta(0, 2, 512, 4, 0), cta(3, 1, 96, 2, 1)]


@pytest.mark.parametrize("seed", range(42))
def test_random_batches_all_paths(ctx, stream, seed):
    rng = np.random.default_rng(5000 + seed)
    shape, lens, tables, load_tables, specs, lb, le = random_case(rng)
    L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size, shape.token_bytes,
                       shape.num_pages)
    c = CONFIGS[seed % len(CONFIGS)]
    arena_bytes = wl._arena_bytes(specs, shape)
    src = Requests(tables, lens)
    dst = Requests(load_tables, lens)
    for op_store, op_load, where in (("store", "load", "host"), ("gather", "scatter", "device"),
                                     ("dma", "dma", "host"), ("dma", "dma", "device")):
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(seed * 31 + 1)
        arena = Arena(arena_bytes, where)
        _store(ctx, op_store, dpool, src, specs, arena, lb, le, c, stream)
        exp = expected_store(dpool, src, specs, arena_bytes, lb, le)
        assert_bytes_equal(arena.numpy(), exp, f"seed {seed} {op_store}/{where}")
        # Load random chunk bytes into the disjoint page set of a random pool.
        data = rng.integers(0, 256, arena_bytes + 4096, dtype=np.uint8)
        arena.write(data)
        pre = dpool.host_copy()
        _load(ctx, op_load, dpool, dst, specs, arena, lb, le, c, stream)
        exp_pool = expected_load(pre, dst, specs, data.copy(), lb, le)
        assert_pool_equal(dpool, exp_pool)
        arena.close()


def test_random_launch_shapes(ctx, stream):
    """150 random batches, each under a random launch shape (SM cap, CTAs per SM, threads,
    unroll, hint, batch, sometimes the CTA mapping) through a store then load, a round trip
    or an exchange with a random share of the batch loaded."""
    for seed in range(150):
        rng = np.random.default_rng(90000 + seed)
        shape, lens, tables, load_tables, specs, lb, le = random_case(rng)
        L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size,
                           shape.token_bytes, shape.num_pages)
        c = cfg(int(rng.integers(0, 9)), int(rng.integers(1, 4)), 32 * int(rng.integers(1, 33)),
                int(rng.choice([1, 2, 4, 8])), int(rng.integers(0, 2)),
                batch=int(rng.choice([0, 0, 1, 2, 3, 7, 16, 32])))
        op = int(rng.integers(0, 3))  # 0 store + load, 1 round trip, 2 exchange
        if op == 0 and rng.random() < 0.3:
            c.mapping = kvx.KVX_MAP_CTA
        nbytes = wl._arena_bytes(specs, shape)
        src, dst = Requests(tables, lens), Requests(load_tables, lens)
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(seed)
        pre = dpool.host_copy()
        out = Arena(nbytes, "host")
        ch = kvx.chunks_array(specs, out.ptr)
        exp = np.full(nbytes + 4096, CANARY, np.uint8)
        oracle.store(pre, src.oracle(), oracle_chunks(specs, exp), lb, le)
        what = f"seed {seed} op {op} cfg {c.as_dict()}"
        if op == 0:
            kvx.kvx_store_chunks(ctx, dpool.pool, src.array, ch, lb, le, c, stream.cuda_stream)
            stream.synchronize()
            assert_bytes_equal(out.numpy(), exp, what)
            kvx.kvx_load_chunks(ctx, dpool.pool, dst.array, ch, lb, le, c, stream.cuda_stream)
            oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp), lb, le)
        elif op == 1:
            kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array, ch, lb, le, c,
                                     stream.cuda_stream)
            oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp), lb, le)
        else:
            inp = Arena(nbytes, "host")
            data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
            inp.write(data)
            lspecs = specs[:int(rng.integers(0, len(specs) + 1))]
            kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, ch, dst.array,
                                    kvx.chunks_array(lspecs, inp.ptr), lb, le, c,
                                    stream.cuda_stream)
            stream.synchronize()
            inp.close()
            oracle.load(pre, dst.oracle(), oracle_chunks(lspecs, data), lb, le)
        stream.synchronize()
        assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0, what
        assert_bytes_equal(out.numpy(), exp, what)
        assert_pool_equal(dpool, pre)
        out.close()


@pytest.mark.parametrize("unroll", [1, 2, 4, 8])
@pytest.mark.parametrize("hint", [0, 1])
@pytest.mark.parametrize("batch", [1, 7, 32])
@pytest.mark.parametrize("layout", ["layer", "token"])
def test_every_kernel_variant(ctx, stream, unroll, hint, batch, layout):
    """Every (unroll, hint, direction) instantiation, one and several segments resolved per
    warp, on a multi-tile ragged batch.  layout "token": token-major chunks over all layers
    (pages of strided rows, the row-walking kernel), with one layer-major chunk in the same
    launch so that kernel copies contiguous segments too."""
    rng = np.random.default_rng(77 + unroll * 10 + hint)
    L, KV, P, v = 3, 2, 16, 2048
    lens = [1000, 333, 17]
    pages = [-(-n // P) for n in lens]
    NP = sum(pages) * 2
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[at + sum(pages):at + sum(pages) + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        lay = wl.TOKEN_MAJOR if layout == "token" and r != 1 else wl.LAYER_MAJOR
        specs += wl.split_tokens(r, 0, n, 100, 0, L, lay)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    c = cfg(4, 1, 256, unroll, hint, batch=batch)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(unroll + 10 * hint + 100 * batch)
    arena = Arena(nbytes, "host")
    _store(ctx, "store", dpool, src, specs, arena, 0, None, c, stream)
    assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), "store")
    pre = dpool.host_copy()
    _load(ctx, "load", dpool, dst, specs, arena, 0, None, c, stream)
    assert_pool_equal(dpool, expected_load(pre, dst, specs, arena.numpy().copy()))
    arena.close()


@pytest.mark.parametrize("unroll", [1, 2, 4, 8])
@pytest.mark.parametrize("hint", [0, 1])
@pytest.mark.parametrize("layout", [wl.LAYER_MAJOR, wl.TOKEN_MAJOR])
def test_cta_mapping_every_variant(ctx, stream, unroll, hint, layout):
    """CTA-per-segment mapping: every (unroll, hint, direction) instantiation, more segments
    than one batch of 32 per CTA, a ragged last batch, partial pages and both contiguous and
    token-major chunk rows; store, load and the HBM transform."""
    rng = np.random.default_rng(91 + unroll * 10 + hint + 100 * layout)
    L, KV, P, v = 3, 2, 16, 1024
    lens = [1000, 333, 17]
    pages = [-(-n // P) for n in lens]
    NP = sum(pages) * 2
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[at + sum(pages):at + sum(pages) + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, 90, 0, L, layout)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    c = cta(2, 1, 160, unroll, hint)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    for op_store, op_load, where in (("store", "load", "host"), ("gather", "scatter", "device")):
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(unroll + 10 * hint + 1000 * layout)
        arena = Arena(nbytes, where)
        _store(ctx, op_store, dpool, src, specs, arena, 0, None, c, stream)
        assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), op_store)
        pre = dpool.host_copy()
        _load(ctx, op_load, dpool, dst, specs, arena, 0, None, c, stream)
        assert_pool_equal(dpool, expected_load(pre, dst, specs, arena.numpy().copy()))
        arena.close()


@pytest.mark.parametrize("layout", [wl.LAYER_MAJOR, wl.TOKEN_MAJOR, wl.STRIPED])
@pytest.mark.parametrize("unroll", [1, 8])
def test_small_transfers_cut_segments_into_row_slices(ctx, stream, layout, unroll):
    """A batch with fewer page segments than the grid has warps: each segment is cut into
    row slices, one per warp; partial pages leave some slices empty.  Store, load and a
    prepared plan, each against the oracle."""
    rng = np.random.default_rng(1300 + layout * 10 + unroll)
    L, KV, P, v = 2, 2, 16, 2048
    lens = [37, 19]  # 3 and 2 pages, the last ones partial (5 and 3 rows)
    pages = [-(-n // P) for n in lens]
    NP = 4 * sum(pages)
    perm = rng.permutation(NP).astype(np.int32)
    t_src = [perm[:3], perm[3:5]]
    t_dst = [perm[5:8], perm[8:10]]
    specs = [wl.ChunkSpec(0, 0, 37, 0, L, layout), wl.ChunkSpec(1, 0, 19, 0, L, layout)]
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape, align=wl.STRIPE_ALIGN)
    nbytes = wl._arena_bytes(specs, shape)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    c = cfg(4, 1, 1024, unroll, 0)  # 128 warps for 20 segments
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(1301 + layout)
    arena = Arena(nbytes, "host")
    _store(ctx, "store", dpool, src, specs, arena, 0, None, c, stream)
    segments = (3 + 2) * L * KV
    assert kvx.kvx_last_launch(ctx)[0] == segments
    assert kvx.kvx_last_launch(ctx)[1] * 32 > segments  # more warps than segments
    assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), "split store")
    pre = dpool.host_copy()
    _load(ctx, "load", dpool, dst, specs, arena, 0, None, c, stream)
    assert_pool_equal(dpool, expected_load(pre, dst, specs, arena.numpy().copy()))
    # The same load as a plan, into a third page set.
    third = Requests([perm[10:13], perm[13:15]], lens)
    plan = kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, dpool.pool, third.array,
                               kvx.chunks_array(specs, arena.ptr), cfg=c,
                               stream=stream.cuda_stream)
    pre = dpool.host_copy()
    kvx.kvx_plan_launch(plan, stream.cuda_stream)
    stream.synchronize()
    kvx.kvx_plan_destroy(plan)
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    assert_pool_equal(dpool, expected_load(pre, third, specs, arena.numpy().copy()))
    arena.close()


@pytest.mark.parametrize("stages,stage_bytes,ctas", [(2, 16, 1), (3, 1040, 2), (3, 32768, 1),
                                                    (8, 13312, 1), (2, 53248, 1)])
def test_bulk_mapping_multi_tile_ragged(ctx, stream, stages, stage_bytes, ctas):
    """The bulk-copy mapping on every direction: segments longer and shorter than a stage,
    chunk cuts inside pages, both layouts, host and device chunks."""
    rng = np.random.default_rng(900 + stages)
    L, KV, P, v = 3, 2, 16, 1152
    lens = [700, 129, 16]
    pages = [-(-n // P) for n in lens]
    NP = 2 * sum(pages) + 3
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[at + sum(pages):at + sum(pages) + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, 77, 0, L, r % 2)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    c = bulk(5, ctas, stages, stage_bytes)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    for op_s, op_l, where in (("store", "load", "host"), ("gather", "scatter", "device")):
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(stages * 7 + ctas)
        arena = Arena(nbytes, where)
        _store(ctx, op_s, dpool, src, specs, arena, 0, None, c, stream)
        assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), op_s)
        pre = dpool.host_copy()
        _load(ctx, op_l, dpool, dst, specs, arena, 0, None, c, stream)
        assert_pool_equal(dpool, expected_load(pre, dst, specs, arena.numpy().copy()))
        arena.close()


@pytest.mark.parametrize("table", ["consecutive", "random"])
def test_bulk_mapping_piece_cap_and_merged_runs(ctx, stream, table):
    """The bulk mapping's two packing rules against the oracle.  16-byte tokens in
    token-major chunks make every row its own piece, so each 32 KiB stage closes at its
    32-piece cap long before it is full.  Pages placed back to back in the pool
    ("consecutive") let pieces of neighbouring page segments merge into one bulk copy on the
    page side, while layer-major chunks merge them on the chunk side."""
    rng = np.random.default_rng(4242 if table == "random" else 4343)
    L, KV, P, v = 2, 2, 8, 16
    lens = [600, 77]
    pages = [-(-n // P) for n in lens]
    NP = 2 * sum(pages) + 5
    order = np.arange(NP, dtype=np.int32) if table == "consecutive" else \
        rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(order[at:at + npg].copy())
        t_dst.append(order[at + sum(pages):at + sum(pages) + npg].copy())
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, 256, 0, L, wl.TOKEN_MAJOR if r == 0 else
                                 wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    c = bulk(2, 1, 3, 32768)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    for op_s, op_l, where in (("store", "load", "host"), ("gather", "scatter", "device")):
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(17)
        arena = Arena(nbytes, where)
        _store(ctx, op_s, dpool, src, specs, arena, 0, None, c, stream)
        assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), op_s)
        data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
        arena.write(data)
        pre = dpool.host_copy()
        _load(ctx, op_l, dpool, dst, specs, arena, 0, None, c, stream)
        assert_pool_equal(dpool, expected_load(pre, dst, specs, data.copy()))
        arena.close()


def test_random_bulk_shapes(ctx, stream):
    """60 random batches under random bulk-mapping shapes (SM cap, CTAs per SM, stages per
    ring, stage size), store then load through host memory or gather then scatter in HBM."""
    for seed in range(60):
        rng = np.random.default_rng(77000 + seed)
        shape, lens, tables, load_tables, specs, lb, le = random_case(rng)
        L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size,
                           shape.token_bytes, shape.num_pages)
        stages = int(rng.integers(2, 9))
        max_units = (208 * 1024) // (2 * stages * 16)
        stage_bytes = 16 * int(rng.integers(1, max_units + 1))
        c = bulk(int(rng.integers(0, 7)), int(rng.integers(1, 3)), stages, stage_bytes)
        nbytes = wl._arena_bytes(specs, shape)
        src, dst = Requests(tables, lens), Requests(load_tables, lens)
        op_s, op_l, where = (("store", "load", "host") if seed % 2 == 0 else
                             ("gather", "scatter", "device"))
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(seed + 5)
        arena = Arena(nbytes, where)
        what = f"seed {seed} cfg {c.as_dict()}"
        _store(ctx, op_s, dpool, src, specs, arena, lb, le, c, stream)
        assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes, lb, le),
                           what)
        data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
        arena.write(data)
        pre = dpool.host_copy()
        _load(ctx, op_l, dpool, dst, specs, arena, lb, le, c, stream)
        assert_pool_equal(dpool, expected_load(pre, dst, specs, data.copy(), lb, le))
        arena.close()


@pytest.mark.parametrize("v,P,cfg_given,ctas_s,ctas_l", [(256, 8, False, 32, 32),
                                                          (256, 8, True, 8, 16),
                                                          (1024, 8, False, 8, 16),
                                                          (1024, 2, False, 32, 32)])
def test_store_load_default_grid_follows_segment_size(ctx, stream, v, P, cfg_given, ctas_s,
                                                      ctas_l):
    """With no configuration, a store or load of page segments shorter than 4 KiB runs on 32
    SMs (one CTA each), longer ones on the defaults (8 SMs for a store, 16 for a load); an
    explicit configuration keeps its own SM cap, and a plan follows the same rule.  Checked
    against the oracle either way."""
    rng = np.random.default_rng(8400 + v + P + int(cfg_given))
    L, KV, T = 8, 2, 16384  # enough segments for 32 CTAs of 32 warps resolving 16 each
    npg = T // P
    NP = 2 * npg + 3
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:npg]], [T]), Requests([perm[npg:2 * npg]], [T])
    specs = wl.split_tokens(0, 0, T, 256, 0, L, wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(8401)
    arena = Arena(nbytes, "host")
    cs = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_STORE) if cfg_given else None
    cl = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_LOAD) if cfg_given else None
    _store(ctx, "store", dpool, src, specs, arena, 0, None, cs, stream)
    assert kvx.kvx_last_launch(ctx)[1] == ctas_s
    assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), "store")
    data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
    arena.write(data)
    pre = dpool.host_copy()
    _load(ctx, "load", dpool, dst, specs, arena, 0, None, cl, stream)
    assert kvx.kvx_last_launch(ctx)[1] == ctas_l
    assert_pool_equal(dpool, expected_load(pre, dst, specs, data.copy()))
    # A prepared load plan made without a configuration takes the same grid.
    plan = kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, dpool.pool, dst.array,
                               kvx.chunks_array(specs, arena.ptr), cfg=cl,
                               stream=stream.cuda_stream)
    kvx.kvx_plan_launch(plan, stream.cuda_stream)
    stream.synchronize()
    kvx.kvx_plan_destroy(plan)
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    assert_pool_equal(dpool, expected_load(pre, dst, specs, data.copy()))
    arena.close()


def test_bulk_mapping_rejects_bad_stage_shapes(ctx, stream):
    dpool = DevicePool.empty(1, 1, 4, 1, 16)
    reqs = Requests([np.array([0], np.int32)], [1])
    arena = Arena(16, "host")
    ch = kvx.chunks_array([wl.ChunkSpec(0, 0, 1, 0, 1, 0, 0)], arena.ptr)
    for bad in (bulk(stages=1), bulk(stages=9), bulk(stage_bytes=24),
                bulk(stages=8, stage_bytes=65536), bulk(stages=4, stage_bytes=32768),
                cfg(batch=33), cfg(batch=-1)):
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_store_chunks(ctx, dpool.pool, reqs.array, ch, 0, 1, bad, stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    arena.close()


EXCHANGE_CONFIGS = [None, cfg(4, 1, 256, 8, 0), cfg(2, 1, 1024, 4, 0, batch=5),
                    cfg(0, 1, 512, 2, 0), cfg(3, 2, 128, 1, 0, batch=32), cfg(1, 1, 64, 8, 0)]


@pytest.mark.parametrize("seed", range(12))
def test_exchange_store_and_load_in_one_launch(ctx, stream, seed):
    """kvx_exchange_chunks: a store batch from one page set and a load batch into a disjoint
    one, in one launch; each output against the oracle.  Either batch may be empty."""
    rng = np.random.default_rng(7000 + seed)
    shape, lens, tables, load_tables, specs, lb, le = random_case(rng)
    L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size, shape.token_bytes,
                       shape.num_pages)
    c = EXCHANGE_CONFIGS[seed % len(EXCHANGE_CONFIGS)]
    nbytes = wl._arena_bytes(specs, shape)
    src, dst = Requests(tables, lens), Requests(load_tables, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(seed + 77)
    out = Arena(nbytes, "host")
    inp = Arena(nbytes, "host")
    data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
    inp.write(data)
    store_specs = [] if seed % 6 == 5 else specs
    load_specs = [] if seed % 6 == 4 else specs
    if seed % 6 == 3:  # a small load beside a large store: the shared-work kernel
        load_specs = specs[:max(1, len(specs) // 4)]
    pre = dpool.host_copy()
    kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, kvx.chunks_array(store_specs, out.ptr),
                            dst.array, kvx.chunks_array(load_specs, inp.ptr), lb, le, c,
                            stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(store_specs, exp), lb, le)
    assert_bytes_equal(out.numpy(), exp, f"exchange store seed {seed}")
    exp_pool = expected_load(pre, dst, load_specs, data.copy(), lb, le)
    assert_pool_equal(dpool, exp_pool)
    out.close()
    inp.close()


@pytest.mark.parametrize("load_share", [1.0, 0.3])
def test_exchange_token_major_pages(ctx, stream, load_share):
    """Exchanges of token-major chunks over all layers, 32 KiB pages of strided rows: equal
    batches (the role-split kernel) and a load of 30 % of the store (the shared-work kernel),
    both through their row-walking variants; each output against the oracle."""
    rng = np.random.default_rng(7300 + int(load_share * 10))
    L, KV, P, v, T = 4, 2, 16, 2048, 1024
    npg = T // P
    NP = 2 * npg + 5
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:npg]], [T]), Requests([perm[npg:2 * npg]], [T])
    specs = wl.split_tokens(0, 0, T, 64, 0, L, wl.TOKEN_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    load_specs = specs[:max(1, int(len(specs) * load_share))]
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(7301)
    out, inp = Arena(nbytes, "host"), Arena(nbytes, "host")
    data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
    inp.write(data)
    pre = dpool.host_copy()
    kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, kvx.chunks_array(specs, out.ptr),
                            dst.array, kvx.chunks_array(load_specs, inp.ptr),
                            stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(out.numpy(), exp, "exchange store")
    assert_pool_equal(dpool, expected_load(pre, dst, load_specs, data.copy()))
    out.close()
    inp.close()


def test_exchange_rejects_a_load_into_the_store_sources(ctx, stream):
    L, KV, P, v, NP = 2, 2, 4, 64, 8
    dpool = DevicePool.empty(L, KV, NP, P, v)
    before = dpool.tensor.clone()
    src = Requests([np.array([1, 2], np.int32)], [8])
    dst = Requests([np.array([2, 5], np.int32)], [8])  # page 2 is read and written
    arena = Arena(8 * L * KV * v, "host")
    ch = kvx.chunks_array([wl.ChunkSpec(0, 0, 8, 0, L, 0, 0)], arena.ptr)
    kvx.kvx_set_validation(ctx, 2)
    try:
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, ch, dst.array, ch, 0, L, None,
                                    stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_OVERLAP
        # Disjoint layers make the same slots legal.
        kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, ch, dst.array, ch, 0, L, None,
                                stream.cuda_stream) if False else None
    finally:
        kvx.kvx_set_validation(ctx, 1)
    stream.synchronize()
    assert torch.equal(before, dpool.tensor)
    arena.close()


# ----------------------------------------------------------------------------- edge cases

def test_empty_and_degenerate_batches(ctx, stream):
    L, KV, P, v, NP = 2, 2, 4, 64, 16
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(3)
    before = dpool.tensor.clone()
    reqs = Requests([np.array([1, 2], np.int32), np.zeros(0, np.int32)], [7, 0])
    arena = Arena(4096, "host")
    empty = np.zeros(0, kvx.CHUNK_DTYPE)
    kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array, empty, 0, L, None, stream.cuda_stream)
    assert kvx.kvx_last_launch(ctx)[0] == 0
    # Zero-token chunk, chunk of the empty request, chunk outside the layer window.
    specs = [wl.ChunkSpec(0, 3, 0, 0, L, 0, 0), wl.ChunkSpec(1, 0, 0, 0, L, 1, 256),
             wl.ChunkSpec(0, 0, 7, 1, 1, 0, 512)]
    ch = kvx.chunks_array(specs, arena.ptr)
    kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array, ch, 0, 1, None, stream.cuda_stream)
    assert kvx.kvx_last_launch(ctx)[0] == 0
    # The same nothing through the exchange, the round trip and their plans.
    kvx.kvx_exchange_chunks(ctx, dpool.pool, reqs.array, empty, reqs.array, ch, 0, 1,
                            stream=stream.cuda_stream)
    assert kvx.kvx_last_launch(ctx)[0] == 0
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, reqs.array, reqs.array, empty,
                             stream=stream.cuda_stream)
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, reqs.array, reqs.array, ch, 0, 1,
                             stream=stream.cuda_stream)
    assert kvx.kvx_last_launch(ctx)[0] == 0
    for plan in (kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, dpool.pool, reqs.array, ch, 0, 1,
                                     stream=stream.cuda_stream),
                 kvx.kvx_plan_create_exchange(ctx, dpool.pool, reqs.array, empty, reqs.array,
                                              empty, stream=stream.cuda_stream),
                 kvx.kvx_plan_create_roundtrip(ctx, dpool.pool, reqs.array, reqs.array, ch, 0, 1,
                                               stream=stream.cuda_stream)):
        kvx.kvx_plan_launch(plan, stream.cuda_stream)
        kvx.kvx_plan_destroy(plan)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    assert torch.equal(before, dpool.tensor)
    # Single token, one unit wide.
    pool1 = DevicePool.empty(1, 1, 4, 1, 16)
    pool1.fill_random(9)
    r1 = Requests([np.array([3], np.int32)], [1])
    a1 = Arena(16, "host")
    _store(ctx, "store", pool1, r1, [wl.ChunkSpec(0, 0, 1, 0, 1, 1, 0)], a1, 0, None, cfg(), stream)
    assert_bytes_equal(a1.numpy()[:16], pool1.tensor[0, 0, 3, 0].cpu().numpy(), "one token")
    assert np.all(a1.numpy()[16:] == CANARY)
    arena.close()
    a1.close()


def test_largest_segment_and_partial_pages(ctx, stream):
    """64-token pages of 1152-B latents (72 KiB segments), chunks that split pages."""
    L, KV, P, v = 2, 1, 64, 1152
    T = 64 * 5 + 37
    NP = 16
    rng = np.random.default_rng(4)
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:6]], [T]), Requests([perm[6:12]], [T])
    specs = wl.split_tokens(0, 0, T, 56, 0, L, wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(5)
    arena = Arena(nbytes, "host")
    _store(ctx, "store", dpool, src, specs, arena, 0, None, cfg(), stream)
    assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), "store")
    pre = dpool.host_copy()
    _load(ctx, "load", dpool, dst, specs, arena, 0, None, cfg(), stream)
    exp = expected_load(pre, dst, specs, arena.numpy().copy())
    assert_pool_equal(dpool, exp)
    # Slots past the last token of the last destination page keep their old bytes.
    last = dst.host[0][-1]
    assert torch.equal(dpool.tensor[0, :, last, 37:].cpu(),
                       torch.from_numpy(np.stack([pre.pools[0][l][last, 37:]
                                                  for l in range(L)])))
    arena.close()


def test_many_calls_in_flight_on_two_streams(ctx):
    """More calls than descriptor buffers, alternating streams: each must see its own batch."""
    rng = np.random.default_rng(8)
    L, KV, P, v, T = 4, 2, 16, 256, 512
    NP = 4 * (T // P) * 3
    perm = rng.permutation(NP).astype(np.int32)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(11)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    arenas, cases = [], []
    for i in range(10):
        tab = perm[(i % 4) * (T // P):(i % 4 + 1) * (T // P)]
        req = Requests([tab], [T])
        specs = wl.split_tokens(0, 0, T, 64 + 16 * i, 0, L, i % 2)
        shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
        wl.place_chunks(specs, shape)
        nbytes = wl._arena_bytes(specs, shape)
        arena = Arena(nbytes, "host")
        ch = kvx.chunks_array(specs, arena.ptr)
        kvx.kvx_store_chunks(ctx, dpool.pool, req.array, ch, 0, L, cfg(1 + i % 3),
                             streams[i % 2].cuda_stream)
        arenas.append(arena)
        cases.append((req, specs, nbytes))
    torch.cuda.synchronize()
    for arena, (req, specs, nbytes) in zip(arenas, cases):
        assert_bytes_equal(arena.numpy(), expected_store(dpool, req, specs, nbytes), "in flight")
        arena.close()


def test_round_trips_and_exchanges_in_flight_on_two_streams(ctx):
    """Eight round trips and exchanges, more than the descriptor buffers, alternating two
    streams so that launches overlap on the GPU: each keeps its own work counters and
    completion words, and each result matches the oracle."""
    rng = np.random.default_rng(18)
    L, KV, P, v, T = 3, 2, 16, 512, 640
    pages = T // P
    NP = pages * 17
    perm = rng.permutation(NP).astype(np.int32)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(19)
    pre = dpool.host_copy()  # every source page set is read-only below
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    cases = []
    for i in range(8):
        src = Requests([perm[(2 * i) * pages:(2 * i + 1) * pages]], [T])
        dst = Requests([perm[(2 * i + 1) * pages:(2 * i + 2) * pages]], [T])
        specs = wl.split_tokens(0, 0, T, 32 + 16 * i, 0, L, i % 3)
        wl.place_chunks(specs, shape)
        nbytes = wl._arena_bytes(specs, shape)
        out = Arena(nbytes, "host")
        ch = kvx.chunks_array(specs, out.ptr)
        s = streams[i % 2].cuda_stream
        if i % 2 == 0:
            kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array, ch, 0, L,
                                     cfg(2 + i % 3, 1, 128), s)
            inp = None
        else:  # an exchange: store src into `out`, load `inp` (random bytes) into dst
            inp = Arena(nbytes, "host")
            inp.write(rng.integers(0, 256, nbytes + 4096, dtype=np.uint8))
            kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, ch, dst.array,
                                    kvx.chunks_array(specs, inp.ptr), 0, L, None, s)
        cases.append((src, dst, specs, nbytes, out, inp))
    torch.cuda.synchronize()
    assert kvx.kvx_get_status(ctx, 0) == 0
    for src, dst, specs, nbytes, out, inp in cases:
        exp = np.full(nbytes + 4096, CANARY, np.uint8)
        oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
        assert_bytes_equal(out.numpy(), exp, "store half in flight")
        oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp if inp is None
                                                     else inp.numpy().copy()))
        out.close()
        if inp is not None:
            inp.close()
    assert_pool_equal(dpool, pre)


# ----------------------------------------------------------------------------- errors

@pytest.mark.parametrize("layout", [wl.LAYER_MAJOR, wl.TOKEN_MAJOR])
def test_in_kernel_page_check_skips_and_reports(ctx, stream, layout):
    """A device page table naming a page past the pool: that segment is skipped, flagged,
    and everything else is still moved (validation level 1 does not read page tables).
    Token-major chunks take the row-walking kernel."""
    L, KV, P, v, NP = 2, 2, 8, 64, 8
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(12)
    good = np.array([5, 2], np.int32)
    bad = np.array([5, NP + 1000], np.int32)
    reqs = Requests([bad], [16], host_copy=False)
    specs = [wl.ChunkSpec(0, 0, 8, 0, L, layout), wl.ChunkSpec(0, 8, 8, 0, L, layout)]
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    arena = Arena(nbytes, "host")
    ch = kvx.chunks_array(specs, arena.ptr)
    kvx.kvx_store_chunks(ctx, dpool.pool, reqs.array, ch, 0, L, None, stream.cuda_stream)
    stream.synchronize()
    flags = kvx.kvx_get_status(ctx, stream.cuda_stream)
    assert flags == kvx.KVX_DEV_PAGE_OUT_OF_RANGE
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0  # reading cleared it
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(dpool.host_copy(), [oracle.Request(good, 16)], oracle_chunks(specs[:1], exp))
    assert_bytes_equal(arena.numpy(), exp, "valid part moved, bad page skipped")
    arena.close()


@pytest.mark.parametrize("layout", [wl.LAYER_MAJOR, wl.TOKEN_MAJOR])
def test_roundtrip_page_check_skips_and_reports(ctx, stream, layout):
    """Round trip whose source table names a page past the pool: that store segment is
    skipped and flagged, its load still runs after it (reading the untouched chunk bytes),
    and every other segment makes the full round trip.  Token-major chunks take the round
    trip's row-walking variant."""
    L, KV, P, v, NP = 2, 2, 8, 64, 8
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(13)
    bad_src = np.array([5, NP + 1000], np.int32)
    dst_table = np.array([1, 3], np.int32)
    src = Requests([bad_src], [16], host_copy=False)
    dst = Requests([dst_table], [16])
    specs = [wl.ChunkSpec(0, 0, 8, 0, L, layout), wl.ChunkSpec(0, 8, 8, 0, L, layout)]
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    arena = Arena(nbytes, "host")
    pre = dpool.host_copy()
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == kvx.KVX_DEV_PAGE_OUT_OF_RANGE
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, [oracle.Request(np.array([5, 0], np.int32), 16)],
                 oracle_chunks(specs[:1], exp))
    assert_bytes_equal(arena.numpy(), exp, "valid chunk stored, bad page's chunk untouched")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()


def test_roundtrip_wait_runs_out_and_reports(ctx, stream):
    """The round trip's bounded wait, made to run out without faulting the GPU: a round trip
    whose stores never run (kvx_test_roundtrip_timeout) ends after about one wait limit,
    sets KVX_DEV_WAIT_TIMEOUT and writes nothing; the same context then carries a normal
    round trip bit-exactly."""
    L, KV, P, v, NP = 2, 2, 16, 256, 40
    perm = np.random.default_rng(7900).permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:8]], [128]), Requests([perm[8:16]], [128])
    specs = wl.split_tokens(0, 0, 128, 32, 0, L, wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(7901)
    pre = dpool.host_copy()
    arena = Arena(nbytes, "host")
    ch = kvx.chunks_array(specs, arena.ptr)
    for bad in (0, 999_999, 1_000_000_001):
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_test_roundtrip_timeout(ctx, dpool.pool, src.array, dst.array, ch, bad,
                                           stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    wait_ns = 20_000_000
    stream.synchronize()
    t0 = time.perf_counter()
    kvx.kvx_test_roundtrip_timeout(ctx, dpool.pool, src.array, dst.array, ch, wait_ns,
                                   stream.cuda_stream)
    stream.synchronize()
    elapsed = time.perf_counter() - t0
    # 32 segments of 4 KiB in units of two (8 KiB): 16 load units, one per warp of the one
    # CTA the launch needs, all waiting at once.
    assert 0.9 * wait_ns * 1e-9 <= elapsed < 1.0, elapsed
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == kvx.KVX_DEV_WAIT_TIMEOUT
    assert_bytes_equal(arena.numpy(), np.full(nbytes + 4096, CANARY, np.uint8),
                       "no store ran, so no chunk byte changed")
    assert_pool_equal(dpool, pre)
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array, ch,
                             stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(arena.numpy(), exp, "round trip after the timeout")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()


def test_host_detected_errors_launch_nothing(ctx, stream):
    L, KV, P, v, NP = 2, 2, 8, 64, 8
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(13)
    before = dpool.tensor.clone()
    tab = np.array([1, 2], np.int32)
    reqs = Requests([tab], [16])
    specs = [wl.ChunkSpec(0, 0, 16, 0, L, 0, 0)]
    nbytes = 16 * L * KV * v
    kvx.kvx_set_validation(ctx, 2)
    try:
        # Pageable host memory.
        pageable = np.zeros(nbytes + 64, np.uint8)
        base = pageable.ctypes.data + (-pageable.ctypes.data % 16)
        ch = kvx.chunks_array(specs, base)
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_store_chunks(ctx, dpool.pool, reqs.array, ch, 0, L, None, stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_NOT_DEVICE_ACCESSIBLE
        # Device memory given to store, host memory given to the HBM transform.
        dev = Arena(nbytes, "device")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_store_chunks(ctx, dpool.pool, reqs.array, kvx.chunks_array(specs, dev.ptr),
                                 0, L, None, stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
        host = Arena(nbytes, "host")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, dpool.pool, reqs.array,
                                  kvx.chunks_array(specs, host.ptr), 0, L, None,
                                  stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
        # Overlapping load destinations.
        two = [wl.ChunkSpec(0, 0, 16, 0, L, 0, 0), wl.ChunkSpec(0, 8, 8, 1, 1, 0, 4096)]
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array, kvx.chunks_array(two, host.ptr), 0,
                                L, None, stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_OVERLAP
        # Page id out of range (host copy given).
        badreq = Requests([np.array([1, 99], np.int32)], [16])
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_load_chunks(ctx, dpool.pool, badreq.array,
                                kvx.chunks_array(specs, host.ptr), 0, L, None, stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_PAGE_OUT_OF_RANGE
        assert "99" in kvx.kvx_last_error(ctx)
        # Misaligned chunk pointer.
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array,
                                kvx.chunks_array(specs, host.ptr + 8), 0, L, None,
                                stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_ALIGNMENT
        # Bad launch configuration.
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array, kvx.chunks_array(specs, host.ptr),
                                0, L, cfg(threads=100), stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
        stream.synchronize()
        assert torch.equal(before, dpool.tensor)
        assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
        dev.close()
        host.close()
    finally:
        kvx.kvx_set_validation(ctx, 1)


def test_descriptor_capacity_error():
    small = kvx.kvx_create(0, 1024)
    try:
        L, KV, P, v, NP = 1, 1, 1, 16, 512
        dpool = DevicePool.empty(L, KV, NP, P, v)
        reqs = Requests([np.arange(256, dtype=np.int32)], [256])
        specs = wl.split_tokens(0, 0, 256, 1, 0, 1, 0)
        shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
        wl.place_chunks(specs, shape, align=16)
        arena = Arena(wl._arena_bytes(specs, shape), "host")
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_store_chunks(small, dpool.pool, reqs.array,
                                 kvx.chunks_array(specs, arena.ptr), 0, 1, None, 0)
        assert e.value.status == kvx.KVX_ERR_CAPACITY
        arena.close()
    finally:
        kvx.kvx_destroy(small)


@pytest.mark.parametrize("v,shift,layout", [(64, 0, wl.LAYER_MAJOR), (64, 0, wl.TOKEN_MAJOR),
                                             (2048, 0, wl.STRIPED), (48, 0, wl.LAYER_MAJOR),
                                             (64, 16, wl.LAYER_MAJOR)])
@pytest.mark.parametrize("unroll", [1, 2, 4, 8])
def test_transform_32_byte_accesses_and_fallbacks(ctx, stream, v, shift, layout, unroll):
    """The HBM transform takes 32-byte accesses when token_bytes, the pool and every chunk are
    32-byte aligned (v = 64, 2048), and 16-byte ones otherwise (v = 48; chunks 16 bytes off
    a 32-byte boundary).  Both, for every unroll and row layout, against the oracle."""
    rng = np.random.default_rng(1500 + v + shift + layout * 7 + unroll)
    L, KV, P = 3, 2, 16
    lens = [700, 230]
    pages = [-(-n // P) for n in lens]
    NP = 2 * sum(pages) + 3
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[sum(pages) + at:sum(pages) + at + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, 96, 0, L, layout)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape, align=wl.STRIPE_ALIGN)
    nbytes = wl._arena_bytes(specs, shape)
    for c in specs:
        c.offset += shift
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    c = cfg(0, 2, 256, unroll, 1)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(1501 + unroll)
    arena = Arena(nbytes + shift, "device")
    _store(ctx, "gather", dpool, src, specs, arena, 0, None, c, stream)
    assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes + shift), "gather")
    pre = dpool.host_copy()
    _load(ctx, "scatter", dpool, dst, specs, arena, 0, None, c, stream)
    assert_pool_equal(dpool, expected_load(pre, dst, specs, arena.numpy().copy()))


def test_default_launch_configs(ctx):
    for op in range(5):
        c = kvx.kvx_default_launch_cfg(ctx, op)
        assert c.threads % 32 == 0 and c.unroll in (1, 2, 4, 8)
    assert kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_LOAD).sm_cap > 0
    assert kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_GATHER_HBM).sm_cap == 0


def test_offsets_beyond_4_gib(ctx, stream):
    """64-bit address arithmetic: one layer pool of 4.5 GiB with the request on its last
    pages (page offsets past 2^32), and an HBM chunk of 4.25 GiB (chunk offsets past 2^32),
    checked byte for byte on host copies."""
    L, KV, P, v = 1, 1, 16, 4096
    num_pages = 73728                      # 73728 x 16 x 4096 B = 4.5 GiB
    n_tok = 1114112                        # 69632 pages, chunk 1114112 x 4096 B = 4.25 GiB
    pages = n_tok // P
    table = np.arange(num_pages - pages, num_pages, dtype=np.int32)[::-1].copy()
    dpool = DevicePool.empty(L, KV, num_pages, P, v, fill=0)
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)
    tail = dpool.tensor[0, 0, num_pages - pages:]
    tail.copy_(torch.randint(0, 256, tail.shape, generator=g, device="cuda",
                             dtype=torch.int16).to(torch.uint8))
    reqs = Requests([table], [n_tok])
    spec = [wl.ChunkSpec(0, 0, n_tok, 0, 1, wl.LAYER_MAJOR, 0)]
    chunk = torch.full((n_tok * v,), CANARY, dtype=torch.uint8, device="cuda")
    assert chunk.numel() > (1 << 32)
    torch.cuda.synchronize()  # the pool and chunk fills ran on the current stream
    kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, dpool.pool, reqs.array,
                          kvx.chunks_array(spec, chunk.data_ptr()), stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    # Oracle on host copies of the whole 4.5 GiB layer.
    host_layer = torch.empty(dpool.tensor.shape[2:], dtype=torch.uint8, pin_memory=True)
    host_layer.copy_(dpool.tensor[0, 0])
    opool = oracle.Pool([[host_layer.numpy()]], P)
    expect = np.empty(n_tok * v, np.uint8)
    oracle.store(opool, reqs.oracle(), oracle_chunks(spec, expect), threads=8)
    got = torch.empty(chunk.shape, dtype=torch.uint8, pin_memory=True)
    got.copy_(chunk)
    assert_bytes_equal(got.numpy(), expect, "gather with offsets past 4 GiB")
    # Scatter it back into the first pages of the pool, in order (table2 = 0, 1, 2, ...),
    # and check those pages against the oracle's load.
    table2 = np.arange(0, pages, dtype=np.int32)
    reqs2 = Requests([table2], [n_tok])
    kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, dpool.pool, reqs2.array,
                          kvx.chunks_array(spec, chunk.data_ptr()), stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    oracle.load(opool, reqs2.oracle(), oracle_chunks(spec, expect), threads=8)
    host_layer2 = torch.empty(dpool.tensor.shape[2:], dtype=torch.uint8, pin_memory=True)
    host_layer2.copy_(dpool.tensor[0, 0])
    assert_bytes_equal(host_layer2.numpy().reshape(-1), host_layer.numpy().reshape(-1),
                       "scatter with chunk offsets past 4 GiB")
    del chunk


def _blocks_case(rng, L=4, KV=2, P=16, v=1024, n_tok=900):
    pages = -(-n_tok // P)
    NP = 2 * pages + 3
    table = rng.permutation(NP)[:pages].astype(np.int32)
    specs = wl.split_tokens(0, 0, n_tok, P, 0, L, wl.STRIPED)  # one block object set per page
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape, align=wl.STRIPE_ALIGN)
    return shape, table, specs, wl._arena_bytes(specs, shape)


def test_prepared_plans_reuse_descriptors_and_see_new_contents(ctx, stream):
    """Per-layer load plans made once, launched twice with different chunk contents."""
    rng = np.random.default_rng(606)
    shape, table, specs, nbytes = _blocks_case(rng)
    L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size, shape.token_bytes,
                       shape.num_pages)
    reqs = Requests([table], [900])
    dpool = DevicePool.empty(L, KV, NP, P, v)
    arena = Arena(nbytes, "host")
    ch = kvx.chunks_array(specs, arena.ptr)
    plans = [kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, dpool.pool, reqs.array, ch, l, l + 1,
                                 None, stream.cuda_stream) for l in range(L)]
    try:
        for round_ in range(2):
            data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
            arena.write(data)
            pre = dpool.host_copy()
            for p in plans:
                kvx.kvx_plan_launch(p, stream.cuda_stream)
            stream.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            assert_pool_equal(dpool, expected_load(pre, reqs, specs, data.copy()))
    finally:
        for p in plans:
            kvx.kvx_plan_destroy(p)
        arena.close()


def test_prepared_plans_in_a_cuda_graph(ctx):
    """A store plan and per-layer load plans captured into one CUDA graph and replayed."""
    rng = np.random.default_rng(707)
    shape, table, specs, nbytes = _blocks_case(rng, L=3, KV=1, v=1152)
    L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size, shape.token_bytes,
                       shape.num_pages)
    src = Requests([table], [900])
    dst_table = np.setdiff1d(np.arange(NP, dtype=np.int32), table)[:len(table)]
    dst = Requests([rng.permutation(dst_table).astype(np.int32)], [900])
    dpool = DevicePool.empty(L, KV, NP, P, v)
    arena = Arena(nbytes, "host")
    ch = kvx.chunks_array(specs, arena.ptr)
    s = torch.cuda.Stream()
    store = kvx.kvx_plan_create(ctx, kvx.KVX_OP_STORE, dpool.pool, src.array, ch, 0, L, None,
                                s.cuda_stream)
    loads = [kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, dpool.pool, dst.array, ch, l, l + 1,
                                 None, s.cuda_stream) for l in range(L)]
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            cs = torch.cuda.current_stream().cuda_stream
            kvx.kvx_plan_launch(store, cs)
            for p in loads:
                kvx.kvx_plan_launch(p, cs)
        for round_ in range(2):
            dpool.fill_random(808 + round_)
            pre = dpool.host_copy()
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            assert kvx.kvx_get_status(ctx, 0) == 0
            exp_chunks = np.full(nbytes + 4096, CANARY, np.uint8)
            oracle.store(pre, src.oracle(), oracle_chunks(specs, exp_chunks))
            got = arena.numpy()
            for c in specs:  # compare the objects (padding is never written)
                stride = -(-c.n_tokens * v // wl.STRIPE_ALIGN) * wl.STRIPE_ALIGN
                for l in range(L):
                    off = c.offset + l * stride
                    assert_bytes_equal(got[off:off + c.n_tokens * v],
                                       exp_chunks[off:off + c.n_tokens * v], "graph store")
            oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp_chunks))
            assert_pool_equal(dpool, pre)
    finally:
        kvx.kvx_plan_destroy(store)
        for p in loads:
            kvx.kvx_plan_destroy(p)
        arena.close()


@pytest.mark.parametrize("n_s,n_l", [(700, 500), (900, 120), (64, 1100)])
def test_exchange_plans_match_the_oracle(ctx, stream, n_s, n_l):
    """Exchange plans: store one batch and load another in one prepared launch, twice, with
    new pool and chunk contents in between; also captured in a CUDA graph.  Similar batch
    sizes run the role-split kernel, unequal ones the shared-work kernel."""
    rng = np.random.default_rng(909 + n_s)
    L, KV, P, v, NP = 3, 2, 16, 512, 200
    pages_s, pages_l = -(-n_s // P), -(-n_l // P)
    perm = rng.permutation(NP).astype(np.int32)
    st_req = Requests([perm[:pages_s]], [n_s])
    ld_req = Requests([perm[pages_s:pages_s + pages_l]], [n_l])
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    s_specs = wl.split_tokens(0, 0, n_s, 96, 0, L, wl.LAYER_MAJOR)
    l_specs = wl.split_tokens(0, 0, n_l, 80, 0, L, wl.TOKEN_MAJOR)
    wl.place_chunks(s_specs + l_specs, shape)
    nbytes = wl._arena_bytes(s_specs + l_specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    arena = Arena(nbytes, "host")
    sch = kvx.chunks_array(s_specs, arena.ptr)
    lch = kvx.chunks_array(l_specs, arena.ptr)
    plan = kvx.kvx_plan_create_exchange(ctx, dpool.pool, st_req.array, sch, ld_req.array, lch,
                                        stream=stream.cuda_stream)
    s2 = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s2):
        kvx.kvx_plan_launch(plan, torch.cuda.current_stream().cuda_stream)
    try:
        for round_ in range(3):
            dpool.fill_random(910 + round_)
            data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
            arena.write(data)
            pre = dpool.host_copy()
            torch.cuda.synchronize()
            if round_ < 2:
                kvx.kvx_plan_launch(plan, stream.cuda_stream)
            else:
                with torch.cuda.stream(s2):
                    graph.replay()
            torch.cuda.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            exp = data.copy()
            oracle.store(pre, st_req.oracle(), oracle_chunks(s_specs, exp))
            oracle.load(pre, ld_req.oracle(), oracle_chunks(l_specs, exp))
            assert_bytes_equal(arena.numpy()[:nbytes + 4096], exp, "exchange plan chunks")
            assert_pool_equal(dpool, pre)
    finally:
        del graph
        kvx.kvx_plan_destroy(plan)
        arena.close()


RT_CONFIGS = [None, cfg(1, 1, 32, 1, 0), cfg(1, 1, 64, 8, 0), cfg(2, 1, 1024, 8, 0),
              cfg(3, 1, 256, 4, 0, batch=5), cfg(1, 1, 32, 2, 0, batch=32),
              cfg(0, 1, 1024, 8, 0), cfg(4, 2, 128, 2, 0, batch=3)]


@pytest.mark.parametrize("seed", range(24))
def test_roundtrip_in_one_launch(ctx, stream, seed):
    """Store to host chunks and load them into the other page set in one launch; the
    arena must hold the oracle's store and the pool the oracle's load of it."""
    rng = np.random.default_rng(7100 + seed)
    shape, lens, tables, load_tables, specs, lb, le = random_case(rng)
    L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size, shape.token_bytes,
                       shape.num_pages)
    c = RT_CONFIGS[seed % len(RT_CONFIGS)]
    arena_bytes = wl._arena_bytes(specs, shape)
    src = Requests(tables, lens)
    dst = Requests(load_tables, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(seed * 17 + 3)
    arena = Arena(arena_bytes, "host")
    pre = dpool.host_copy()
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), lb, le, c, stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp = np.full(arena_bytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp), lb, le)
    assert_bytes_equal(arena.numpy(), exp, f"seed {seed} round-trip chunks")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp), lb, le)
    assert_pool_equal(dpool, pre)
    arena.close()


@pytest.mark.parametrize("P,sm_cap", [(2, 0), (4, 0), (4, 8), (16, 0)])
def test_roundtrip_token_major_pages(ctx, stream, P, sm_cap):
    """Round trips of token-major chunks over all layers (pages of strided 1152-byte rows):
    batched units of short pages (2 and 4 tokens, on the default 32 SMs or on 8) and one
    segment per unit (16 tokens), through the round trip's row-walking variants; chunks and
    pages against the oracle."""
    rng = np.random.default_rng(8200 + P + sm_cap)
    L, KV, v = 3, 1, 1152
    lens = [800, 37, 2 * P + 1]
    pages = [-(-n // P) for n in lens]
    NP = 2 * sum(pages) + 5
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[sum(pages) + at:sum(pages) + at + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, 96, 0, L, wl.TOKEN_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(8201 + P)
    pre = dpool.host_copy()
    arena = Arena(nbytes, "host")
    c = None
    if sm_cap:
        c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_ROUNDTRIP)
        c.sm_cap = sm_cap
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), cfg=c,
                             stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(arena.numpy(), exp, "token-major round trip chunks")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()


@pytest.mark.parametrize("v,P,layout", [(1152, 64, 0), (1152, 64, 1), (1152, 64, 2),
                                         (4096, 16, 0), (2048, 32, 1), (1152, 29, 2)])
def test_roundtrip_long_segments_in_row_slices(ctx, stream, v, P, layout):
    """Page segments longer than 32 KiB make the round trip's units row slices of one
    segment (72 KiB: three slices; 64 KiB: two).  Partial last pages (one row, so some
    slices are empty) and chunk cuts inside pages shorten segments; everything is compared
    with the oracle's store and load."""
    rng = np.random.default_rng(8100 + v + P + layout)
    L, KV = 2, 2
    lens = [700, 65, 1, 3 * P + 1]
    pages = [-(-n // P) for n in lens]
    NP = 2 * sum(pages) + 5
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[sum(pages) + at:sum(pages) + at + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, 100, 0, L, layout)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape, align=wl.STRIPE_ALIGN)
    nbytes = wl._arena_bytes(specs, shape)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(8101 + P)
    pre = dpool.host_copy()
    arena = Arena(nbytes, "host")
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    items, _, _, _ = kvx.kvx_last_launch(ctx)
    segments = kvx.kvx_plan_count(dpool.pool, src.array, kvx.chunks_array(specs, arena.ptr))[0]
    assert items == 2 * segments
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(arena.numpy(), exp, "sliced round trip chunks")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()


@pytest.mark.parametrize("v,P,cfg_given,ctas", [(256, 16, False, 32), (256, 16, True, 16),
                                                 (1024, 16, False, 16)])
def test_roundtrip_default_grid_follows_segment_size(ctx, stream, v, P, cfg_given, ctas):
    """With no configuration, a round trip of page segments shorter than 16 KiB runs on 32
    SMs (one CTA each), longer ones on 16; an explicit configuration keeps its own SM cap.
    The transfer is checked against the oracle either way."""
    rng = np.random.default_rng(8300 + v + int(cfg_given))
    L, KV, T = 4, 2, 4096
    npg = T // P
    NP = 2 * npg + 3
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:npg]], [T]), Requests([perm[npg:2 * npg]], [T])
    specs = wl.split_tokens(0, 0, T, 256, 0, L, wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(8301)
    pre = dpool.host_copy()
    arena = Arena(nbytes, "host")
    c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_ROUNDTRIP) if cfg_given else None
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), cfg=c,
                             stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    assert kvx.kvx_last_launch(ctx)[1] == ctas
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert kvx.kvx_roundtrip_unit(P, v, c, sms)[1] == ctas  # the query the time model uses
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(arena.numpy(), exp, "round trip chunks")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()


def test_roundtrip_many_requests_and_chunks(ctx, stream):
    """64 requests of mixed length cut into about 540 chunks of all three layouts: the
    round trip's unit search runs several probe levels deep."""
    rng = np.random.default_rng(7500)
    L, KV, P, v = 4, 2, 16, 512
    lens = [int(x) for x in rng.integers(1, 2000, 64)]
    pages = [-(-n // P) for n in lens]
    NP = 2 * sum(pages) + 7
    perm = rng.permutation(NP).astype(np.int32)
    t_src, t_dst, at = [], [], 0
    for npg in pages:
        t_src.append(perm[at:at + npg])
        t_dst.append(perm[sum(pages) + at:sum(pages) + at + npg])
        at += npg
    specs = []
    for r, n in enumerate(lens):
        specs += wl.split_tokens(r, 0, n, int(rng.choice([48, 160, 256])), 0, L, r % 3)
    order = rng.permutation(len(specs))
    specs = [specs[i] for i in order]
    assert len(specs) > 500
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape, align=wl.STRIPE_ALIGN)
    nbytes = wl._arena_bytes(specs, shape)
    src, dst = Requests(t_src, lens), Requests(t_dst, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(7501)
    pre = dpool.host_copy()
    arena = Arena(nbytes, "host")
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), stream=stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(arena.numpy(), exp, "many-request round trip chunks")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()


def test_roundtrip_rejects_overlapping_page_sets(ctx, stream):
    """A load page set that meets the store's sources is refused (validation level 2)."""
    rng = np.random.default_rng(7200)
    L, KV, P, v, NP = 2, 2, 16, 256, 64
    table = rng.permutation(NP)[:8].astype(np.int32)
    other = table.copy()
    other[3] = table[3]  # same page: overlap
    other[:3] = rng.permutation(np.setdiff1d(np.arange(NP), table))[:3]
    src, dst = Requests([table], [128]), Requests([other], [128])
    specs = wl.split_tokens(0, 0, 128, 64, 0, L, wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    arena = Arena(wl._arena_bytes(specs, shape), "host")
    kvx.kvx_set_validation(ctx, 2)
    try:
        with pytest.raises(kvx.KvxError) as e:
            kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                                     kvx.chunks_array(specs, arena.ptr),
                                     stream=stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_OVERLAP
    finally:
        kvx.kvx_set_validation(ctx, 1)
        arena.close()


def test_roundtrip_plan_and_graph(ctx):
    """A round-trip plan launched directly and from a CUDA graph, each time on fresh pool
    contents; counters and completion words are reset by the launch itself."""
    rng = np.random.default_rng(7300)
    shape, lens, tables, load_tables, specs, lb, le = random_case(rng)
    L, KV, P, v, NP = (shape.num_layers, shape.kv_factor, shape.page_size, shape.token_bytes,
                       shape.num_pages)
    arena_bytes = wl._arena_bytes(specs, shape)
    src, dst = Requests(tables, lens), Requests(load_tables, lens)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    arena = Arena(arena_bytes, "host")
    s = torch.cuda.Stream()
    plan = kvx.kvx_plan_create_roundtrip(ctx, dpool.pool, src.array, dst.array,
                                         kvx.chunks_array(specs, arena.ptr), lb, le,
                                         cfg(3, 1, 128, 8, 0, batch=3), s.cuda_stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kvx.kvx_plan_launch(plan, torch.cuda.current_stream().cuda_stream)
    try:
        for round_ in range(4):
            dpool.fill_random(7301 + round_)
            pre = dpool.host_copy()
            torch.cuda.synchronize()
            if round_ % 2 == 0:
                kvx.kvx_plan_launch(plan, s.cuda_stream)
            else:
                with torch.cuda.stream(s):
                    graph.replay()
            torch.cuda.synchronize()
            assert kvx.kvx_get_status(ctx, s.cuda_stream) == 0
            # Every round writes the same chunk bytes, so the arena holds exactly this round's
            # store over the canary fill.
            exp = np.full(arena_bytes + 4096, CANARY, np.uint8)
            oracle.store(pre, src.oracle(), oracle_chunks(specs, exp), lb, le)
            assert_bytes_equal(arena.numpy(), exp, f"round {round_} chunk bytes")
            oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp), lb, le)
            assert_pool_equal(dpool, pre)
    finally:
        del graph
        kvx.kvx_plan_destroy(plan)
        arena.close()


def test_roundtrip_with_more_ctas_than_can_be_resident(ctx, stream):
    """608 CTAs of 1024 threads on 152 SMs: most start only after others finish, so a warp
    may wait on a store held by any running warp but never on one not yet started."""
    rng = np.random.default_rng(7400)
    L, KV, P, v, n_tok = 32, 2, 16, 2048, 4096        # 16,384 segments of 32 KiB each way
    pages = n_tok // P
    NP = 2 * pages + 5
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:pages]], [n_tok]), Requests([perm[pages:2 * pages]], [n_tok])
    specs = wl.split_tokens(0, 0, n_tok, 256, 0, L, wl.LAYER_MAJOR)
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    dpool = DevicePool.empty(L, KV, NP, P, v)
    dpool.fill_random(7401)
    arena = Arena(nbytes, "host")
    pre = dpool.host_copy()
    kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array,
                             kvx.chunks_array(specs, arena.ptr), 0, L, cfg(0, 4, 1024, 8, 0),
                             stream.cuda_stream)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert kvx.kvx_last_launch(ctx)[1] == 4 * n_sms
    exp = np.full(nbytes + 4096, CANARY, np.uint8)
    oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
    assert_bytes_equal(arena.numpy(), exp, "round trip, oversubscribed grid")
    oracle.load(pre, dst.oracle(), oracle_chunks(specs, exp))
    assert_pool_equal(dpool, pre)
    arena.close()
