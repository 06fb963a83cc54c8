"""Overlapped launches (kvx_launch_cfg.overlap, programmatic dependent launch): consecutive
per-layer transfers may start while the previous one drains, yet still complete in stream
order, and every byte still matches the oracle."""
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
from tests.gpu_common import (Arena, DevicePool, Requests, assert_bytes_equal,  # noqa: E402
                              assert_pool_equal, expected_load, expected_store, oracle_chunks)

L, KV, P, V, T = 8, 1, 16, 1152, 1024  # an MLA-like latent cache, 64 pages per request


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


def _overlap_cfg(ctx, op):
    c = kvx.kvx_default_launch_cfg(ctx, op)
    c.overlap = 1
    return c


def _layer_case(seed):
    """Per-layer chunks (four of 256 tokens per layer, all three layouts) of one request,
    its source pages and a disjoint destination page set."""
    rng = np.random.default_rng(seed)
    npg = T // P
    NP = 2 * npg + 5
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:npg]], [T]), Requests([perm[npg:2 * npg]], [T])
    specs = []
    for layer in range(L):
        specs += wl.split_tokens(0, 0, T, 256, layer, 1, layer % 3)
    shape = wl.KVShape(L, KV, 1, V, "fp8_e4m3", P, NP)  # token_bytes == V
    wl.place_chunks(specs, shape, align=wl.STRIPE_ALIGN)
    return NP, src, dst, specs, wl._arena_bytes(specs, shape)


def test_overlapped_layer_load_plans_complete_in_order(ctx, stream):
    """Eight per-layer load plans launched to overlap: an event recorded after the fourth
    means layers 0-3 are complete (another stream copies them while later layers may still
    be loading); every layer matches the oracle, launched directly and replayed from a
    CUDA graph onto fresh destination pages."""
    NP, src, dst, specs, nbytes = _layer_case(9100)
    dpool = DevicePool.empty(L, KV, NP, P, V)
    dpool.fill_random(9101)
    arena = Arena(nbytes, "host")
    ch = kvx.chunks_array(specs, arena.ptr)
    kvx.kvx_store_chunks(ctx, dpool.pool, src.array, ch, stream=stream.cuda_stream)
    stream.synchronize()
    assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), "store")
    c = _overlap_cfg(ctx, kvx.KVX_OP_LOAD)
    plans = [kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, dpool.pool, dst.array, ch, layer,
                                 layer + 1, c, stream.cuda_stream) for layer in range(L)]
    graph = None
    try:
        for round_ in range(2):
            dpool.fill_random(9102 + round_)
            pre = dpool.host_copy()
            exp = expected_load(pre, dst, specs, arena.numpy().copy())
            side = torch.cuda.Stream()
            if round_ == 0:
                ev = torch.cuda.Event()
                for layer, plan in enumerate(plans):
                    kvx.kvx_plan_launch(plan, stream.cuda_stream)
                    if layer == 3:
                        ev.record(stream)
                side.wait_event(ev)
                with torch.cuda.stream(side):
                    early = dpool.tensor[:, :4].clone()
            else:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    cs = torch.cuda.current_stream().cuda_stream
                    for plan in plans:
                        kvx.kvx_plan_launch(plan, cs)
                with torch.cuda.stream(stream):
                    graph.replay()
            torch.cuda.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            if round_ == 0:
                got = early.cpu().numpy()
                for layer in range(4):
                    assert np.array_equal(got[0, layer], exp.pools[0][layer]), \
                        f"layer {layer} not complete at the event after layer 3"
            assert_pool_equal(dpool, exp)
    finally:
        del graph
        torch.cuda.synchronize()
        for plan in plans:
            kvx.kvx_plan_destroy(plan)
        arena.close()


@pytest.mark.parametrize("op", ["store", "load", "gather", "scatter"])
def test_overlapped_per_layer_calls(ctx, stream, op):
    """Per-layer calls of each single-transfer operation launched to overlap, against the
    oracle (host chunks for store and load, device chunks for the transform)."""
    NP, src, dst, specs, nbytes = _layer_case(9200)
    dpool = DevicePool.empty(L, KV, NP, P, V)
    dpool.fill_random(9201)
    where = "host" if op in ("store", "load") else "device"
    arena = Arena(nbytes, where)
    ch = kvx.chunks_array(specs, arena.ptr)
    if op in ("store", "gather"):
        kop = kvx.KVX_OP_STORE if op == "store" else kvx.KVX_OP_GATHER_HBM
        c = _overlap_cfg(ctx, kop)
        for layer in range(L):
            if op == "store":
                kvx.kvx_store_chunks(ctx, dpool.pool, src.array, ch, layer, layer + 1, c,
                                     stream.cuda_stream)
            else:
                kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, dpool.pool, src.array, ch, layer,
                                      layer + 1, c, stream.cuda_stream)
        stream.synchronize()
        assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
        assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), op)
    else:
        data = np.random.default_rng(9202).integers(0, 256, nbytes + 4096, dtype=np.uint8)
        arena.write(data)
        torch.cuda.synchronize()
        pre = dpool.host_copy()
        kop = kvx.KVX_OP_LOAD if op == "load" else kvx.KVX_OP_SCATTER_HBM
        c = _overlap_cfg(ctx, kop)
        for layer in range(L):
            if op == "load":
                kvx.kvx_load_chunks(ctx, dpool.pool, dst.array, ch, layer, layer + 1, c,
                                    stream.cuda_stream)
            else:
                kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, dpool.pool, dst.array, ch,
                                      layer, layer + 1, c, stream.cuda_stream)
        stream.synchronize()
        assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
        oracle.load(pre, dst.oracle(), oracle_chunks(specs, data.copy()))
        assert_pool_equal(dpool, pre)
    arena.close()


def test_overlapped_layer_load_calls_complete_in_order(ctx, stream):
    """Per-layer load calls launched to overlap, three passes back to back onto the same
    pages: an event recorded after the fourth layer of the last pass means layers 0-3 hold
    that pass's bytes (each pass loads other host bytes), and the whole pool matches the
    oracle."""
    NP, src, dst, specs, nbytes = _layer_case(9300)
    dpool = DevicePool.empty(L, KV, NP, P, V)
    dpool.fill_random(9301)
    pre = dpool.host_copy()
    arenas = [Arena(nbytes, "host") for _ in range(3)]
    try:
        datas = []
        for i, a in enumerate(arenas):
            d = np.random.default_rng(9302 + i).integers(0, 256, nbytes + 4096, dtype=np.uint8)
            a.write(d)
            datas.append(d)
        torch.cuda.synchronize()
        c = _overlap_cfg(ctx, kvx.KVX_OP_LOAD)
        ev = torch.cuda.Event()
        for i, a in enumerate(arenas):
            ch = kvx.chunks_array(specs, a.ptr)
            for layer in range(L):
                kvx.kvx_load_chunks(ctx, dpool.pool, dst.array, ch, layer, layer + 1, c,
                                    stream.cuda_stream)
                if i == 2 and layer == 3:
                    ev.record(stream)
        side = torch.cuda.Stream()
        side.wait_event(ev)
        with torch.cuda.stream(side):
            early = dpool.tensor[:, :4].clone()
        torch.cuda.synchronize()
        assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
        oracle.load(pre, dst.oracle(), oracle_chunks(specs, datas[-1].copy()))
        got = early.cpu().numpy()
        for layer in range(4):
            assert np.array_equal(got[0, layer], pre.pools[0][layer]), \
                f"layer {layer} not complete at the event after layer 3"
        assert_pool_equal(dpool, pre)
    finally:
        for a in arenas:
            a.close()


@pytest.mark.parametrize("op", ["store", "load"])
def test_overlapped_token_major_layer_calls(ctx, stream, op):
    """Per-layer calls on token-major chunks of K and V (pages of strided rows: the
    row-walking kernel's overlapped variant), against the oracle."""
    rng = np.random.default_rng(9400)
    KV2, npg = 2, T // P
    NP = 2 * npg + 3
    perm = rng.permutation(NP).astype(np.int32)
    src, dst = Requests([perm[:npg]], [T]), Requests([perm[npg:2 * npg]], [T])
    specs = []
    for layer in range(L):
        specs += wl.split_tokens(0, 0, T, 200, layer, 1, wl.TOKEN_MAJOR)
    shape = wl.KVShape(L, KV2, 1, V, "fp8_e4m3", P, NP)
    wl.place_chunks(specs, shape)
    nbytes = wl._arena_bytes(specs, shape)
    dpool = DevicePool.empty(L, KV2, NP, P, V)
    dpool.fill_random(9401)
    arena = Arena(nbytes, "host")
    try:
        ch = kvx.chunks_array(specs, arena.ptr)
        if op == "store":
            c = _overlap_cfg(ctx, kvx.KVX_OP_STORE)
            for layer in range(L):
                kvx.kvx_store_chunks(ctx, dpool.pool, src.array, ch, layer, layer + 1, c,
                                     stream.cuda_stream)
            stream.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            assert_bytes_equal(arena.numpy(), expected_store(dpool, src, specs, nbytes), op)
        else:
            data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
            arena.write(data)
            torch.cuda.synchronize()
            pre = dpool.host_copy()
            c = _overlap_cfg(ctx, kvx.KVX_OP_LOAD)
            for layer in range(L):
                kvx.kvx_load_chunks(ctx, dpool.pool, dst.array, ch, layer, layer + 1, c,
                                    stream.cuda_stream)
            stream.synchronize()
            assert kvx.kvx_get_status(ctx, stream.cuda_stream) == 0
            oracle.load(pre, dst.oracle(), oracle_chunks(specs, data.copy()))
            assert_pool_equal(dpool, pre)
    finally:
        arena.close()


def test_overlap_rejected_where_not_supported(ctx, stream):
    """overlap = 1 is refused, with nothing launched, outside single transfers on the
    warp-segment mapping: exchange, round trip, CTA and bulk mappings, the allocation-free
    load, and values other than 0 and 1."""
    NP, src, dst, specs, nbytes = _layer_case(9300)
    dpool = DevicePool.empty(L, KV, NP, P, V)
    dpool.fill_random(9301)
    before = dpool.tensor.clone()
    arena = Arena(nbytes, "host")
    ch = kvx.chunks_array(specs, arena.ptr)
    bad = []
    for op, mapping, value in [(kvx.KVX_OP_EXCHANGE, kvx.KVX_MAP_WARP_SEGMENT, 1),
                               (kvx.KVX_OP_ROUNDTRIP, kvx.KVX_MAP_WARP_SEGMENT, 1),
                               (kvx.KVX_OP_LOAD, kvx.KVX_MAP_CTA, 1),
                               (kvx.KVX_OP_LOAD, kvx.KVX_MAP_BULK, 1),
                               (kvx.KVX_OP_LOAD, kvx.KVX_MAP_WARP_SEGMENT, 2)]:
        c = kvx.kvx_default_launch_cfg(ctx, op)
        c.mapping, c.overlap = mapping, value
        bad.append((op, c))
    for op, c in bad:
        with pytest.raises(kvx.KvxError) as e:
            if op == kvx.KVX_OP_EXCHANGE:
                kvx.kvx_exchange_chunks(ctx, dpool.pool, src.array, ch, dst.array, ch[:0],
                                        cfg=c, stream=stream.cuda_stream)
            elif op == kvx.KVX_OP_ROUNDTRIP:
                kvx.kvx_roundtrip_chunks(ctx, dpool.pool, src.array, dst.array, ch, cfg=c,
                                         stream=stream.cuda_stream)
            else:
                kvx.kvx_load_chunks(ctx, dpool.pool, dst.array, ch, cfg=c,
                                    stream=stream.cuda_stream)
        assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_LOAD)
    c.overlap = 1
    with pytest.raises(kvx.KvxError) as e:
        kvx.kvx_load_chunks_noalloc(dpool.pool, dst.array, ch, cfg=c,
                                    stream=stream.cuda_stream)
    assert e.value.status == kvx.KVX_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(dpool.tensor, before)
    arena.close()
