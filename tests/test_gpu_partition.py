"""SM partitioning with green contexts: the I/O stream's transfers stay bit-exact and a GEMM
on the compute stream runs beside them."""
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
import oracle  # noqa: E402
from tests.gpu_common import (CANARY, Arena, DevicePool, Requests,  # noqa: E402
                              assert_bytes_equal, assert_pool_equal, expected_load,
                              oracle_chunks)


def test_partition_load_and_concurrent_gemm():
    part = kvx.kvx_partition_create(0, 8)
    try:
        n_sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert part.io_sms >= 8 and part.compute_sms > 0
        assert part.io_sms + part.compute_sms <= n_sms
        assert part.io_stream and part.compute_stream
        rng = np.random.default_rng(31)
        L, KV, P, v = 4, 2, 16, 2048
        lens = [1000, 777]
        pages = [-(-n // P) for n in lens]
        NP = sum(pages) + 5
        perm = rng.permutation(NP).astype(np.int32)
        tables, at = [], 0
        for npg in pages:
            tables.append(perm[at:at + npg])
            at += npg
        specs = []
        for r, n in enumerate(lens):
            specs += wl.split_tokens(r, 0, n, 200, 0, L, r % 3)
        shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
        wl.place_chunks(specs, shape)
        nbytes = wl._arena_bytes(specs, shape)
        arena = Arena(nbytes, "host")
        data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
        arena.write(data)
        reqs = Requests(tables, lens)
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(32)
        pre = dpool.host_copy()
        torch.cuda.synchronize()
        ctx = kvx.kvx_create(0)
        A = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
        B = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
        ref = A @ B
        torch.cuda.synchronize()  # A and B were made on the current stream
        compute = torch.cuda.ExternalStream(part.compute_stream)
        with torch.cuda.stream(compute):
            C = A @ B
        kvx.kvx_load_chunks(ctx, dpool.pool, reqs.array, kvx.chunks_array(specs, arena.ptr),
                            cfg=None, stream=part.io_stream)
        torch.cuda.synchronize()
        compute.synchronize()
        assert kvx.kvx_get_status(ctx, part.io_stream) == 0
        assert_pool_equal(dpool, expected_load(pre, reqs, specs, data.copy()))
        assert torch.equal(C, ref)
        kvx.kvx_destroy(ctx)
        arena.close()
    finally:
        part.close()


def test_two_io_partitions_store_and_load_at_once():
    """Two I/O partitions plus compute: a store on one and a load on the other run at the
    same time on disjoint SM sets, both bit-exact."""
    part = kvx.kvx_partition_create(0, 8, io_groups=2)
    try:
        assert len(part.io_streams) == 2 and all(part.io_sms_list[g] >= 8 for g in range(2))
        rng = np.random.default_rng(41)
        L, KV, P, v, T = 3, 2, 16, 2048, 900
        pages = -(-T // P)
        NP = 2 * pages + 4
        perm = rng.permutation(NP).astype(np.int32)
        src, dst = Requests([perm[:pages]], [T]), Requests([perm[pages:2 * pages]], [T])
        specs = wl.split_tokens(0, 0, T, 256, 0, L, wl.LAYER_MAJOR)
        shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, NP)
        wl.place_chunks(specs, shape)
        nbytes = wl._arena_bytes(specs, shape)
        out, inp = Arena(nbytes, "host"), Arena(nbytes, "host")
        data = rng.integers(0, 256, nbytes + 4096, dtype=np.uint8)
        inp.write(data)
        dpool = DevicePool.empty(L, KV, NP, P, v)
        dpool.fill_random(42)
        pre = dpool.host_copy()
        ctx_a, ctx_b = kvx.kvx_create(0), kvx.kvx_create(0)
        kvx.kvx_store_chunks(ctx_a, dpool.pool, src.array, kvx.chunks_array(specs, out.ptr),
                             stream=part.io_streams[0])
        kvx.kvx_load_chunks(ctx_b, dpool.pool, dst.array, kvx.chunks_array(specs, inp.ptr),
                            stream=part.io_streams[1])
        torch.cuda.synchronize()
        assert kvx.kvx_get_status(ctx_a, part.io_streams[0]) == 0
        assert kvx.kvx_get_status(ctx_b, part.io_streams[1]) == 0
        exp = np.full(nbytes + 4096, CANARY, np.uint8)
        oracle.store(pre, src.oracle(), oracle_chunks(specs, exp))
        assert_bytes_equal(out.numpy(), exp, "store on I/O partition 0")
        assert_pool_equal(dpool, expected_load(pre, dst, specs, data.copy()))
        kvx.kvx_destroy(ctx_a)
        kvx.kvx_destroy(ctx_b)
        out.close()
        inp.close()
    finally:
        torch.cuda.synchronize()
        part.close()


def test_partition_rejects_bad_sizes():
    with pytest.raises(kvx.KvxError):
        kvx.kvx_partition_create(0, 0)
    with pytest.raises(kvx.KvxError):
        kvx.kvx_partition_create(0, 100000)
