"""Host-side tests of libkvx.so that need no GPU: symbols, validation, counting, policy."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from paged_kv_gather_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
build()
from paged_kv_gather_gb300 import kvx  # noqa: E402
from paged_kv_gather_gb300 import workloads as wl  # noqa: E402

GOLDEN = os.path.join(ROOT, "tests", "golden")


def header_symbols():
    text = open(os.path.join(ROOT, "include", "kvx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvx_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = header_symbols()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", kvx.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvx_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in names:
        assert hasattr(kvx.raw(), n)
    assert sorted(kvx.EXPORTED) == names, "binding and header disagree"


def test_version_and_status_strings():
    assert kvx.kvx_version() == 2
    seen = set()
    for st in range(9):
        s = kvx.kvx_status_string(st)
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 9
    assert kvx.kvx_status_string(99) == "unknown status"


# ----------------------------------------------------------------------------- fixtures

class FakeBatch:
    """Pointers only: host logic never dereferences pool or chunk memory."""

    def __init__(self, L=4, KV=2, P=16, num_pages=64, v=256):
        self.L, self.KV, self.P, self.num_pages, self.v = L, KV, P, num_pages, v
        base = 1 << 40
        layer = num_pages * P * v
        self.pool = kvx.Pool(L, KV, P, num_pages, v, [base + l * layer for l in range(L)],
                             [base + (L + l) * layer for l in range(L)] if KV == 2 else None)

    def reqs(self, tables, host=True):
        return kvx.requests_array([(0x1000 + 0x100000 * i, t if host else None, n)
                                   for i, (t, n) in enumerate(tables)])

    @staticmethod
    def chunks(specs, base=1 << 44):
        a = np.zeros(len(specs), kvx.CHUNK_DTYPE)
        for i, (r, t0, n, l0, nl, layout, off) in enumerate(specs):
            a[i] = (r, t0, n, l0, nl, layout, base + off)
        return a


def _v(batch, reqs, chunks, lb=0, le=None, op=kvx.KVX_OP_STORE, level=1):
    return kvx.kvx_validate(batch.pool, reqs, chunks, lb, le, op, level)


def test_validate_accepts_a_good_batch():
    b = FakeBatch()
    reqs = b.reqs([(np.arange(8, dtype=np.int32), 128)])
    ch = b.chunks([(0, 0, 64, 0, 4, 0, 0), (0, 64, 64, 0, 4, 1, 1 << 20)])
    for op in range(4):
        for level in (0, 1, 2):
            assert _v(b, reqs, ch, op=op, level=level)[0] == kvx.KVX_OK


@pytest.mark.parametrize("case,status", [
    ("token_bytes", kvx.KVX_ERR_ALIGNMENT),
    ("chunk_align", kvx.KVX_ERR_ALIGNMENT),
    ("request_index", kvx.KVX_ERR_INVALID_ARG),
    ("token_range", kvx.KVX_ERR_INVALID_ARG),
    ("layer_range", kvx.KVX_ERR_INVALID_ARG),
    ("window", kvx.KVX_ERR_INVALID_ARG),
    ("layout", kvx.KVX_ERR_INVALID_ARG),
    ("null_chunk", kvx.KVX_ERR_INVALID_ARG),
    ("negative", kvx.KVX_ERR_INVALID_ARG),
    ("null_table", kvx.KVX_ERR_INVALID_ARG),
    ("page_bytes", kvx.KVX_ERR_INVALID_ARG),
    ("token_bytes_max", kvx.KVX_ERR_INVALID_ARG),
])
def test_validate_rejects(case, status):
    b = FakeBatch(v=40 if case == "token_bytes" else 256)
    if case == "page_bytes":  # a page of 2^16 tokens x 512 KiB = 32 GiB
        b = FakeBatch(P=1 << 16, v=1 << 19)
    elif case == "token_bytes_max":  # one token of 2 GiB in a page of one
        b = FakeBatch(P=1, v=1 << 31)
    reqs = b.reqs([(np.arange(8, dtype=np.int32), 128)])
    spec = [0, 0, 64, 0, 4, 0, 0]
    lb, le = 0, None
    if case == "chunk_align":
        spec[6] = 8
    elif case == "request_index":
        spec[0] = 1
    elif case == "token_range":
        spec[1], spec[2] = 100, 64
    elif case == "layer_range":
        spec[3], spec[4] = 2, 3
    elif case == "window":
        lb, le = 3, 2
    elif case == "layout":
        spec[5] = 3
    elif case == "negative":
        spec[2] = -1
    elif case == "null_table":
        reqs = kvx.requests_array([(0, None, 128)])
    ch = b.chunks([tuple(spec)])
    if case == "null_chunk":
        ch["ptr"] = 0
    st, msg = _v(b, reqs, ch, lb, le)
    assert st == status, msg
    assert msg


def test_validate_level2_page_ids_and_overlap():
    b = FakeBatch()
    bad = np.arange(8, dtype=np.int32)
    bad[5] = 64
    reqs = b.reqs([(bad, 128)])
    ch = b.chunks([(0, 0, 128, 0, 4, 0, 0)])
    assert _v(b, reqs, ch, level=1)[0] == kvx.KVX_OK  # level 1 does not read page tables
    st, msg = _v(b, reqs, ch, level=2)
    assert st == kvx.KVX_ERR_PAGE_OUT_OF_RANGE and "64" in msg

    # Two requests sharing page 3 at the same slot: a load that writes both overlaps.
    t1 = np.array([0, 1, 2, 3], np.int32)
    t2 = np.array([3, 4], np.int32)
    reqs = b.reqs([(t1, 64), (t2, 32)])
    both = b.chunks([(0, 48, 16, 0, 4, 0, 0), (1, 0, 16, 0, 4, 0, 1 << 20)])
    assert _v(b, reqs, both, op=kvx.KVX_OP_LOAD, level=2)[0] == kvx.KVX_ERR_OVERLAP
    assert _v(b, reqs, both, op=kvx.KVX_OP_SCATTER_HBM, level=2)[0] == kvx.KVX_ERR_OVERLAP
    # A store may read one slot twice.
    assert _v(b, reqs, both, op=kvx.KVX_OP_STORE, level=2)[0] == kvx.KVX_OK
    # Same slots but disjoint layers: per-layer chunks of a streamed load are fine.
    per_layer = b.chunks([(0, 48, 16, 0, 2, 0, 0), (1, 0, 16, 2, 2, 0, 1 << 20)])
    assert _v(b, reqs, per_layer, op=kvx.KVX_OP_LOAD, level=2)[0] == kvx.KVX_OK
    # ... unless the call's layer windows make them meet: here they do not.
    assert _v(b, reqs, per_layer, 1, 3, op=kvx.KVX_OP_LOAD, level=2)[0] == kvx.KVX_OK
    # Overlap inside one chunk list of one request (two chunks over the same tokens).
    dup = b.chunks([(0, 0, 32, 0, 4, 0, 0), (0, 16, 32, 3, 1, 1, 1 << 20)])
    assert _v(b, reqs, dup, op=kvx.KVX_OP_LOAD, level=2)[0] == kvx.KVX_ERR_OVERLAP
    assert _v(b, reqs, dup, 0, 3, op=kvx.KVX_OP_LOAD, level=2)[0] == kvx.KVX_OK


def _golden(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        f = line.split("#")[0].split()
        if f:
            rows[f[0]] = [int(x) for x in f[1:]]
    return rows


def test_plan_count_reproduces_per_page_dma_example():
    g = _golden("strata_dma_count.txt")
    T, P, L = g["tokens"][0], g["page_size"][0], g["layers"][0]
    b = FakeBatch(L=L, KV=1, P=P, num_pages=T // P, v=2048)
    reqs = b.reqs([(np.arange(T // P, dtype=np.int32), T)])
    one = b.chunks([(0, 0, T, 0, L, 0, 0)])
    segs, nbytes = kvx.kvx_plan_count(b.pool, reqs, one)
    assert segs == g["copies_per_request"][0]
    assert nbytes == T * L * 2048
    for layer in (0, 17, L - 1):
        assert kvx.kvx_plan_count(b.pool, reqs, one, layer, layer + 1)[0] == \
            g["copies_per_layer"][0]
    # One chunk per page gives the same count: chunking at page boundaries adds no copy.
    per_page = b.chunks([(0, p * P, P, 0, L, 0, p * L * P * 2048) for p in range(T // P)])
    assert kvx.kvx_plan_count(b.pool, reqs, per_page)[0] == g["copies_per_request"][0]


def _pool_for(shape):
    return kvx.Pool(shape.num_layers, shape.kv_factor, shape.page_size, shape.num_pages,
                    shape.token_bytes, [1 << 40] * shape.num_layers,
                    [1 << 41] * shape.num_layers if shape.kv_factor == 2 else None)


def test_plan_count_of_workloads():
    w = wl.llama8b()
    pool = _pool_for(w.shape)
    reqs = kvx.requests_array([(0x1000, None, w.load_requests[0].n_tokens)])
    ch = kvx.chunks_array(w.load_chunks, 1 << 44)
    assert kvx.kvx_plan_count(pool, reqs, ch) == (131072, 4 << 30)
    for P in wl.MLA_PAGE_SIZES:
        for C in wl.MLA_CHUNK_BYTES:
            w = wl.mla_sweep(P, C)
            pool = _pool_for(w.shape)
            reqs = kvx.requests_array([(0x1000, None, 16384)])
            ch = kvx.chunks_array(w.load_chunks, 1 << 44)
            segs, nbytes = kvx.kvx_plan_count(pool, reqs, ch)
            assert nbytes == 1151336448
            expect = 61 * sum((c.token_begin + c.n_tokens - 1) // P - c.token_begin // P + 1
                              for c in w.load_chunks if c.layer_begin == 0)
            assert segs == expect
            if P == 1:
                assert segs == 999424
            if C % (P * 1152) == 0:
                assert segs == 61 * (16384 // P)


def test_chunk_policy_properties():
    for w in (wl.tiny(), wl.llama8b(), wl.llama70b(), wl.qwen7b_batch(), wl.mla_sweep(1),
              wl.mla_sweep(64)):
        pool = _pool_for(w.shape)
        s = w.shape
        for streaming in (False, True):
            for target in (0, 64 << 10, 1 << 20, 4 << 20, 64 << 20):
                tpc, lpc = kvx.kvx_chunk_policy(pool, streaming, target)
                assert tpc > 0 and tpc % s.page_size == 0
                assert lpc == (1 if streaming else s.num_layers)
                chunk = tpc * lpc * s.kv_factor * s.token_bytes
                page = s.page_size * lpc * s.kv_factor * s.token_bytes
                eff = target or (2 << 20)
                if page <= eff:
                    assert chunk <= eff < chunk + page
                else:
                    assert tpc == s.page_size
    with pytest.raises(kvx.KvxError):
        kvx.kvx_chunk_policy(_pool_for(wl.tiny().shape), False, -1)


def test_chunk_and_request_dtypes_match_c_structs():
    assert kvx.CHUNK_DTYPE.itemsize == ctypes.sizeof(kvx.kvx_chunk) == 32
    assert kvx.REQUEST_DTYPE.itemsize == ctypes.sizeof(kvx.kvx_request) == 24
    for name, _ in kvx.kvx_chunk._fields_:
        assert kvx.CHUNK_DTYPE.fields[name][1] == getattr(kvx.kvx_chunk, name).offset
    for name, _ in kvx.kvx_request._fields_:
        assert kvx.REQUEST_DTYPE.fields[name][1] == getattr(kvx.kvx_request, name).offset


# ----------------------------------------------------------------------------- estimator

def test_estimator_littles_law_and_link_cap():
    m = kvx.kvx_default_link_model()
    N = 4 << 30
    prev = 0.0
    for cap in (1, 2, 4, 8, 16, 32, 0):
        c = kvx.kvx_launch_cfg()
        c.sm_cap, c.ctas_per_sm, c.threads, c.unroll = cap, 1, 1024, 8
        us = kvx.kvx_estimate_us(m, kvx.KVX_OP_LOAD, N, c)
        gbs = N / ((us - m.launch_us) * 1e3)
        sms = cap if cap else m.num_sms
        # X = C * S / L with 1024 threads x 8 units x 16 B in flight per SM, capped by the link.
        assert gbs == pytest.approx(min(m.h2d_gbs, sms * 1024 * 8 * 16 / (m.latency_us * 1e3)))
        assert gbs >= prev
        prev = gbs
    # Halving the bytes in flight halves the Little's-law rate below the cap.
    c = kvx.kvx_launch_cfg()
    c.sm_cap, c.ctas_per_sm, c.threads, c.unroll = 2, 1, 1024, 4
    us = kvx.kvx_estimate_us(m, kvx.KVX_OP_STORE, N, c)
    assert N / ((us - m.launch_us) * 1e3) == pytest.approx(2 * 1024 * 4 * 16 / 2600.0)
    # The bulk mapping keeps its two rings' loading stages in flight: 2 x (stages - 1) x
    # stage_bytes per CTA, whatever the thread count.
    c = kvx.kvx_launch_cfg()
    c.sm_cap, c.ctas_per_sm, c.mapping, c.unroll, c.stage_bytes = 1, 1, kvx.KVX_MAP_BULK, 3, 32768
    us = kvx.kvx_estimate_us(m, kvx.KVX_OP_LOAD, N, c)
    assert N / ((us - m.launch_us) * 1e3) == pytest.approx(2 * 2 * 32768 / 2600.0)
    c.unroll, c.stage_bytes = 0, 0  # the bulk defaults: 3 stages of 32 KiB
    assert kvx.kvx_estimate_us(m, kvx.KVX_OP_LOAD, N, c) == pytest.approx(us)
    c.sm_cap = 4
    us = kvx.kvx_estimate_us(m, kvx.KVX_OP_LOAD, N, c)
    assert N / ((us - m.launch_us) * 1e3) == pytest.approx(min(m.h2d_gbs, 4 * 4 * 32768 / 2600.0))
    # Without a configuration: the defaults, a store on 8 SMs and a load on 16 (both already
    # at their link's peak by Little's law).
    for op, sms in ((kvx.KVX_OP_STORE, 8), (kvx.KVX_OP_LOAD, 16)):
        c = kvx.kvx_launch_cfg()
        c.sm_cap, c.ctas_per_sm, c.threads, c.unroll = sms, 1, 1024, 8
        assert kvx.kvx_estimate_us(m, op, N, None) == pytest.approx(
            kvx.kvx_estimate_us(m, op, N, c))
    c.sm_cap = 2  # a quarter of the store's default grid: below the D2H peak
    assert kvx.kvx_estimate_us(m, kvx.KVX_OP_STORE, N, c) > kvx.kvx_estimate_us(
        m, kvx.KVX_OP_STORE, N, None)
    # The HBM transform moves 2N through HBM at the copy peak, whatever the SM cap.
    us = kvx.kvx_estimate_us(m, kvx.KVX_OP_GATHER_HBM, N, None)
    assert us == pytest.approx(m.launch_us + 2 * N / (m.hbm_gbs * 1e3))
    with pytest.raises(kvx.KvxError):
        kvx.kvx_estimate_us(m, 7, N, None)


def test_estimator_layer_streaming_bounds():
    # Loading-bound (io > compute): e2e = L * io + compute; the compute stream waits for
    # the first load and then io - compute per layer.
    e2e, bubble = kvx.kvx_estimate_stream_us(1290.0, 560.0, 80)
    assert e2e == pytest.approx(1290 + 79 * 1290 + 560)
    assert bubble == pytest.approx(1290 + 79 * 730)
    assert e2e >= max(80 * 1290, 80 * 560)
    # Compute-bound: only the first load is exposed.
    e2e, bubble = kvx.kvx_estimate_stream_us(300.0, 560.0, 80)
    assert e2e == pytest.approx(300 + 79 * 560 + 560)
    assert bubble == pytest.approx(300)
    # One layer: load then compute.
    assert kvx.kvx_estimate_stream_us(5.0, 7.0, 1) == (12.0, 5.0)
    with pytest.raises(kvx.KvxError):
        kvx.kvx_estimate_stream_us(1.0, 1.0, 0)


def test_estimator_exchange_and_round_trip():
    m = kvx.kvx_default_link_model()
    X, R = kvx.KVX_OP_EXCHANGE, kvx.KVX_OP_ROUNDTRIP
    G = 1 << 30
    launch = m.launch_us
    # Exchange: each direction capped by its own peak, both by the bidirectional peak.
    assert kvx.kvx_estimate_pair_us(m, X, 4 * G, 4 * G) == pytest.approx(
        launch + 8 * G / m.bidir_gbs * 1e-3)
    assert kvx.kvx_estimate_pair_us(m, X, 4 * G, 0) == pytest.approx(
        launch + 4 * G / m.d2h_gbs * 1e-3)
    assert kvx.kvx_estimate_pair_us(m, X, 0, 4 * G) == pytest.approx(
        launch + 4 * G / m.h2d_gbs * 1e-3)
    # A small store beside a large load: the load's own peak decides.
    assert kvx.kvx_estimate_pair_us(m, X, G, 10 * G) == pytest.approx(
        launch + 10 * G / m.h2d_gbs * 1e-3)
    # Round trip: fill and drain of one unit per warp (16 SMs x 32 warps x 32 KiB = 16 MiB).
    F = 16 * 32 * (32 << 10)
    want = launch + (F / m.d2h_gbs + (8 * G - 2 * F) / m.bidir_gbs + F / m.h2d_gbs) * 1e-3
    assert kvx.kvx_estimate_pair_us(m, R, 4 * G, 4 * G, 32 << 10) == pytest.approx(want)
    # The fill never exceeds the transfer: a tiny round trip is one store then one load.
    tiny = 1 << 20
    assert kvx.kvx_estimate_pair_us(m, R, tiny, tiny, 32 << 10) == pytest.approx(
        launch + (tiny / m.d2h_gbs + tiny / m.h2d_gbs) * 1e-3)
    # Too few bytes in flight: Little's law caps both directions together.
    c = kvx.kvx_launch_cfg()
    c.sm_cap, c.ctas_per_sm, c.threads, c.unroll = 1, 1, 32, 1
    little = 32 * 16 / (m.latency_us * 1e3)
    assert kvx.kvx_estimate_pair_us(m, X, G, G, 0, c) == pytest.approx(
        launch + 2 * G / little * 1e-3)
    for bad in ((kvx.KVX_OP_STORE, G, G), (R, G, 2 * G), (X, -1, G)):
        with pytest.raises(kvx.KvxError):
            kvx.kvx_estimate_pair_us(m, *bad)


def test_binding_rejects_malformed_inputs():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):  # not in device memory
        kvx.Pool.from_tensor(torch.zeros((2, 1, 4, 16, 64), dtype=torch.uint8), 16)
    with pytest.raises(ValueError):  # wrong rank
        kvx.Pool.from_tensor(torch.zeros((1, 4, 16, 64), dtype=torch.uint8), 16)
    with pytest.raises(ValueError):  # wrong element size
        kvx.Pool.from_tensor(torch.zeros((2, 1, 4, 16, 64), dtype=torch.float32), 16)
    pool = kvx.Pool(1, 1, 16, 4, 64, [0x1000], None)
    reqs = kvx.requests_array([(0x2000, None, 16)])
    bad = np.zeros(2, dtype=np.int64)  # not the chunk struct dtype
    with pytest.raises(ValueError):
        kvx.kvx_validate(pool, reqs, bad)


def test_oracle_and_library_share_nothing():
    """The CUDA path and the oracle are independent: neither imports, includes or links the
    other, and the package's source never names the oracle."""
    import pathlib
    import re
    root = pathlib.Path(__file__).resolve().parents[1]
    pkg = root / "paged_kv_gather_gb300"
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")) + \
            list(pkg.rglob("*.cpp")) + list(pkg.rglob("*.h")) + [root / "include" / "kvx.h"]:
        text = f.read_text()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
        assert "kv_oracle" not in text, f
    for f in (root / "oracle").glob("*"):
        if f.suffix in (".py", ".c"):
            text = f.read_text()
            assert not re.search(r"^\s*(import|from)\s+paged_kv_gather_gb300", text, re.M), f
            assert "libkvx" not in text and '#include "kvx' not in text, f


def test_binding_fails_loudly_without_the_library(tmp_path):
    """The binding, away from its built library, refuses to import (no CPU fallback)."""
    import shutil
    import subprocess
    import sys
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "paged_kv_gather_gb300", "kvx.py")
    shutil.copy(src, tmp_path / "kvx_copy.py")
    code = ("import importlib.util as u; "
            "s = u.spec_from_file_location('kvx_copy', %r); "
            "m = u.module_from_spec(s); s.loader.exec_module(m)") % str(tmp_path / "kvx_copy.py")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert r.returncode != 0 and "is missing" in r.stderr, r.stderr[-500:]


def test_roundtrip_unit_follows_segment_size():
    """kvx_roundtrip_unit reports the round trip's own unit rule: about 8 KiB units on 32 SMs
    for segments under 8 KiB, one segment per unit up to 32 KiB (32 SMs under 16 KiB), row
    slices of at most 32 KiB beyond; an explicit configuration keeps its SM cap, and its
    batch if it gives one."""
    u = kvx.kvx_roundtrip_unit
    assert u(1, 1152) == (8 * 1152, 32)       # 8 one-token segments per unit
    assert u(2, 1152) == (4 * 2304, 32)
    assert u(4, 1152) == (2 * 4608, 32)
    assert u(8, 1152) == (9216, 32)            # one 9 KiB segment, still short: 32 SMs
    assert u(16, 1152) == (18432, 16)          # 18 KiB: one per unit on 16 SMs
    assert u(16, 2048) == (32768, 16)          # llama8b pages
    assert u(32, 1152) == (16 * 1152, 16)      # 36 KiB: two slices of 16 rows
    assert u(64, 1152) == (22 * 1152, 16)      # 72 KiB: three slices of at most 22 rows
    assert u(4, 65536) == (65536, 16)          # rows longer than 32 KiB: one row per slice
    c = kvx.kvx_launch_cfg()
    c.sm_cap, c.ctas_per_sm, c.threads, c.unroll = 16, 1, 1024, 8
    assert u(16, 256, c) == (8 * 4096, 16)     # given 16 SMs: the 32 KiB units of one-way
    assert u(1, 1152, c) == (29 * 1152, 16)
    c.batch = 3
    assert u(16, 256, c) == (3 * 4096, 16)
    assert u(64, 1152, c) == (3 * 73728, 16)   # an explicit batch keeps whole segments
    c.batch, c.sm_cap = 0, 0                   # every SM
    assert u(1, 1152, c, num_sms=152) == (8 * 1152, 0)
    assert u(1, 1152, c, num_sms=16) == (29 * 1152, 0)
    for bad in [(0, 1152), (16, 0), (-1, 64)]:
        with pytest.raises(kvx.KvxError):
            u(*bad)
    with pytest.raises(kvx.KvxError):
        u(16, 1152, None, 0)

