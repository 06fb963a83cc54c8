"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these re-types the oracle's address arithmetic.  The expected values come from:
  * P-a  brute force with identity tags: every token vector carries a tag that names its
         logical (request, layer, kv, token, word); the pool is filled through the page
         table (PagedAttention's definition) and the chunk is read through a numpy
         reshape in the layout's axis order, so a wrong index, a dropped term or a
         transposed axis in the oracle shows up as a misplaced tag;
  * P-b  exactly-once with canaries: every tag lands once, nothing else is touched;
  * P-c  round trip store -> load into a disjoint page set, and load -> store;
  * P-d  closed-form byte counts (tests/golden/closed_form_bytes.txt);
  * P-e  library routines: numpy fancy indexing and stack/transpose; the identity page
         table reduces to a plain copy; one-page chunks with K/V folded reproduce the
         index mapping of the GPU-assisted load kernel printed in "Strata Guide:
         Hierarchical Context Caching for Long LLMs", section "Step 1" (worked example in
         tests/golden/strata_load_index.txt).
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from oracle import LAYER_MAJOR, STRIPED, TOKEN_MAJOR, Chunk, Pool, Request
from paged_kv_gather_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CANARY32 = np.int32(np.uint32(0xA5A5A5A5).view(np.int32))


# ----------------------------------------------------------------------------- helpers

def empty_pool(L, KV, num_pages, P, v, fill=0xA5):
    return Pool([[np.full((num_pages, P, v), fill, np.uint8) for _ in range(L)]
                 for _ in range(KV)], P)


def tag(r, l, k, t, w, L, KV, T, W):
    """Unique positive int32 naming word w of (request r, layer l, kv k, token t)."""
    return (((r * L + l) * KV + k) * T + t) * W + w + 1


def fill_pool_with_tags(pool, reqs, Tmax):
    """Write each request's logical token t into slot page_table[t // P]*P + t % P."""
    L, KV, P, v = pool.num_layers, pool.kv_factor, pool.page_size, pool.token_bytes
    W = v // 4
    for r, req in enumerate(reqs):
        for l in range(L):
            for k in range(KV):
                words = pool.pools[k][l].view(np.int32)  # [pages, P, W]
                for t in range(req.n_tokens):
                    page = req.page_table[t // P]
                    words[page, t % P, :] = [tag(r, l, k, t, w, L, KV, Tmax, W)
                                             for w in range(W)]


def expected_chunk_words(c, r, L, KV, W, Tmax, lb, le):
    """Chunk contents by the layout definition, CANARY32 outside the layer window (and in
    the padding after each object of a STRIPED chunk)."""
    lr = np.arange(c.n_layers)[:, None, None, None]
    k = np.arange(KV)[None, :, None, None]
    tr = np.arange(c.n_tokens)[None, None, :, None]
    w = np.arange(W)[None, None, None, :]
    l = c.layer_begin + lr
    e = tag(r, l, k, c.token_begin + tr, w, L, KV, Tmax, W)
    e = np.broadcast_to(e, (c.n_layers, KV, c.n_tokens, W)).astype(np.int32).copy()
    in_window = (l >= lb) & (l < le)
    e = np.where(np.broadcast_to(in_window, e.shape), e, CANARY32)
    if c.layout == TOKEN_MAJOR:
        e = e.transpose(2, 0, 1, 3)  # [layer][kv][token] -> [token][layer][kv]
    if c.layout == STRIPED:
        # Each (layer, kv) object padded with canaries up to the next 4096-byte multiple.
        obj_words = c.n_tokens * W
        stride_words = -(-obj_words * 4 // 4096) * 4096 // 4
        padded = np.full((c.n_layers, KV, stride_words), CANARY32, np.int32)
        padded[:, :, :obj_words] = e.reshape(c.n_layers, KV, obj_words)
        e = padded
    return e.reshape(-1)


def make_chunks(specs, KV, v, pad=16):
    out = []
    for (r, t0, n, l0, nl, layout) in specs:
        buf = np.full(oracle.chunk_bytes(nl, KV, n, v, layout) + pad, 0xA5, np.uint8)
        out.append(Chunk(r, t0, n, l0, nl, layout, buf))
    return out


def chunk_words(c, KV, v):
    return c.buf[: oracle.chunk_bytes(c.n_layers, KV, c.n_tokens, v, c.layout)].view(np.int32)


def random_table(rng, n_pages_needed, num_pages):
    return rng.permutation(num_pages)[:n_pages_needed].astype(np.int32)


def check_store(pool, reqs, chunk_specs, lb, le, Tmax):
    L, KV, v = pool.num_layers, pool.kv_factor, pool.token_bytes
    W = v // 4
    chunks = make_chunks(chunk_specs, KV, v)
    oracle.store(pool, reqs, chunks, lb, le)
    for c in chunks:
        got = chunk_words(c, KV, v)
        exp = expected_chunk_words(c, c.request, L, KV, W, Tmax, lb, le)
        np.testing.assert_array_equal(got, exp)
        assert np.all(c.buf[got.nbytes:] == 0xA5), "wrote past the chunk end"
    return chunks


def check_load(L, KV, P, v, num_pages, reqs, chunk_specs, lb, le, Tmax):
    """Load tag-filled chunks into a canary pool; check slots, canaries, exactly-once."""
    W = v // 4
    pool = empty_pool(L, KV, num_pages, P, v)
    chunks = make_chunks(chunk_specs, KV, v)
    for c in chunks:
        words = chunk_words(c, KV, v)
        words[:] = expected_chunk_words(c, c.request, L, KV, W, Tmax, 0, L)
    oracle.load(pool, reqs, chunks, lb, le)
    # Expected pool, built from the PagedAttention definition slot by slot.
    exp = [[np.full((num_pages, P, W), CANARY32, np.int32) for _ in range(L)] for _ in range(KV)]
    for c in chunks:
        req = reqs[c.request]
        for l in range(max(lb, c.layer_begin), min(le, c.layer_begin + c.n_layers)):
            for k in range(KV):
                for t in range(c.token_begin, c.token_begin + c.n_tokens):
                    page = req.page_table[t // P]
                    exp[k][l][page, t % P, :] = [tag(c.request, l, k, t, w, L, KV, Tmax, W)
                                                 for w in range(W)]
    for k in range(KV):
        for l in range(L):
            np.testing.assert_array_equal(pool.pools[k][l].view(np.int32), exp[k][l])
    return pool


# ----------------------------------------------------------------------------- P-a

@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_bruteforce_all_injective_page_maps(P):
    """Every injective map of <= 3 logical pages into a 4-page pool, both layouts."""
    L, KV, v, num_pages = 2, 2, 16, 4
    for T in sorted({1, P, P + 1, 3 * P}):
        n_pages = -(-T // P)
        for perm in itertools.permutations(range(num_pages), n_pages):
            pt = np.array(perm, np.int32)
            reqs = [Request(pt, T)]
            for layout in (LAYER_MAJOR, TOKEN_MAJOR, STRIPED):
                pool = empty_pool(L, KV, num_pages, P, v)
                fill_pool_with_tags(pool, reqs, T)
                check_store(pool, reqs, [(0, 0, T, 0, L, layout)], 0, L, T)
                check_load(L, KV, P, v, num_pages, reqs, [(0, 0, T, 0, L, layout)], 0, L, T)


@pytest.mark.parametrize("KV,v", [(1, 16), (2, 16), (1, 32), (2, 64)])
def test_bruteforce_every_cut_and_layer_window(KV, v):
    """Two chunks cut at every position, every chunk layer range, every call window."""
    L, P = 3, 3
    T = 13
    num_pages = 8
    rng = np.random.default_rng(7 + KV * 100 + v)
    pt = random_table(rng, -(-T // P), num_pages)
    reqs = [Request(pt, T)]
    pool = empty_pool(L, KV, num_pages, P, v)
    fill_pool_with_tags(pool, reqs, T)
    layer_ranges = [(a, b - a) for a in range(L) for b in range(a + 1, L + 1)]
    windows = [(a, b) for a in range(L + 1) for b in range(a, L + 1)]
    for cut in range(T + 1):
        layout = cut % 3
        l0, nl = layer_ranges[cut % len(layer_ranges)]
        specs = [(0, 0, cut, l0, nl, layout), (0, cut, T - cut, 0, L, (layout + 1) % 3)]
        for lb, le in windows:
            check_store(pool, reqs, specs, lb, le, T)
            check_load(L, KV, P, v, num_pages, reqs, specs, lb, le, T)


def test_bruteforce_random_multi_request_mixes():
    """Seeded random shapes within the brute-force box, several requests and chunks."""
    rng = np.random.default_rng(2024)
    for _ in range(120):
        L = int(rng.integers(1, 4))
        KV = int(rng.integers(1, 3))
        v = int(rng.choice([16, 32, 64]))
        P = int(rng.integers(1, 5))
        n_req = int(rng.integers(1, 3))
        lens = [int(rng.integers(1, 14)) for _ in range(n_req)]
        pages = [-(-n // P) for n in lens]
        num_pages = max(8, sum(pages))
        perm = rng.permutation(num_pages).astype(np.int32)
        reqs, at = [], 0
        for n, npg in zip(lens, pages):
            reqs.append(Request(perm[at:at + npg].copy(), n))
            at += npg
        Tmax = max(lens)
        specs = []
        for r, n in enumerate(lens):
            cuts = sorted(set([0, n] + list(rng.integers(0, n + 1, size=2))))
            for a, b in zip(cuts[:-1], cuts[1:]):
                l0 = int(rng.integers(0, L))
                nl = int(rng.integers(1, L - l0 + 1))
                specs.append((r, a, b - a, l0, nl, int(rng.integers(0, 3))))
        lb = int(rng.integers(0, L + 1))
        le = int(rng.integers(lb, L + 1))
        pool = empty_pool(L, KV, num_pages, P, v)
        fill_pool_with_tags(pool, reqs, Tmax)
        check_store(pool, reqs, specs, lb, le, Tmax)
        check_load(L, KV, P, v, num_pages, reqs, specs, lb, le, Tmax)


# ----------------------------------------------------------------------------- P-b

def test_exactly_once_and_canaries_tiny_shape():
    """tiny workload shape: each tag once in the chunk, each tag once in the pool."""
    w = wl.tiny()
    s = w.shape
    L, KV, P, v = s.num_layers, s.kv_factor, s.page_size, s.token_bytes
    W = v // 4
    T = w.store_requests[0].n_tokens
    reqs = [Request(w.store_requests[0].page_table, T)]
    pool = empty_pool(L, KV, s.num_pages, P, v)
    fill_pool_with_tags(pool, reqs, T)
    arena = np.full(w.store_arena_bytes + 4096, 0xA5, np.uint8)
    chunks = [Chunk(c.request, c.token_begin, c.n_tokens, c.layer_begin, c.n_layers, c.layout,
                    arena[c.offset:]) for c in w.store_chunks]
    oracle.store(pool, reqs, chunks)
    words = arena.view(np.int32)
    vals, counts = np.unique(words, return_counts=True)
    tags = vals[vals != CANARY32]
    assert len(tags) == T * L * KV * W
    assert np.all(counts[vals != CANARY32] == 1)
    assert tags.min() == 1 and tags.max() == T * L * KV * W
    assert int(np.sum(words != CANARY32)) * 4 == 2097152  # closed form for tiny

    # Load those chunks into the disjoint page set of a fresh canary pool.
    dst = [Request(w.load_requests[0].page_table, T)]
    pool2 = empty_pool(L, KV, s.num_pages, P, v)
    oracle.load(pool2, dst, chunks)
    all_words = np.concatenate([pool2.pools[k][l].view(np.int32).reshape(-1)
                                for k in range(KV) for l in range(L)])
    vals, counts = np.unique(all_words, return_counts=True)
    assert np.all(counts[vals != CANARY32] == 1)
    assert int(np.sum(all_words != CANARY32)) == T * L * KV * W
    # Untouched: every page outside the destination table.
    untouched = np.setdiff1d(np.arange(s.num_pages), dst[0].page_table)
    for k in range(KV):
        for l in range(L):
            assert np.all(pool2.pools[k][l][untouched] == 0xA5)


def test_partial_last_page_slots_untouched():
    L, KV, P, v, num_pages = 2, 2, 4, 32, 6
    T = 10  # pages 0..2, last page holds 2 of 4 tokens
    pt = np.array([4, 0, 3], np.int32)
    pool = check_load(L, KV, P, v, num_pages, [Request(pt, T)],
                      [(0, 0, T, 0, L, LAYER_MAJOR)], 0, L, T)
    for k in range(KV):
        for l in range(L):
            assert np.all(pool.pools[k][l][3, 2:] == 0xA5)


# ----------------------------------------------------------------------------- P-c

@pytest.mark.parametrize("layout", [LAYER_MAJOR, TOKEN_MAJOR, STRIPED])
def test_round_trip_store_then_load_disjoint_pages(layout):
    rng = np.random.default_rng(99 + layout)
    L, KV, P, v, T = 3, 2, 16, 64, 200
    n = -(-T // P)
    num_pages = 3 * n
    perm = rng.permutation(num_pages).astype(np.int32)
    src, dst = Request(perm[:n], T), Request(perm[n:2 * n], T)
    pool = Pool([[rng.integers(0, 256, (num_pages, P, v), dtype=np.uint8) for _ in range(L)]
                 for _ in range(KV)], P)
    specs = [(0, a, min(48, T - a), 0, L, layout) for a in range(0, T, 48)]
    chunks = make_chunks(specs, KV, v)
    oracle.store(pool, [src], chunks)
    pool2 = empty_pool(L, KV, num_pages, P, v, fill=0)
    oracle.load(pool2, [dst], chunks)
    for k in range(KV):
        for l in range(L):
            a = pool.pools[k][l][src.page_table].reshape(-1, v)[:T]
            b = pool2.pools[k][l][dst.page_table].reshape(-1, v)[:T]
            np.testing.assert_array_equal(a, b)


def test_round_trip_load_then_store_is_identity_on_chunks():
    rng = np.random.default_rng(5)
    L, KV, P, v, T = 2, 1, 8, 48, 61
    n = -(-T // P)
    pt = rng.permutation(2 * n)[:n].astype(np.int32)
    specs = [(0, 0, 20, 0, 2, TOKEN_MAJOR), (0, 20, 41, 0, 2, LAYER_MAJOR)]
    chunks = make_chunks(specs, KV, v, pad=0)
    for c in chunks:
        c.buf[:] = rng.integers(0, 256, c.buf.shape, dtype=np.uint8)
    originals = [c.buf.copy() for c in chunks]
    pool = empty_pool(L, KV, 2 * n, P, v)
    oracle.load(pool, [Request(pt, T)], chunks)
    for c in chunks:
        c.buf[:] = 0
    oracle.store(pool, [Request(pt, T)], chunks)
    for c, o in zip(chunks, originals):
        np.testing.assert_array_equal(c.buf, o)


# ----------------------------------------------------------------------------- P-d

def _golden_rows(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].split()
        if line:
            rows[line[0]] = line[1:]
    return rows


def test_closed_form_bytes_of_workloads():
    g = _golden_rows("closed_form_bytes.txt")
    cases = {"tiny": wl.tiny(), "llama8b": wl.llama8b(), "llama70b": wl.llama70b()}
    for p in wl.MLA_PAGE_SIZES:
        for cb in wl.MLA_CHUNK_BYTES:
            cases[f"mla_sweep:{p}:{cb}"] = wl.mla_sweep(p, cb)
    for key, w in cases.items():
        row = g[key.split(":")[0]]
        T, L, KV, H, D, b, N = map(int, row)
        s = w.shape
        assert (s.num_layers, s.kv_factor, s.kv_heads, s.head_dim) == (L, KV, H, D)
        assert T * L * KV * H * D * b == N  # the golden row is self-consistent
        chunks = w.load_chunks
        assert oracle.moved_bytes(s.num_layers, s.kv_factor, s.token_bytes, chunks) == N, key
        if w.store_chunks:
            assert oracle.moved_bytes(s.num_layers, s.kv_factor, s.token_bytes,
                                      w.store_chunks) == N, key
    s = wl.llama8b().shape
    assert s.page_bytes * s.kv_factor == int(g["page_kv_llama8b"][0])
    assert wl.llama8b().load_chunks[0].nbytes(s) == 32 << 20  # 32 MiB all-layer chunk


def test_closed_form_bytes_batched_partial_hits():
    w = wl.qwen7b_batch()
    s = w.shape
    lens = [r.n_tokens for r in w.load_requests]
    total = sum(lens) * s.num_layers * 2 * 4 * 128 * 1
    moved = (oracle.moved_bytes(s.num_layers, 2, s.token_bytes, w.load_chunks) +
             oracle.moved_bytes(s.num_layers, 2, s.token_bytes, w.store_chunks))
    assert moved == total
    hits = [sum(c.n_tokens for c in w.load_chunks if c.request == r) for r in range(len(lens))]
    for L_, h in zip(lens, hits):
        assert h % 16 == 0 and h == math.floor(0.8 * L_ / 16) * 16


def test_layer_window_closed_form():
    w = wl.llama70b()
    s = w.shape
    for lb, le in [(0, 1), (10, 11), (0, 80), (79, 80), (5, 5)]:
        got = oracle.moved_bytes(s.num_layers, 2, s.token_bytes, w.load_chunks, lb, le)
        assert got == 65536 * (le - lb) * 2 * 8 * 128 * 2


# ----------------------------------------------------------------------------- P-e

@pytest.mark.parametrize("layout", [LAYER_MAJOR, TOKEN_MAJOR])
def test_numpy_fancy_indexing_cross_check(layout):
    rng = np.random.default_rng(11 + layout)
    L, KV, H, D, P, T = 4, 2, 2, 8, 16, 333  # fp16 -> v = 32 B
    v = H * D * 2
    n = -(-T // P)
    num_pages = 2 * n + 3
    pt = rng.permutation(num_pages)[:n].astype(np.int32)
    pool = Pool([[rng.integers(0, 256, (num_pages, P, v), dtype=np.uint8) for _ in range(L)]
                 for _ in range(KV)], P)
    specs = [(0, t0, min(100, T - t0), 1, 3, layout) for t0 in range(0, T, 100)]
    chunks = make_chunks(specs, KV, v, pad=0)
    oracle.store(pool, [Request(pt, T)], chunks)
    for c in chunks:
        seq = np.stack([np.stack([pool.pools[k][l][pt].reshape(-1, H, D * 2)
                                  for k in range(KV)]) for l in range(c.layer_begin,
                                                                      c.layer_begin + c.n_layers)])
        ref = seq[:, :, c.token_begin:c.token_begin + c.n_tokens]  # [l][kv][t][H][D*2]
        if layout == TOKEN_MAJOR:
            ref = np.transpose(ref, (2, 0, 1, 3, 4))
        np.testing.assert_array_equal(c.buf, ref.reshape(-1))


def test_identity_page_table_is_plain_copy():
    rng = np.random.default_rng(3)
    T, v = 96, 128
    pool = Pool([[rng.integers(0, 256, (1, T, v), dtype=np.uint8)]], T)
    chunks = make_chunks([(0, 0, T, 0, 1, LAYER_MAJOR)], 1, v, pad=0)
    oracle.store(pool, [Request(np.array([0], np.int32), T)], chunks)
    assert chunks[0].buf.tobytes() == pool.pools[0][0].tobytes()


def _strata_dst(src_unit, num_layers, cpl, total_pages, page_indices):
    """Index mapping of the GPU-assisted load kernel ("Strata Guide", section "Step 1")."""
    p = src_unit // (num_layers * cpl)
    rem = src_unit % (num_layers * cpl)
    layer = rem // cpl
    c = rem % cpl
    return layer * total_pages * cpl + page_indices[p] * cpl + c


def _load_page_first(num_layers, cpl, total_pages, page_indices, P, v):
    """Load a page-first host buffer with one chunk per page (K/V folded, all layers)."""
    n = len(page_indices)
    units = n * num_layers * cpl
    host = np.arange(1, units + 1, dtype=np.int32).repeat(4).view(np.uint8)  # 16-B units
    host = host.reshape(units, 16).copy()
    assert cpl * 16 == P * v
    # One allocation holding the layer pools back to back: [layer][page][P][v].
    flat = np.zeros((num_layers, total_pages, P, v), np.uint8)
    pool = Pool([[flat[l] for l in range(num_layers)]], P)
    chunks = []
    for p in range(n):
        seg = host[p * num_layers * cpl:(p + 1) * num_layers * cpl].reshape(-1)
        chunks.append(Chunk(0, p * P, P, 0, num_layers, LAYER_MAJOR, seg))
    oracle.load(pool, [Request(np.asarray(page_indices, np.int32), n * P)], chunks)
    return host, flat.reshape(-1, 16)


def test_strata_worked_example_golden():
    g = _golden_rows("strata_load_index.txt")
    L = int(g["num_layers"][0])
    cpl = int(g["units_per_page_layer"][0])
    total = int(g["total_gpu_pages"][0])
    pages = [int(x) for x in g["page_indices"]]
    P, v = cpl, 16  # one 16-B unit per token
    host, dst = _load_page_first(L, cpl, total, pages, P, v)
    maps = []
    for line in open(os.path.join(GOLDEN, "strata_load_index.txt")):
        f = line.split("#")[0].split()
        if f and f[0] == "map":
            maps.append((int(f[1]), int(f[2])))
    assert len(maps) == 8
    for s, d in maps:
        assert _strata_dst(s, L, cpl, total, pages) == d  # the hand computation
        np.testing.assert_array_equal(dst[d], host[s])


def test_strata_index_formula_randomised():
    rng = np.random.default_rng(17)
    for _ in range(10):
        L = int(rng.integers(1, 5))
        P = int(rng.integers(1, 5))
        v = 16 * int(rng.integers(1, 4))
        cpl = P * v // 16
        total = int(rng.integers(3, 12))
        n = int(rng.integers(1, total + 1))
        pages = rng.permutation(total)[:n]
        host, dst = _load_page_first(L, cpl, total, pages, P, v)
        touched = np.zeros(dst.shape[0], bool)
        for s in range(host.shape[0]):
            d = _strata_dst(s, L, cpl, total, pages)
            np.testing.assert_array_equal(dst[d], host[s])
            touched[d] = True
        assert np.all(dst[~touched] == 0)


def test_striped_object_offsets_closed_form():
    """One block of the MLA latent cache (16 tokens x 1152 B = 18,432 B per object) in the
    STRIPED layout: objects start at 0, 20480, 40960, ... and hold the block's bytes of
    that layer; the 2,048 padding bytes after each object are never written."""
    L, KV, P, v = 61, 1, 16, 1152
    assert oracle.chunk_bytes(L, KV, P, v, STRIPED) == L * 20480
    assert oracle.chunk_bytes(L, KV, P, v, LAYER_MAJOR) == L * 18432
    rng = np.random.default_rng(12)
    pool = Pool([[rng.integers(0, 256, (4, P, v), dtype=np.uint8) for _ in range(L)]], P)
    chunks = make_chunks([(0, 0, P, 0, L, STRIPED)], KV, v, pad=0)
    oracle.store(pool, [Request(np.array([2], np.int32), P)], chunks)
    buf = chunks[0].buf
    for l in range(L):
        assert buf[l * 20480:l * 20480 + 18432].tobytes() == pool.pools[0][l][2].tobytes()
        assert np.all(buf[l * 20480 + 18432:(l + 1) * 20480] == 0xA5)
    # A 4 KiB-multiple object needs no padding: STRIPED and LAYER_MAJOR coincide.
    assert oracle.chunk_bytes(32, 2, 16, 2048, STRIPED) == oracle.chunk_bytes(32, 2, 16, 2048,
                                                                               LAYER_MAJOR)


# ----------------------------------------------------------------------------- errors

def test_oracle_rejects_bad_inputs():
    L, KV, P, v = 2, 2, 4, 16
    pool = empty_pool(L, KV, 4, P, v)
    good = np.array([0, 1], np.int32)
    with pytest.raises(ValueError, match="page id"):
        oracle.store(pool, [Request(np.array([0, 9], np.int32), 8)],
                     make_chunks([(0, 0, 8, 0, L, 0)], KV, v))
    with pytest.raises(ValueError, match="token range"):
        oracle.store(pool, [Request(good, 8)], make_chunks([(0, 4, 8, 0, L, 0)], KV, v))
    with pytest.raises(ValueError, match="layer range"):
        oracle.store(pool, [Request(good, 8)], make_chunks([(0, 0, 8, 1, 2, 0)], KV, v))
    with pytest.raises(ValueError, match="layer range"):
        oracle.store(pool, [Request(good, 8)], make_chunks([(0, 0, 8, 0, 2, 0)], KV, v), 0, 3)


def test_chunk_parallel_timing_wrapper_matches_single_thread():
    """The CPU baseline runs the oracle over disjoint chunk ranges on host threads; the bytes
    must be those of the single-threaded loops."""
    rng = np.random.default_rng(21)
    L, KV, P, v, T = 3, 2, 8, 64, 500
    n = -(-T // P)
    pt = rng.permutation(2 * n)[:n].astype(np.int32)
    pool = Pool([[rng.integers(0, 256, (2 * n, P, v), dtype=np.uint8) for _ in range(L)]
                 for _ in range(KV)], P)
    specs = [(0, a, min(37, T - a), 0, L, (a // 37) % 3) for a in range(0, T, 37)]
    one = make_chunks(specs, KV, v)
    many = make_chunks(specs, KV, v)
    oracle.store(pool, [Request(pt, T)], one)
    oracle.store(pool, [Request(pt, T)], many, threads=5)
    for a, b in zip(one, many):
        np.testing.assert_array_equal(a.buf, b.buf)
    p1, p2 = empty_pool(L, KV, 2 * n, P, v), empty_pool(L, KV, 2 * n, P, v)
    oracle.load(p1, [Request(pt, T)], one, 1, 3)
    oracle.load(p2, [Request(pt, T)], one, 1, 3, threads=4)
    for k in range(KV):
        for l in range(L):
            np.testing.assert_array_equal(p1.pools[k][l], p2.pools[k][l])
