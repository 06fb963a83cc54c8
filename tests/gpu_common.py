"""Helpers shared by the GPU parity tests: device pools, chunk arenas, oracle comparison.

Every helper that writes device memory with torch (on the current stream) synchronizes
before returning, because the tests launch the library's kernels on other streams.

Inputs come from the seeded generators of paged_kv_gather_gb300.workloads (or a seeded
numpy generator for the small random cases); expected values come only from the CPU
oracle run on host copies of the same inputs.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
from paged_kv_gather_gb300 import kvx
from paged_kv_gather_gb300 import workloads as wl

CANARY = 0xA5


@dataclass
class DevicePool:
    tensor: torch.Tensor      # uint8 [KV, L, num_pages, P, v] on cuda
    pool: kvx.Pool
    page_size: int

    @classmethod
    def empty(cls, L, KV, num_pages, P, v, fill=CANARY):
        t = torch.full((KV, L, num_pages, P, v), fill, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()  # the tests launch on other streams
        return cls(t, kvx.Pool.from_tensor(t, P), P)

    def fill_random(self, seed: int):
        g = torch.Generator(device="cuda")
        g.manual_seed(seed)
        flat = self.tensor.view(-1)
        step = 1 << 30
        for s in range(0, flat.numel(), step):
            e = min(flat.numel(), s + step)
            flat[s:e] = torch.randint(0, 256, (e - s,), generator=g, device="cuda",
                                      dtype=torch.int16).to(torch.uint8)
        torch.cuda.synchronize()  # the tests launch on other streams

    def host_copy(self, layers=None) -> oracle.Pool:
        """Oracle pool holding host copies of the given layers (None = all)."""
        KV, L = self.tensor.shape[:2]
        want = range(L) if layers is None else layers
        pools = [[None] * L for _ in range(KV)]
        for k in range(KV):
            for l in want:
                pools[k][l] = self.tensor[k, l].cpu().numpy()
        return oracle.Pool(pools, self.page_size)


class Requests:
    """Page tables on the device plus their host copies."""

    def __init__(self, tables: List[np.ndarray], n_tokens: List[int], host_copy=True):
        self.host = [np.ascontiguousarray(t, dtype=np.int32) for t in tables]
        self.n_tokens = list(n_tokens)
        self.dev = [torch.from_numpy(t.copy()).cuda() if len(t) else
                    torch.zeros(1, dtype=torch.int32, device="cuda") for t in self.host]
        self.array = kvx.requests_array(
            [(d.data_ptr(), h if host_copy else None, n)
             for d, h, n in zip(self.dev, self.host, self.n_tokens)])

    def oracle(self):
        return [oracle.Request(h, n) for h, n in zip(self.host, self.n_tokens)]


class Arena:
    """Chunk memory: mapped pinned host (kvx_host_alloc) or device, with a canary tail."""

    def __init__(self, nbytes: int, where: str = "host", pad: int = 4096):
        self.nbytes = nbytes
        self.where = where
        total = nbytes + pad
        if where == "host":
            self.hb = kvx.HostBuffer(total)
            self.view = self.hb.array
            self.view[:] = CANARY
            self.ptr = self.hb.ptr
        else:
            self.t = torch.full((total,), CANARY, dtype=torch.uint8, device="cuda")
            torch.cuda.synchronize()  # the tests launch on other streams
            self.ptr = self.t.data_ptr()

    def numpy(self) -> np.ndarray:
        if self.where == "host":
            return self.view
        return self.t.cpu().numpy()

    def write(self, data: np.ndarray) -> None:
        if self.where == "host":
            self.view[:len(data)] = data
        else:
            self.t[:len(data)] = torch.from_numpy(data).cuda()
            torch.cuda.synchronize()

    def close(self):
        if self.where == "host":
            self.hb.close()


def oracle_chunks(specs, arena_np: np.ndarray) -> List[oracle.Chunk]:
    return [oracle.Chunk(c.request, c.token_begin, c.n_tokens, c.layer_begin, c.n_layers,
                         c.layout, arena_np[c.offset:]) for c in specs]


def expected_store(dpool: DevicePool, reqs: Requests, specs, arena_bytes: int, lb=0, le=None,
                   pad=4096, layers=None):
    """Arena contents the oracle produces from host copies of the pool."""
    exp = np.full(arena_bytes + pad, CANARY, np.uint8)
    host_pool = dpool.host_copy(layers)
    oracle.store(host_pool, reqs.oracle(), oracle_chunks(specs, exp), lb, le)
    return exp


def expected_load(pre_pool: oracle.Pool, reqs: Requests, specs, arena_np: np.ndarray, lb=0,
                  le=None):
    oracle.load(pre_pool, reqs.oracle(), oracle_chunks(specs, arena_np), lb, le)
    return pre_pool


def assert_pool_equal(dpool: DevicePool, exp: oracle.Pool, layers=None):
    KV, L = dpool.tensor.shape[:2]
    for k in range(KV):
        for l in (range(L) if layers is None else layers):
            got = dpool.tensor[k, l].cpu().numpy()
            e = exp.pools[k][l]
            if not np.array_equal(got, e):
                bad = np.argwhere(got != e)
                raise AssertionError(f"pool kv={k} layer={l}: {len(bad)} bytes differ, first at "
                                     f"{bad[0].tolist()}")


def assert_bytes_equal(got: np.ndarray, exp: np.ndarray, what: str):
    if not np.array_equal(got, exp):
        bad = np.flatnonzero(got != exp)
        raise AssertionError(f"{what}: {len(bad)} bytes differ, first at {bad[0]} "
                             f"(got {got[bad[0]]}, want {exp[bad[0]]})")


def cfg(sm_cap=None, ctas_per_sm=0, threads=0, unroll=0, hint=0, mapping=0, stage_bytes=0,
        batch=0):
    c = kvx.kvx_launch_cfg()
    c.batch = batch
    c.sm_cap = 0 if sm_cap is None else sm_cap
    c.ctas_per_sm = ctas_per_sm
    c.threads = threads
    c.unroll = unroll
    c.store_hint = hint
    c.mapping = mapping
    c.stage_bytes = stage_bytes
    return c


def bulk(sm_cap=None, ctas_per_sm=0, stages=0, stage_bytes=0):
    """Launch configuration of the bulk-copy (shared-memory stage) mapping."""
    return cfg(sm_cap, ctas_per_sm, 0, stages, 0, kvx.KVX_MAP_BULK, stage_bytes)


def random_case(rng: np.random.Generator, max_tokens=700):
    """A small random batch: shape, page tables on disjoint pages, disjoint-token chunks."""
    L = int(rng.integers(1, 6))
    KV = int(rng.integers(1, 3))
    v = int(rng.choice([16, 32, 48, 256, 1152, 2048]))
    P = int(rng.choice([1, 2, 3, 7, 16, 32, 64]))
    n_req = int(rng.integers(1, 5))
    lens = [int(rng.integers(0 if i else 1, max_tokens)) for i in range(n_req)]
    pages = [-(-n // P) for n in lens]
    num_pages = sum(pages) * 2 + int(rng.integers(1, 9))
    perm = rng.permutation(num_pages).astype(np.int32)
    tables, at = [], 0
    for npg in pages:
        tables.append(perm[at:at + npg].copy())
        at += npg
    load_tables, at2 = [], at
    for npg in pages:
        load_tables.append(perm[at2:at2 + npg].copy())
        at2 += npg
    specs = []
    for r, n in enumerate(lens):
        cuts = sorted(set([0, n] + [int(x) for x in rng.integers(0, n + 1, size=3)]))
        for a, b in zip(cuts[:-1], cuts[1:]):
            l0 = int(rng.integers(0, L))
            nl = int(rng.integers(1, L - l0 + 1))
            specs.append(wl.ChunkSpec(r, a, b - a, l0, nl, int(rng.integers(0, 3))))
    if rng.random() < 0.2:  # an empty chunk now and then
        specs.append(wl.ChunkSpec(0, 0, 0, 0, L, 0))
    order = rng.permutation(len(specs))
    specs = [specs[i] for i in order]
    shape = wl.KVShape(L, KV, 1, v, "fp8_e4m3", P, num_pages)  # token_bytes == v
    wl.place_chunks(specs, shape)
    lb = int(rng.integers(0, L + 1)) if rng.random() < 0.4 else 0
    le = int(rng.integers(lb, L + 1)) if rng.random() < 0.4 else L
    return shape, lens, tables, load_tables, specs, lb, le


def pinned_copy(t: torch.Tensor, out: Optional[torch.Tensor] = None) -> np.ndarray:
    """Copy a device tensor into pinned host memory (fast D2H) and return a numpy view."""
    if out is None:
        out = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    out.copy_(t)
    return out.numpy()


class HostPool:
    """Oracle pool over a copy of a whole device pool tensor in mapped pinned memory
    (kvx_host_alloc, released by close(), unlike torch's caching host allocator)."""

    def __init__(self, t: torch.Tensor, page_size: int):
        self.hb = kvx.HostBuffer(t.numel())
        h = torch.from_numpy(self.hb.array).view(t.shape)
        h.copy_(t)
        arr = self.hb.array.reshape(t.shape)
        KV, L = t.shape[:2]
        self.pool = oracle.Pool([[arr[k, l] for l in range(L)] for k in range(KV)], page_size)

    def close(self):
        self.pool = None
        self.hb.close()


def host_arena_view(hb, nbytes):
    return hb.array[:nbytes]


def slab_ranges(c, shape, layer):
    """Byte ranges (offset, length) of one layer's slabs inside a layer-major chunk."""
    out = []
    if not (c.layer_begin <= layer < c.layer_begin + c.n_layers):
        return out
    slab = c.n_tokens * shape.token_bytes
    for k in range(shape.kv_factor):
        off = c.offset + ((layer - c.layer_begin) * shape.kv_factor + k) * slab
        out.append((off, slab))
    return out
