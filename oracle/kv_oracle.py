"""Python face of the CPU oracle for paged KV gather/scatter.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this module.  It
shares no code with the CUDA library in ``paged_kv_gather_gb300`` and imports nothing
from it; inputs reach it as plain numpy arrays.

The arithmetic lives in ``kv_oracle.c`` (plain nested loops, one ``memcpy`` per token
vector).  What it follows, from "Strata Guide: Hierarchical Context Caching for Long
LLMs":
  * section "The Conflict Between PagedAttention and Transfer Efficiency" (fragmentation
    figure): a request's KV is split into fixed pages found through a page table;
  * section "Two-Dimensional Memory Layout Decoupling", items 1 and 2: layer-first
    [L, P, H, D] in GPU memory, page-first [P, L, H, D] on the host;
  * section "Step 1: High-Performance GPU-Assisted I/O CUDA Kernel": the page-table
    lookup and the layer-first destination of every transferred unit.

Parity pins for every function here live in ``tests/test_oracle_pins.py``; none is
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv_oracle.c")
_LIB = os.path.join(_HERE, "libkv_oracle.so")

LAYER_MAJOR = 0
TOKEN_MAJOR = 1
STRIPED = 2
STRIPE_ALIGN = 4096


def chunk_bytes(n_layers: int, kv_factor: int, n_tokens: int, token_bytes: int,
                layout: int) -> int:
    """Bytes a chunk occupies in its layout (STRIPED pads each (layer, kv) object)."""
    obj = n_tokens * token_bytes
    if layout == STRIPED:
        obj = -(-obj // STRIPE_ALIGN) * STRIPE_ALIGN
    return n_layers * kv_factor * obj

ERRORS = {0: "ok", -1: "bad argument", -2: "token range", -3: "page id out of range",
          -4: "layer range"}


def build(force: bool = False) -> str:
    """Compile the oracle with the host gcc into oracle/libkv_oracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Pool(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("kv_factor", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("token_bytes", ctypes.c_int64),
                ("pools", ctypes.POINTER(ctypes.c_void_p))]


class _Request(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("n_tokens", ctypes.c_int32),
                ("n_pages", ctypes.c_int32)]


class _Chunk(ctypes.Structure):
    _fields_ = [("request", ctypes.c_int32), ("token_begin", ctypes.c_int32),
                ("n_tokens", ctypes.c_int32), ("layer_begin", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("ptr", ctypes.c_void_p)]


_lib_handle = None
_lib_lock = threading.Lock()


def _lib():
    global _lib_handle
    with _lib_lock:
        if _lib_handle is None:
            lib = ctypes.CDLL(build())
            for name in ("ora_store", "ora_load"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Request), ctypes.c_int,
                               ctypes.POINTER(_Chunk), ctypes.c_int, ctypes.c_int,
                               ctypes.c_int]
            lib.ora_bytes.restype = ctypes.c_int64
            lib.ora_bytes.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Chunk),
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int]
            _lib_handle = lib
    return _lib_handle


@dataclass
class Pool:
    """K/V page pools: ``pools[kv][layer]`` is a uint8 array [num_pages, page_size, token_bytes].

    A layer may be ``None`` (not materialised) when every call on the pool uses a layer
    window that excludes it; the C loops never touch layers outside the window.
    """
    pools: List[List[np.ndarray]]
    page_size: int

    @property
    def kv_factor(self) -> int:
        return len(self.pools)

    @property
    def num_layers(self) -> int:
        return len(self.pools[0])

    @property
    def layer_shape(self):
        for per_kv in self.pools:
            for a in per_kv:
                if a is not None:
                    return a.shape
        raise ValueError("pool has no materialised layer")

    @property
    def num_pages(self) -> int:
        return self.layer_shape[0]

    @property
    def token_bytes(self) -> int:
        return self.layer_shape[2]


@dataclass
class Request:
    page_table: np.ndarray  # int32
    n_tokens: int


@dataclass
class Chunk:
    request: int
    token_begin: int
    n_tokens: int
    layer_begin: int
    n_layers: int
    layout: int
    buf: np.ndarray  # uint8, at least the chunk's bytes


@dataclass
class _Marshalled:
    pool: _Pool
    reqs: ctypes.Array
    chunks: ctypes.Array
    keep: list = field(default_factory=list)


def _check_array(a: np.ndarray, what: str) -> None:
    if a.dtype != np.uint8 or not a.flags["C_CONTIGUOUS"]:
        raise ValueError(f"{what} must be a C-contiguous uint8 array")


def _marshal(pool: Pool, reqs: Sequence[Request], chunks: Sequence[Chunk]) -> _Marshalled:
    keep = []
    ptrs = (ctypes.c_void_p * (pool.kv_factor * pool.num_layers))()
    shape = pool.layer_shape
    for k in range(pool.kv_factor):
        for l in range(pool.num_layers):
            a = pool.pools[k][l]
            if a is None:  # layer not materialised: the call's layer window must skip it
                continue
            _check_array(a, "pool")
            if a.shape != shape:
                raise ValueError("pool arrays must share one shape")
            ptrs[k * pool.num_layers + l] = a.ctypes.data
    cpool = _Pool(pool.num_layers, pool.kv_factor, pool.page_size, pool.num_pages,
                  pool.token_bytes, ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)))
    keep.append(ptrs)
    creqs = (_Request * max(1, len(reqs)))()
    for i, r in enumerate(reqs):
        pt = np.ascontiguousarray(r.page_table, dtype=np.int32)
        keep.append(pt)
        creqs[i] = _Request(pt.ctypes.data, int(r.n_tokens), int(pt.shape[0]))
    cchunks = (_Chunk * max(1, len(chunks)))()
    for i, c in enumerate(chunks):
        _check_array(c.buf, "chunk buffer")
        need = chunk_bytes(c.n_layers, pool.kv_factor, c.n_tokens, pool.token_bytes, c.layout)
        if c.buf.nbytes < need:
            raise ValueError(f"chunk {i} buffer holds {c.buf.nbytes} B, needs {need}")
        cchunks[i] = _Chunk(c.request, c.token_begin, c.n_tokens, c.layer_begin, c.n_layers,
                            c.layout, c.buf.ctypes.data)
    return _Marshalled(cpool, creqs, cchunks, keep)


def _run(name: str, pool: Pool, reqs, chunks, layer_begin: int, layer_end: Optional[int],
         threads: int = 1) -> None:
    if layer_end is None:
        layer_end = pool.num_layers
    m = _marshal(pool, reqs, chunks)
    fn = getattr(_lib(), name)
    n = len(chunks)
    if threads <= 1 or n <= 1:
        rc = fn(ctypes.byref(m.pool), m.reqs, len(reqs), m.chunks, n, layer_begin, layer_end)
        if rc != 0:
            raise ValueError(f"oracle {name}: {ERRORS.get(rc, rc)}")
        return
    # Chunk-parallel timing wrapper: disjoint chunk ranges on host threads (ctypes drops
    # the GIL during the call).  The per-chunk arithmetic is unchanged.
    bounds = [n * i // threads for i in range(threads + 1)]
    rcs = [0] * threads
    size = ctypes.sizeof(_Chunk)
    base = ctypes.addressof(m.chunks)

    def work(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi > lo:
            sub = ctypes.cast(base + lo * size, ctypes.POINTER(_Chunk))
            rcs[i] = fn(ctypes.byref(m.pool), m.reqs, len(reqs), sub, hi - lo, layer_begin,
                        layer_end)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    bad = [rc for rc in rcs if rc != 0]
    if bad:
        raise ValueError(f"oracle {name}: {ERRORS.get(bad[0], bad[0])}")


def store(pool: Pool, reqs: Sequence[Request], chunks: Sequence[Chunk], layer_begin: int = 0,
          layer_end: Optional[int] = None, threads: int = 1) -> None:
    """Gather pages into chunks (pages -> chunks)."""
    _run("ora_store", pool, reqs, chunks, layer_begin, layer_end, threads)


def load(pool: Pool, reqs: Sequence[Request], chunks: Sequence[Chunk], layer_begin: int = 0,
         layer_end: Optional[int] = None, threads: int = 1) -> None:
    """Scatter chunks into pages (chunks -> pages)."""
    _run("ora_load", pool, reqs, chunks, layer_begin, layer_end, threads)


def moved_bytes(num_layers: int, kv_factor: int, token_bytes: int, chunks,
                layer_begin: int = 0, layer_end: Optional[int] = None) -> int:
    """Bytes a store or load over these chunks moves in each direction.

    ``chunks`` may be any objects with request/token_begin/n_tokens/layer_begin/n_layers/
    layout attributes; no buffers are needed.
    """
    if layer_end is None:
        layer_end = num_layers
    cpool = _Pool(num_layers, kv_factor, 1, 1, token_bytes,
                  ctypes.cast(None, ctypes.POINTER(ctypes.c_void_p)))
    cchunks = (_Chunk * max(1, len(chunks)))()
    for i, c in enumerate(chunks):
        cchunks[i] = _Chunk(c.request, c.token_begin, c.n_tokens, c.layer_begin, c.n_layers,
                            c.layout, None)
    return int(_lib().ora_bytes(ctypes.byref(cpool), cchunks, len(chunks), layer_begin,
                                layer_end))
