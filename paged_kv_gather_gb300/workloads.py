"""Seeded synthetic inputs for paged KV gather/scatter: shapes, page tables, chunk lists, values.

This module holds no transfer arithmetic: it only draws inputs (page placements, request
lengths, chunk boundaries, K/V values) from a seeded ``torch.Generator``.  The CUDA path,
the tests and the CPU oracle all take their inputs from here; nothing here imports either.

Workloads (shaped like the long-context serving cases of "Strata Guide: Hierarchical
Context Caching for Long LLMs" and "Tutti: Making SSD-Backed KV Cache Practical"):

* ``tiny``  -- 4 layers, 2 KV heads x 64, fp16, 16-token pages, pool of 256 pages, one
  1024-token request on a random 64-page set; one token-major chunk; load into a disjoint
  random page set.
* ``llama8b`` -- 32 layers, 8 x 128 bf16, 16-token pages, 32768 tokens on 2048 random pages
  of a 16384-page pool; 128 layer-major chunks of 256 tokens x all layers (32 MiB each).
* ``llama70b`` -- 80 layers, 8 x 128 bf16, 32-token pages, 65536 tokens on 2048 pages of a
  4096-page pool; per-layer chunks of 256 tokens (1 MiB); streamed load, layer by layer.
* ``qwen7b_batch`` -- 28 layers, 4 x 128 fp8 e4m3, 16-token pages; 64 requests with
  log-uniform lengths in [1024, 32768]; 80 % of each prefix loaded, 20 % stored, 256-token
  all-layer chunks.
* ``mla_sweep`` -- 61 layers, one 576-element bf16 latent per token (kv_factor 1); 16384
  tokens; page size in {1, 8, 16, 32, 64} x chunk bytes in {64 KiB, 256 KiB, 1 MiB, 4 MiB}
  with per-layer chunks of floor(C / 1152) tokens.

Seeds are 1000 + the workload's index in that list (tiny = 1000, ..., mla_sweep = 1004).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np
import torch

LAYER_MAJOR = 0
TOKEN_MAJOR = 1
STRIPED = 2          # layer-major objects, each starting at a 4096-byte multiple
STRIPE_ALIGN = 4096

DTYPE_BYTES = {"fp16": 2, "bf16": 2, "fp8_e4m3": 1}
TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}

CHUNK_ALIGN = 256  # byte alignment of every chunk inside a chunk arena


@dataclass
class KVShape:
    num_layers: int
    kv_factor: int      # 2 = separate K and V pools, 1 = one latent pool (MLA)
    kv_heads: int
    head_dim: int
    dtype: str          # "fp16" | "bf16" | "fp8_e4m3"
    page_size: int      # tokens per page
    num_pages: int      # pages per pool

    @property
    def token_bytes(self) -> int:
        return self.kv_heads * self.head_dim * DTYPE_BYTES[self.dtype]

    @property
    def page_bytes(self) -> int:
        return self.page_size * self.token_bytes

    @property
    def pool_bytes(self) -> int:
        """Bytes of all K/V pools together: kv_factor x layers x pages x page bytes."""
        return self.kv_factor * self.num_layers * self.num_pages * self.page_bytes


@dataclass
class RequestSpec:
    page_table: np.ndarray   # int32, logical page -> physical page
    n_tokens: int


@dataclass
class ChunkSpec:
    request: int
    token_begin: int
    n_tokens: int
    layer_begin: int
    n_layers: int
    layout: int
    offset: int = 0          # byte offset of the chunk in its arena

    def nbytes(self, shape: KVShape) -> int:
        obj = self.n_tokens * shape.token_bytes
        if self.layout == STRIPED:
            obj = -(-obj // STRIPE_ALIGN) * STRIPE_ALIGN
        return self.n_layers * shape.kv_factor * obj


@dataclass
class Workload:
    name: str
    seed: int
    shape: KVShape
    # Store side: resident pages that are gathered into store_chunks.
    store_requests: List[RequestSpec] = field(default_factory=list)
    store_chunks: List[ChunkSpec] = field(default_factory=list)
    # Load side: freshly allocated pages that load_chunks are scattered into.
    load_requests: List[RequestSpec] = field(default_factory=list)
    load_chunks: List[ChunkSpec] = field(default_factory=list)
    # True when the load reads back exactly what the store wrote (round trip).
    round_trip: bool = True
    notes: str = ""

    @property
    def store_arena_bytes(self) -> int:
        return _arena_bytes(self.store_chunks, self.shape)

    @property
    def load_arena_bytes(self) -> int:
        return _arena_bytes(self.load_chunks, self.shape)

    def store_bytes(self) -> int:
        return sum(c.nbytes(self.shape) for c in self.store_chunks)

    def load_bytes(self) -> int:
        return sum(c.nbytes(self.shape) for c in self.load_chunks)


def _arena_bytes(chunks: List[ChunkSpec], shape: KVShape) -> int:
    if not chunks:
        return 0
    return max(c.offset + c.nbytes(shape) for c in chunks)


def place_chunks(chunks: List[ChunkSpec], shape: KVShape, align: int = CHUNK_ALIGN) -> None:
    """Give each chunk an offset in one arena, in list order, each start aligned."""
    off = 0
    for c in chunks:
        c.offset = off
        off += -(-c.nbytes(shape) // align) * align


def split_tokens(request: int, t_begin: int, t_end: int, tokens_per_chunk: int,
                 layer_begin: int, n_layers: int, layout: int) -> List[ChunkSpec]:
    """Cut [t_begin, t_end) into consecutive chunks of tokens_per_chunk (last one partial)."""
    out = []
    t = t_begin
    while t < t_end:
        n = min(tokens_per_chunk, t_end - t)
        out.append(ChunkSpec(request, t, n, layer_begin, n_layers, layout))
        t += n
    return out


def generator(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _pages_for(n_tokens: int, page_size: int) -> int:
    return -(-n_tokens // page_size)


# ----------------------------------------------------------------------------- workloads

def tiny(seed: int = 1000) -> Workload:
    shape = KVShape(num_layers=4, kv_factor=2, kv_heads=2, head_dim=64, dtype="fp16",
                    page_size=16, num_pages=256)
    g = generator(seed)
    T = 1024
    n = _pages_for(T, shape.page_size)
    perm = torch.randperm(shape.num_pages, generator=g).numpy().astype(np.int32)
    src = RequestSpec(perm[:n].copy(), T)
    dst = RequestSpec(perm[n:2 * n].copy(), T)
    chunks = [ChunkSpec(0, 0, T, 0, shape.num_layers, TOKEN_MAJOR)]
    place_chunks(chunks, shape)
    return Workload("tiny", seed, shape, [src], chunks, [dst],
                    [ChunkSpec(**vars(c)) for c in chunks],
                    True, "one token-major chunk, load into a disjoint random page set")


def llama8b(seed: int = 1001, num_pages: int = 16384, n_tokens: int = 32768,
            tokens_per_chunk: int = 256) -> Workload:
    shape = KVShape(num_layers=32, kv_factor=2, kv_heads=8, head_dim=128, dtype="bf16",
                    page_size=16, num_pages=num_pages)
    g = generator(seed)
    n = _pages_for(n_tokens, shape.page_size)
    perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    src = RequestSpec(perm[:n].copy(), n_tokens)
    dst = RequestSpec(perm[n:2 * n].copy(), n_tokens)
    chunks = split_tokens(0, 0, n_tokens, tokens_per_chunk, 0, shape.num_layers, LAYER_MAJOR)
    place_chunks(chunks, shape)
    return Workload("llama8b", seed, shape, [src], chunks, [dst],
                    [ChunkSpec(**vars(c)) for c in chunks], True,
                    "all-layer layer-major chunks of 256 tokens (32 MiB)")


def llama70b(seed: int = 1002, num_pages: int = 4096, n_tokens: int = 65536,
             tokens_per_chunk: int = 256, num_layers: int = 80) -> Workload:
    shape = KVShape(num_layers=num_layers, kv_factor=2, kv_heads=8, head_dim=128, dtype="bf16",
                    page_size=32, num_pages=num_pages)
    g = generator(seed)
    n = _pages_for(n_tokens, shape.page_size)
    perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    dst = RequestSpec(perm[:n].copy(), n_tokens)
    chunks = []
    for l in range(shape.num_layers):
        chunks += split_tokens(0, 0, n_tokens, tokens_per_chunk, l, 1, LAYER_MAJOR)
    place_chunks(chunks, shape)
    return Workload("llama70b", seed, shape, [], [], [dst], chunks, False,
                    "load only, per-layer chunks, streamed one layer per call")


def qwen7b_batch(seed: int = 1003, n_requests: int = 64, min_len: int = 1024,
                 max_len: int = 32768, load_fraction: float = 0.8,
                 tokens_per_chunk: int = 256, pool_factor: float = 1.25) -> Workload:
    P = 16
    g = generator(seed)
    u = torch.rand(n_requests, generator=g, dtype=torch.float64).numpy()
    lens = np.exp(math.log(min_len) + u * (math.log(max_len) - math.log(min_len)))
    lens = np.maximum(min_len, (lens // P).astype(np.int64) * P)
    hits = (np.floor(load_fraction * lens / P) * P).astype(np.int64)
    pages = [_pages_for(int(L), P) for L in lens]
    total_pages = sum(pages)
    num_pages = int(math.ceil(total_pages * pool_factor))
    shape = KVShape(num_layers=28, kv_factor=2, kv_heads=4, head_dim=128, dtype="fp8_e4m3",
                    page_size=P, num_pages=num_pages)
    perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int32)
    reqs, load_chunks, store_chunks = [], [], []
    at = 0
    for r, (L, h, npg) in enumerate(zip(lens, hits, pages)):
        reqs.append(RequestSpec(perm[at:at + npg].copy(), int(L)))
        at += npg
        load_chunks += split_tokens(r, 0, int(h), tokens_per_chunk, 0, shape.num_layers,
                                    LAYER_MAJOR)
        store_chunks += split_tokens(r, int(h), int(L), tokens_per_chunk, 0, shape.num_layers,
                                     LAYER_MAJOR)
    place_chunks(load_chunks, shape)
    place_chunks(store_chunks, shape)
    return Workload("qwen7b_batch", seed, shape, reqs, store_chunks, reqs, load_chunks, False,
                    "one page table per request; pages of [0, hit) are load destinations, "
                    "pages of [hit, len) are store sources")


MLA_PAGE_SIZES = (1, 8, 16, 32, 64)
MLA_CHUNK_BYTES = (64 << 10, 256 << 10, 1 << 20, 4 << 20)


def mla_sweep(page_size: int = 16, chunk_bytes: int = 1 << 20, seed: int = 1004,
              n_tokens: int = 16384, num_layers: int = 61) -> Workload:
    shape = KVShape(num_layers=num_layers, kv_factor=1, kv_heads=1, head_dim=576, dtype="bf16",
                    page_size=page_size, num_pages=0)
    n = _pages_for(n_tokens, page_size)
    shape.num_pages = 2 * n
    g = generator(seed)
    perm = torch.randperm(shape.num_pages, generator=g).numpy().astype(np.int32)
    src = RequestSpec(perm[:n].copy(), n_tokens)
    dst = RequestSpec(perm[n:2 * n].copy(), n_tokens)
    tpc = chunk_bytes // shape.token_bytes
    chunks = []
    for l in range(num_layers):
        chunks += split_tokens(0, 0, n_tokens, tpc, l, 1, LAYER_MAJOR)
    place_chunks(chunks, shape)
    return Workload(f"mla_sweep_p{page_size}_c{chunk_bytes >> 10}k", seed, shape, [src], chunks,
                    [dst], [ChunkSpec(**vars(c)) for c in chunks], True,
                    f"per-layer chunks of {tpc} tokens ({chunk_bytes >> 10} KiB budget)")


def mla_blocks(page_size: int = 16, seed: int = 1004, n_tokens: int = 16384,
               num_layers: int = 61) -> Workload:
    """The MLA request stored as per-block objects: one STRIPED chunk per page (block) holding
    that block's 61 layer objects, each 4096-byte aligned (Tutti's 2L objects per KV block,
    with kv_factor 1)."""
    w = mla_sweep(page_size, 1 << 20, seed, n_tokens, num_layers)
    chunks = split_tokens(0, 0, n_tokens, page_size, 0, num_layers, STRIPED)
    place_chunks(chunks, w.shape, align=STRIPE_ALIGN)
    w.name = f"mla_blocks_p{page_size}"
    w.store_chunks = chunks
    w.load_chunks = [ChunkSpec(**vars(c)) for c in chunks]
    w.notes = "one 4096-aligned object per (block, layer)"
    return w


WORKLOADS = {"tiny": tiny, "llama8b": llama8b, "llama70b": llama70b,
             "qwen7b_batch": qwen7b_batch, "mla_sweep": mla_sweep, "mla_blocks": mla_blocks}


# ----------------------------------------------------------------------------- values

def fp8_e4m3_codes(n: int, g: torch.Generator, device: str = "cpu") -> torch.Tensor:
    """n bytes drawn uniformly over the 254 non-NaN OCP E4M3FN codes (all but 0x7F, 0xFF)."""
    x = torch.randint(0, 254, (n,), generator=g, device=device, dtype=torch.int16)
    x = x + (x >= 0x7F).to(torch.int16)
    return x.to(torch.uint8)


def fill_values(buf: torch.Tensor, dtype: str, g: torch.Generator) -> None:
    """Fill a uint8 tensor with KV values: N(0, 1) for fp16/bf16, uniform fp8 codes."""
    assert buf.dtype == torch.uint8 and buf.is_contiguous()
    flat = buf.view(-1)
    if dtype == "fp8_e4m3":
        flat.copy_(fp8_e4m3_codes(flat.numel(), g, device=str(flat.device)))
        return
    eb = DTYPE_BYTES[dtype]
    assert flat.numel() % eb == 0
    step = 1 << 28  # elements per draw, bounds the float32 temporary
    view = flat.view(TORCH_DTYPES[dtype])
    for s in range(0, view.numel(), step):
        e = min(view.numel(), s + step)
        view[s:e].copy_(torch.randn(e - s, generator=g, device=str(flat.device),
                                    dtype=torch.float32))


def values_generator(seed: int, device: str = "cpu", stream: int = 0) -> torch.Generator:
    """Generator for K/V values of a workload; ``stream`` separates independent draws."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 7919 + 17 + stream)
    return g


CANARY = 0xA5
