"""Python binding of libkvx.so (include/kvx.h): the same entry points, argument marshalling only.

Every byte of a transfer is moved by the library's CUDA kernels (or, for
``kvx_dma_baseline``, by the driver copies it issues).  There is no Python or CPU
fallback: importing this module fails if libkvx.so has not been built
(``python -m paged_kv_gather_gb300.build``).

Batches are passed as numpy structured arrays whose layout matches the C structs
(``CHUNK_DTYPE`` = ``kvx_chunk``, ``REQUEST_DTYPE`` = ``kvx_request``), so building a
batch of thousands of chunks stays cheap.  Streams are raw ``cudaStream_t`` handles
(``torch.cuda.Stream().cuda_stream``), pointers are integers.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvx.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m paged_kv_gather_gb300.build` (needs nvcc)")

_lib = ctypes.CDLL(_LIB_PATH)

# ---------------------------------------------------------------------------- constants

KVX_OK = 0
KVX_ERR_INVALID_ARG = 1
KVX_ERR_ALIGNMENT = 2
KVX_ERR_NOT_DEVICE_ACCESSIBLE = 3
KVX_ERR_PAGE_OUT_OF_RANGE = 4
KVX_ERR_OVERLAP = 5
KVX_ERR_CUDA = 6
KVX_ERR_DEVICE_STATUS = 7
KVX_ERR_CAPACITY = 8

KVX_DEV_PAGE_OUT_OF_RANGE = 0x1
KVX_DEV_WAIT_TIMEOUT = 0x2

KVX_CHUNK_LAYER_MAJOR = 0
KVX_CHUNK_TOKEN_MAJOR = 1
KVX_CHUNK_STRIPED = 2
KVX_STRIPE_ALIGN = 4096

KVX_DIR_GATHER = 0
KVX_DIR_SCATTER = 1

KVX_MAP_WARP_SEGMENT = 0
KVX_MAP_BULK = 1
KVX_MAP_CTA = 2

KVX_HINT_DEFAULT = 0
KVX_HINT_STREAMING = 1

KVX_OP_STORE = 0
KVX_OP_LOAD = 1
KVX_OP_GATHER_HBM = 2
KVX_OP_SCATTER_HBM = 3
KVX_OP_EXCHANGE = 4
KVX_OP_ROUNDTRIP = 5

# ---------------------------------------------------------------------------- structs


class kvx_pool(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("kv_factor", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("token_bytes", ctypes.c_int64),
                ("k_pages", ctypes.POINTER(ctypes.c_void_p)),
                ("v_pages", ctypes.POINTER(ctypes.c_void_p))]


class kvx_request(ctypes.Structure):
    _fields_ = [("page_table", ctypes.c_void_p), ("page_table_host", ctypes.c_void_p),
                ("n_tokens", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class kvx_chunk(ctypes.Structure):
    _fields_ = [("request", ctypes.c_int32), ("token_begin", ctypes.c_int32),
                ("n_tokens", ctypes.c_int32), ("layer_begin", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("ptr", ctypes.c_void_p)]


class kvx_launch_cfg(ctypes.Structure):
    _fields_ = [("sm_cap", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("unroll", ctypes.c_int32),
                ("store_hint", ctypes.c_int32), ("mapping", ctypes.c_int32),
                ("stage_bytes", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("overlap", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class kvx_link_model(ctypes.Structure):
    _fields_ = [("h2d_gbs", ctypes.c_double), ("d2h_gbs", ctypes.c_double),
                ("hbm_gbs", ctypes.c_double), ("bidir_gbs", ctypes.c_double),
                ("latency_us", ctypes.c_double),
                ("launch_us", ctypes.c_double), ("num_sms", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


CHUNK_DTYPE = np.dtype([("request", "<i4"), ("token_begin", "<i4"), ("n_tokens", "<i4"),
                        ("layer_begin", "<i4"), ("n_layers", "<i4"), ("layout", "<i4"),
                        ("ptr", "<u8")])
REQUEST_DTYPE = np.dtype([("page_table", "<u8"), ("page_table_host", "<u8"),
                          ("n_tokens", "<i4"), ("reserved", "<i4")])
assert CHUNK_DTYPE.itemsize == ctypes.sizeof(kvx_chunk)
assert REQUEST_DTYPE.itemsize == ctypes.sizeof(kvx_request)

# ---------------------------------------------------------------------------- prototypes

_c = ctypes
_P = _c.POINTER
_ctx_t = _c.c_void_p
_batch = [_P(kvx_pool), _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int, _c.c_int, _c.c_int]


def _proto(name, restype, argtypes):
    fn = getattr(_lib, name)
    fn.restype = restype
    fn.argtypes = argtypes
    return fn


_proto("kvx_create", _c.c_int, [_P(_ctx_t), _c.c_int, _c.c_size_t])
_proto("kvx_destroy", None, [_ctx_t])
_proto("kvx_set_validation", _c.c_int, [_ctx_t, _c.c_int])
_proto("kvx_default_launch_cfg", _c.c_int, [_ctx_t, _c.c_int, _P(kvx_launch_cfg)])
_proto("kvx_store_chunks", _c.c_int, [_ctx_t, *_batch, _P(kvx_launch_cfg), _c.c_void_p])
_proto("kvx_load_chunks", _c.c_int, [_ctx_t, *_batch, _P(kvx_launch_cfg), _c.c_void_p])
_proto("kvx_exchange_chunks", _c.c_int,
       [_ctx_t, _P(kvx_pool), _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int,
        _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _P(kvx_launch_cfg), _c.c_void_p])
_proto("kvx_plan_create", _c.c_int, [_ctx_t, _c.c_int, *_batch, _P(kvx_launch_cfg), _c.c_void_p,
                                     _P(_c.c_void_p)])
_proto("kvx_roundtrip_chunks", _c.c_int,
       [_ctx_t, _P(kvx_pool), _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int, _c.c_int,
        _c.c_int, _P(kvx_launch_cfg), _c.c_void_p])
_proto("kvx_roundtrip_unit", _c.c_int,
       [_c.c_int32, _c.c_int64, _P(kvx_launch_cfg), _c.c_int32, _P(_c.c_int64),
        _P(_c.c_int32)])
_proto("kvx_test_roundtrip_timeout", _c.c_int,
       [_ctx_t, _P(kvx_pool), _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int,
        _c.c_uint64, _c.c_void_p])
_proto("kvx_plan_create_exchange", _c.c_int,
       [_ctx_t, _P(kvx_pool), _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int,
        _c.c_void_p, _c.c_int, _c.c_int, _c.c_int, _P(kvx_launch_cfg), _c.c_void_p,
        _P(_c.c_void_p)])
_proto("kvx_plan_create_roundtrip", _c.c_int,
       [_ctx_t, _P(kvx_pool), _c.c_void_p, _c.c_void_p, _c.c_int, _c.c_void_p, _c.c_int, _c.c_int,
        _c.c_int, _P(kvx_launch_cfg), _c.c_void_p, _P(_c.c_void_p)])
_proto("kvx_plan_launch", _c.c_int, [_c.c_void_p, _c.c_void_p])
_proto("kvx_plan_destroy", None, [_c.c_void_p])
_proto("kvx_transform_hbm", _c.c_int,
       [_ctx_t, _c.c_int, *_batch, _P(kvx_launch_cfg), _c.c_void_p])
_proto("kvx_dma_baseline", _c.c_int,
       [_ctx_t, _c.c_int, *_batch, _c.c_void_p, _P(_c.c_int64)])
_proto("kvx_get_status", _c.c_int, [_ctx_t, _c.c_void_p, _P(_c.c_uint32)])
_proto("kvx_last_error", _c.c_char_p, [_ctx_t])
_proto("kvx_last_launch", _c.c_int,
       [_ctx_t, _P(_c.c_int64), _P(_c.c_int32), _P(_c.c_int32), _P(_c.c_int64)])
_proto("kvx_validate", _c.c_int, [*_batch, _c.c_int, _c.c_int, _c.c_char_p, _c.c_size_t])
_proto("kvx_plan_count", _c.c_int, [*_batch, _P(_c.c_int64), _P(_c.c_int64)])
_proto("kvx_chunk_policy", _c.c_int,
       [_P(kvx_pool), _c.c_int, _c.c_int64, _P(_c.c_int32), _P(_c.c_int32)])
_proto("kvx_host_alloc", _c.c_int, [_P(_c.c_void_p), _c.c_size_t])
_proto("kvx_host_free", _c.c_int, [_c.c_void_p])
_proto("kvx_host_register", _c.c_int, [_c.c_void_p, _c.c_size_t])
_proto("kvx_host_unregister", _c.c_int, [_c.c_void_p])
_proto("kvx_status_string", _c.c_char_p, [_c.c_int])
_proto("kvx_version", _c.c_int, [])
_proto("kvx_default_link_model", _c.c_int, [_P(kvx_link_model)])
_proto("kvx_estimate_us", _c.c_int, [_P(kvx_link_model), _c.c_int, _c.c_int64,
                                     _P(kvx_launch_cfg), _P(_c.c_double)])
_proto("kvx_estimate_pair_us", _c.c_int, [_P(kvx_link_model), _c.c_int, _c.c_int64, _c.c_int64,
                                          _c.c_int64, _P(kvx_launch_cfg), _P(_c.c_double)])
_proto("kvx_estimate_stream_us", _c.c_int, [_c.c_double, _c.c_double, _c.c_int,
                                            _P(_c.c_double), _P(_c.c_double)])
_proto("kvx_partition_create", _c.c_int, [_c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int,
                                          _P(_c.c_void_p), _c.c_char_p, _c.c_size_t])
_proto("kvx_partition_info", _c.c_int, [_c.c_void_p, _c.c_int, _P(_c.c_void_p),
                                        _P(_c.c_int)])
_proto("kvx_partition_destroy", None, [_c.c_void_p])
_proto("kvx_load_chunks_noalloc", _c.c_int, [*_batch, _P(kvx_launch_cfg), _c.c_void_p,
                                             _c.c_void_p])

EXPORTED = ["kvx_create", "kvx_destroy", "kvx_set_validation", "kvx_default_launch_cfg",
            "kvx_store_chunks", "kvx_load_chunks", "kvx_exchange_chunks", "kvx_roundtrip_chunks",
            "kvx_plan_create", "kvx_plan_create_exchange", "kvx_plan_create_roundtrip",
            "kvx_plan_launch", "kvx_plan_destroy", "kvx_transform_hbm", "kvx_dma_baseline",
            "kvx_get_status", "kvx_last_error", "kvx_last_launch", "kvx_validate",
            "kvx_plan_count", "kvx_chunk_policy", "kvx_host_alloc", "kvx_host_free",
            "kvx_host_register", "kvx_host_unregister", "kvx_status_string", "kvx_version",
            "kvx_load_chunks_noalloc", "kvx_default_link_model", "kvx_estimate_us",
            "kvx_estimate_pair_us", "kvx_estimate_stream_us", "kvx_partition_create",
            "kvx_partition_info", "kvx_partition_destroy", "kvx_test_roundtrip_timeout",
            "kvx_roundtrip_unit"]

KVX_NOALLOC_SCRATCH_BYTES = 1 << 20


def library_path() -> str:
    """Path of the loaded libkvx.so."""
    return _LIB_PATH


def raw():
    """The loaded ctypes library (for tests that probe symbols)."""
    return _lib


class KvxError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{kvx_status_string(status)} ({status}): {message}")
        self.status = status
        self.message = message


def kvx_status_string(status: int) -> str:
    """Name of a kvx_status code."""
    return _lib.kvx_status_string(status).decode()


def kvx_version() -> int:
    """KVX_VERSION of the loaded library."""
    return _lib.kvx_version()


# ---------------------------------------------------------------------------- marshalling

class Pool:
    """A kvx_pool plus the host pointer arrays it references (kept alive with it)."""

    def __init__(self, num_layers: int, kv_factor: int, page_size: int, num_pages: int,
                 token_bytes: int, k_ptrs: Sequence[int], v_ptrs: Optional[Sequence[int]]):
        self._k = (ctypes.c_void_p * num_layers)(*k_ptrs)
        self._v = (ctypes.c_void_p * num_layers)(*(v_ptrs or [0] * num_layers))
        self.c = kvx_pool(num_layers, kv_factor, page_size, num_pages, token_bytes,
                          ctypes.cast(self._k, ctypes.POINTER(ctypes.c_void_p)),
                          ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p))
                          if kv_factor == 2 else None)

    @classmethod
    def from_tensor(cls, pools, page_size: int) -> "Pool":
        """pools: a contiguous uint8 CUDA tensor
        [kv_factor, num_layers, num_pages, page_size, token_bytes]."""
        if pools.dim() != 5 or pools.element_size() != 1 or not pools.is_contiguous():
            raise ValueError("pools must be a contiguous byte tensor "
                             "[kv_factor, num_layers, num_pages, page_size, token_bytes]")
        if not pools.is_cuda:
            raise ValueError("pools must be in device memory")
        kv, L, n, P, v = pools.shape
        if P != page_size or kv not in (1, 2):
            raise ValueError(f"pools shape {tuple(pools.shape)} does not match page_size "
                             f"{page_size} and kv_factor 1 or 2")
        base = pools.data_ptr()
        layer = n * P * v
        k = [base + (0 * L + l) * layer for l in range(L)]
        vv = [base + (1 * L + l) * layer for l in range(L)] if kv == 2 else None
        return cls(L, kv, P, n, v, k, vv)


def requests_array(entries) -> np.ndarray:
    """entries: iterable of (page_table_ptr, page_table_host (np.int32 array or None), n_tokens)."""
    entries = list(entries)
    a = np.zeros(len(entries), REQUEST_DTYPE)
    keep = []
    for i, (ptr, host, n) in enumerate(entries):
        a[i]["page_table"] = ptr
        if host is not None:
            h = np.ascontiguousarray(host, dtype=np.int32)
            keep.append(h)
            a[i]["page_table_host"] = h.ctypes.data
        a[i]["n_tokens"] = n
    return _Held(a, keep)


class _Held(np.ndarray):
    """A structured array that keeps the host buffers its pointers refer to alive."""

    def __new__(cls, arr, keep):
        obj = np.asarray(arr).view(cls)
        obj._keep = keep
        return obj

    def __array_finalize__(self, obj):
        self._keep = getattr(obj, "_keep", None)


def chunks_array(specs, base_ptr: int) -> np.ndarray:
    """specs: objects with request/token_begin/n_tokens/layer_begin/n_layers/layout/offset."""
    a = np.zeros(len(specs), CHUNK_DTYPE)
    if len(specs):
        a["request"] = [c.request for c in specs]
        a["token_begin"] = [c.token_begin for c in specs]
        a["n_tokens"] = [c.n_tokens for c in specs]
        a["layer_begin"] = [c.layer_begin for c in specs]
        a["n_layers"] = [c.n_layers for c in specs]
        a["layout"] = [c.layout for c in specs]
        a["ptr"] = np.asarray([c.offset for c in specs], np.uint64) + np.uint64(base_ptr)
    return a


def _arr_ptr(a: Optional[np.ndarray], dtype) -> Tuple[int, int]:
    if a is None or len(a) == 0:
        return None, 0
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"]:
        raise ValueError("batch arrays must be contiguous arrays of the C struct's dtype "
                         "(use requests_array / chunks_array)")
    return a.ctypes.data, len(a)


def _batch_args(pool: Pool, reqs, chunks, layer_begin, layer_end):
    rp, nr = _arr_ptr(reqs, REQUEST_DTYPE)
    cp, nc = _arr_ptr(chunks, CHUNK_DTYPE)
    if layer_end is None:
        layer_end = pool.c.num_layers
    return [ctypes.byref(pool.c), rp, nr, cp, nc, layer_begin, layer_end]


def _cfg_ptr(cfg: Optional[kvx_launch_cfg]):
    return ctypes.byref(cfg) if cfg is not None else None


def _check(ctx, status: int):
    if status != KVX_OK:
        raise KvxError(status, kvx_last_error(ctx) if ctx else "")


# ---------------------------------------------------------------------------- entry points

def kvx_create(device: int = 0, max_descriptor_bytes: int = 0):
    """A context on `device` (descriptor ring, status word, copy stream); raises on failure."""
    ctx = ctypes.c_void_p()
    st = _lib.kvx_create(ctypes.byref(ctx), device, max_descriptor_bytes)
    if st != KVX_OK:
        raise KvxError(st, "kvx_create failed")
    return ctx


def kvx_destroy(ctx) -> None:
    """Wait for the context's launches, then free it."""
    _lib.kvx_destroy(ctx)


def kvx_set_validation(ctx, level: int) -> None:
    """Host validation level: 0, 1 (default) or 2 (page ids, overlap, pointer attributes)."""
    _check(ctx, _lib.kvx_set_validation(ctx, level))


def kvx_default_launch_cfg(ctx, op: int) -> kvx_launch_cfg:
    """The default launch configuration of an operation (KVX_OP_*)."""
    cfg = kvx_launch_cfg()
    _check(ctx, _lib.kvx_default_launch_cfg(ctx, op, ctypes.byref(cfg)))
    return cfg


def kvx_store_chunks(ctx, pool: Pool, reqs, chunks, layer_begin: int = 0,
                     layer_end: Optional[int] = None, cfg: Optional[kvx_launch_cfg] = None,
                     stream: int = 0) -> None:
    """Gather the requests' pages into the chunks (mapped pinned host memory); async on `stream`."""
    _check(ctx, _lib.kvx_store_chunks(ctx, *_batch_args(pool, reqs, chunks, layer_begin,
                                                        layer_end), _cfg_ptr(cfg), stream))


def kvx_load_chunks(ctx, pool: Pool, reqs, chunks, layer_begin: int = 0,
                    layer_end: Optional[int] = None, cfg: Optional[kvx_launch_cfg] = None,
                    stream: int = 0) -> None:
    """Scatter the chunks (mapped pinned host memory) into the requests' pages; async."""
    _check(ctx, _lib.kvx_load_chunks(ctx, *_batch_args(pool, reqs, chunks, layer_begin,
                                                       layer_end), _cfg_ptr(cfg), stream))


def kvx_exchange_chunks(ctx, pool: Pool, store_reqs, store_chunks, load_reqs, load_chunks,
                        layer_begin: int = 0, layer_end: Optional[int] = None,
                        cfg: Optional[kvx_launch_cfg] = None, stream: int = 0) -> None:
    """One launch that stores store_chunks and loads load_chunks (either may be empty)."""
    srp, nsr = _arr_ptr(store_reqs, REQUEST_DTYPE)
    scp, nsc = _arr_ptr(store_chunks, CHUNK_DTYPE)
    lrp, nlr = _arr_ptr(load_reqs, REQUEST_DTYPE)
    lcp, nlc = _arr_ptr(load_chunks, CHUNK_DTYPE)
    if layer_end is None:
        layer_end = pool.c.num_layers
    _check(ctx, _lib.kvx_exchange_chunks(ctx, ctypes.byref(pool.c), srp, nsr, scp, nsc, lrp, nlr,
                                         lcp, nlc, layer_begin, layer_end, _cfg_ptr(cfg),
                                         stream))


def kvx_roundtrip_chunks(ctx, pool: Pool, src_reqs, dst_reqs, chunks, layer_begin: int = 0,
                         layer_end: Optional[int] = None, cfg: Optional[kvx_launch_cfg] = None,
                         stream: int = 0) -> None:
    """One launch: store src_reqs' pages into chunks, then load them into dst_reqs' pages."""
    srp, nsr = _arr_ptr(src_reqs, REQUEST_DTYPE)
    drp, ndr = _arr_ptr(dst_reqs, REQUEST_DTYPE)
    if nsr != ndr:
        raise ValueError("src_reqs and dst_reqs need the same number of requests")
    cp, nc = _arr_ptr(chunks, CHUNK_DTYPE)
    if layer_end is None:
        layer_end = pool.c.num_layers
    _check(ctx, _lib.kvx_roundtrip_chunks(ctx, ctypes.byref(pool.c), srp, drp, nsr, cp, nc,
                                          layer_begin, layer_end, _cfg_ptr(cfg), stream))


def kvx_plan_create(ctx, op: int, pool: Pool, reqs, chunks, layer_begin: int = 0,
                    layer_end: Optional[int] = None, cfg: Optional[kvx_launch_cfg] = None,
                    stream: int = 0):
    """Validate and pack a transfer once; returns the plan handle for kvx_plan_launch."""
    h = ctypes.c_void_p()
    _check(ctx, _lib.kvx_plan_create(ctx, op, *_batch_args(pool, reqs, chunks, layer_begin,
                                                           layer_end), _cfg_ptr(cfg), stream,
                                     ctypes.byref(h)))
    return h


def kvx_plan_create_exchange(ctx, pool: Pool, store_reqs, store_chunks, load_reqs, load_chunks,
                             layer_begin: int = 0, layer_end: Optional[int] = None,
                             cfg: Optional[kvx_launch_cfg] = None, stream: int = 0):
    """kvx_exchange_chunks validated and packed once; launch it with kvx_plan_launch."""
    srp, nsr = _arr_ptr(store_reqs, REQUEST_DTYPE)
    scp, nsc = _arr_ptr(store_chunks, CHUNK_DTYPE)
    lrp, nlr = _arr_ptr(load_reqs, REQUEST_DTYPE)
    lcp, nlc = _arr_ptr(load_chunks, CHUNK_DTYPE)
    if layer_end is None:
        layer_end = pool.c.num_layers
    h = ctypes.c_void_p()
    _check(ctx, _lib.kvx_plan_create_exchange(ctx, ctypes.byref(pool.c), srp, nsr, scp, nsc,
                                              lrp, nlr, lcp, nlc, layer_begin, layer_end,
                                              _cfg_ptr(cfg), stream, ctypes.byref(h)))
    return h


def kvx_plan_create_roundtrip(ctx, pool: Pool, src_reqs, dst_reqs, chunks, layer_begin: int = 0,
                              layer_end: Optional[int] = None,
                              cfg: Optional[kvx_launch_cfg] = None, stream: int = 0):
    """kvx_roundtrip_chunks validated and packed once; launch it with kvx_plan_launch."""
    srp, nsr = _arr_ptr(src_reqs, REQUEST_DTYPE)
    drp, ndr = _arr_ptr(dst_reqs, REQUEST_DTYPE)
    if nsr != ndr:
        raise ValueError("src_reqs and dst_reqs need the same number of requests")
    cp, nc = _arr_ptr(chunks, CHUNK_DTYPE)
    if layer_end is None:
        layer_end = pool.c.num_layers
    h = ctypes.c_void_p()
    _check(ctx, _lib.kvx_plan_create_roundtrip(ctx, ctypes.byref(pool.c), srp, drp, nsr, cp, nc,
                                               layer_begin, layer_end, _cfg_ptr(cfg), stream,
                                               ctypes.byref(h)))
    return h


def kvx_plan_launch(plan, stream: int = 0) -> None:
    """Launch a prepared plan on `stream` (may be captured in a CUDA graph)."""
    st = _lib.kvx_plan_launch(plan, stream)
    if st != KVX_OK:
        raise KvxError(st, "kvx_plan_launch")


def kvx_plan_destroy(plan) -> None:
    """Wait for the device, then free a plan (before its context)."""
    _lib.kvx_plan_destroy(plan)


def kvx_roundtrip_unit(page_size: int, token_bytes: int, cfg: Optional[kvx_launch_cfg] = None,
                       num_sms: int = 152) -> Tuple[int, int]:
    """(unit bytes, SM cap) kvx_roundtrip_chunks uses for these page segments (host only)."""
    unit, sms = ctypes.c_int64(), ctypes.c_int32()
    st = _lib.kvx_roundtrip_unit(page_size, token_bytes, _cfg_ptr(cfg), num_sms,
                                 ctypes.byref(unit), ctypes.byref(sms))
    if st != KVX_OK:
        raise KvxError(st, "kvx_roundtrip_unit")
    return unit.value, sms.value


def kvx_test_roundtrip_timeout(ctx, pool: Pool, src_reqs, dst_reqs, chunks, wait_ns: int,
                               stream: int = 0) -> None:
    """Test support: a round trip whose stores never run, so every load's wait runs out."""
    srp, nsr = _arr_ptr(src_reqs, REQUEST_DTYPE)
    drp, ndr = _arr_ptr(dst_reqs, REQUEST_DTYPE)
    if nsr != ndr:
        raise ValueError("src_reqs and dst_reqs need the same number of requests")
    cp, nc = _arr_ptr(chunks, CHUNK_DTYPE)
    _check(ctx, _lib.kvx_test_roundtrip_timeout(ctx, ctypes.byref(pool.c), srp, drp, nsr, cp, nc,
                                                wait_ns, stream))


def kvx_transform_hbm(ctx, direction: int, pool: Pool, reqs, chunks, layer_begin: int = 0,
                      layer_end: Optional[int] = None, cfg: Optional[kvx_launch_cfg] = None,
                      stream: int = 0) -> None:
    """The same gather (KVX_DIR_GATHER) or scatter (KVX_DIR_SCATTER) with chunks in HBM."""
    _check(ctx, _lib.kvx_transform_hbm(ctx, direction,
                                       *_batch_args(pool, reqs, chunks, layer_begin, layer_end),
                                       _cfg_ptr(cfg), stream))


def kvx_load_chunks_noalloc(pool: Pool, reqs, chunks, layer_begin: int = 0,
                            layer_end: Optional[int] = None,
                            cfg: Optional[kvx_launch_cfg] = None, stream: int = 0,
                            device_flags: int = 0) -> None:
    """kvx_load_chunks without a context: for callers that may not allocate device memory.

    Descriptors travel through one fixed device array inside the library (see
    include/kvx.h), so calls must not overlap on the GPU.  device_flags: address of a
    device word that collects KVX_DEV_* bits, or 0.
    """
    st = _lib.kvx_load_chunks_noalloc(*_batch_args(pool, reqs, chunks, layer_begin, layer_end),
                                      _cfg_ptr(cfg), stream, device_flags or None)
    if st != KVX_OK:
        raise KvxError(st, "kvx_load_chunks_noalloc")


def kvx_dma_baseline(ctx, direction: int, pool: Pool, reqs, chunks, layer_begin: int = 0,
                     layer_end: Optional[int] = None, stream: int = 0) -> int:
    """Comparison only: one cudaMemcpyAsync per segment; returns the number of copies."""
    n = ctypes.c_int64(0)
    _check(ctx, _lib.kvx_dma_baseline(ctx, direction,
                                      *_batch_args(pool, reqs, chunks, layer_begin, layer_end),
                                      stream, ctypes.byref(n)))
    return n.value


def kvx_get_status(ctx, stream: int = 0) -> int:
    """Device status flags (0 = clean); reading clears them.  Never raises on flags."""
    f = ctypes.c_uint32(0)
    st = _lib.kvx_get_status(ctx, stream, ctypes.byref(f))
    if st not in (KVX_OK, KVX_ERR_DEVICE_STATUS):
        raise KvxError(st, kvx_last_error(ctx))
    return f.value


def kvx_last_error(ctx) -> str:
    """Message of the context's last error ("" if none)."""
    return _lib.kvx_last_error(ctx).decode()


def kvx_last_launch(ctx) -> Tuple[int, int, int, int]:
    """(work items, CTAs, threads per CTA, descriptor bytes) of the last launch."""
    items, ctas, threads = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    desc = ctypes.c_int64()
    _check(ctx, _lib.kvx_last_launch(ctx, ctypes.byref(items), ctypes.byref(ctas),
                                     ctypes.byref(threads), ctypes.byref(desc)))
    return items.value, ctas.value, threads.value, desc.value


def kvx_validate(pool: Pool, reqs, chunks, layer_begin: int = 0,
                 layer_end: Optional[int] = None, op: int = KVX_OP_STORE,
                 level: int = 1) -> Tuple[int, str]:
    """Host validation alone, no launch: (status, message)."""
    buf = ctypes.create_string_buffer(512)
    st = _lib.kvx_validate(*_batch_args(pool, reqs, chunks, layer_begin, layer_end), op, level,
                           buf, len(buf))
    return st, buf.value.decode()


def kvx_plan_count(pool: Pool, reqs, chunks, layer_begin: int = 0,
                   layer_end: Optional[int] = None) -> Tuple[int, int]:
    """Work of a transfer without running it: (page segments, payload bytes one way)."""
    segs, nbytes = ctypes.c_int64(), ctypes.c_int64()
    st = _lib.kvx_plan_count(*_batch_args(pool, reqs, chunks, layer_begin, layer_end),
                             ctypes.byref(segs), ctypes.byref(nbytes))
    if st != KVX_OK:
        raise KvxError(st, "kvx_plan_count")
    return segs.value, nbytes.value


def kvx_chunk_policy(pool: Pool, layer_streaming: bool = False,
                     target_bytes: int = 0) -> Tuple[int, int]:
    """Chunk-size policy: (tokens per chunk, layers per chunk) for a pool."""
    t, l = ctypes.c_int32(), ctypes.c_int32()
    st = _lib.kvx_chunk_policy(ctypes.byref(pool.c), int(layer_streaming), target_bytes,
                               ctypes.byref(t), ctypes.byref(l))
    if st != KVX_OK:
        raise KvxError(st, "kvx_chunk_policy")
    return t.value, l.value


def kvx_default_link_model() -> kvx_link_model:
    """The measured GB300 + NVLink-C2C link model used by the estimators."""
    m = kvx_link_model()
    st = _lib.kvx_default_link_model(ctypes.byref(m))
    if st != KVX_OK:
        raise KvxError(st, "kvx_default_link_model")
    return m


def kvx_estimate_us(model: kvx_link_model, op: int, nbytes: int,
                    cfg: Optional[kvx_launch_cfg] = None) -> float:
    """Predicted microseconds of one store, load or transform call (Little's law)."""
    us = ctypes.c_double()
    st = _lib.kvx_estimate_us(ctypes.byref(model), op, nbytes, _cfg_ptr(cfg), ctypes.byref(us))
    if st != KVX_OK:
        raise KvxError(st, "kvx_estimate_us")
    return us.value


def kvx_estimate_pair_us(model: kvx_link_model, op: int, store_bytes: int, load_bytes: int,
                         unit_bytes: int = 0, cfg: Optional[kvx_launch_cfg] = None) -> float:
    """Predicted microseconds of one exchange or round trip (both link directions)."""
    us = ctypes.c_double()
    st = _lib.kvx_estimate_pair_us(ctypes.byref(model), op, store_bytes, load_bytes, unit_bytes,
                                   _cfg_ptr(cfg), ctypes.byref(us))
    if st != KVX_OK:
        raise KvxError(st, "kvx_estimate_pair_us")
    return us.value


def kvx_estimate_stream_us(io_us: float, compute_us: float, n_layers: int) -> Tuple[float, float]:
    """Layer-streaming model: (end-to-end us, I/O bubble us)."""
    e2e, bubble = ctypes.c_double(), ctypes.c_double()
    st = _lib.kvx_estimate_stream_us(io_us, compute_us, n_layers, ctypes.byref(e2e),
                                     ctypes.byref(bubble))
    if st != KVX_OK:
        raise KvxError(st, "kvx_estimate_stream_us")
    return e2e.value, bubble.value


class Partition:
    """I/O partitions plus one compute partition of the GPU's SMs (green contexts).

    io_streams[g] / io_sms_list[g] for g < io_groups (io_stream / io_sms: group 0);
    compute_stream / compute_sms for the rest.
    """

    def __init__(self, handle, streams, sms):
        self.handle = handle
        self.io_streams = streams[:-1]
        self.io_sms_list = sms[:-1]
        self.compute_stream = streams[-1]
        self.compute_sms = sms[-1]

    @property
    def io_stream(self) -> int:
        return self.io_streams[0]

    @property
    def io_sms(self) -> int:
        return self.io_sms_list[0]

    def close(self):
        if self.handle:
            kvx_partition_destroy(self.handle)
            self.handle = None


def kvx_partition_create(device: int, io_sms: int, io_priority: int = -1,
                         compute_priority: int = 0, io_groups: int = 1) -> Partition:
    """Green-context SM partitions: io_groups I/O partitions of >= io_sms SMs and the rest."""
    h = ctypes.c_void_p()
    msg = ctypes.create_string_buffer(256)
    st = _lib.kvx_partition_create(device, io_groups, io_sms, io_priority, compute_priority,
                                   ctypes.byref(h), msg, len(msg))
    if st != KVX_OK:
        raise KvxError(st, msg.value.decode())
    streams, sms = [], []
    for g in range(io_groups + 1):
        s_ = ctypes.c_void_p()
        n = ctypes.c_int()
        st = _lib.kvx_partition_info(h, g, ctypes.byref(s_), ctypes.byref(n))
        if st != KVX_OK:
            raise KvxError(st, "kvx_partition_info")
        streams.append(s_.value or 0)
        sms.append(n.value)
    return Partition(h, streams, sms)


def kvx_partition_info(p: Partition, group: int):
    """(stream handle, SMs) of partition `group` (io_groups = the compute partition)."""
    if group < len(p.io_streams):
        return p.io_streams[group], p.io_sms_list[group]
    return p.compute_stream, p.compute_sms


def kvx_partition_destroy(handle) -> None:
    """Wait for the device, then free the partitions and their streams."""
    _lib.kvx_partition_destroy(handle)


def kvx_host_alloc(nbytes: int) -> int:
    """Mapped pinned host memory of `nbytes`; returns its address."""
    p = ctypes.c_void_p()
    st = _lib.kvx_host_alloc(ctypes.byref(p), nbytes)
    if st != KVX_OK:
        raise KvxError(st, f"kvx_host_alloc({nbytes})")
    return p.value


def kvx_host_free(ptr: int) -> None:
    """Free memory from kvx_host_alloc."""
    st = _lib.kvx_host_free(ptr)
    if st != KVX_OK:
        raise KvxError(st, "kvx_host_free")


def kvx_host_register(ptr: int, nbytes: int) -> None:
    """Pin and map existing host memory for the device."""
    st = _lib.kvx_host_register(ptr, nbytes)
    if st != KVX_OK:
        raise KvxError(st, "kvx_host_register")


def kvx_host_unregister(ptr: int) -> None:
    """Undo kvx_host_register."""
    st = _lib.kvx_host_unregister(ptr)
    if st != KVX_OK:
        raise KvxError(st, "kvx_host_unregister")


class HostBuffer:
    """Mapped pinned host memory from kvx_host_alloc, viewed as a numpy uint8 array."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.ptr = kvx_host_alloc(self.nbytes)
        self.array = np.ctypeslib.as_array(
            ctypes.cast(self.ptr, ctypes.POINTER(ctypes.c_uint8)), shape=(self.nbytes,))

    def close(self) -> None:
        if self.ptr:
            self.array = None
            kvx_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
