#!/usr/bin/env python3
"""Benchmark of the paged KV gather/scatter path on one GB300 (or N independent replicas).

One step = one full pass of the hot path over the Llama-3.1-8B-shaped request, in ONE
kvx_roundtrip_chunks launch:
  store  32768 tokens x 32 layers x K/V (2048 random pages of a 16384-page pool) gathered
         into 128 layer-major chunks of 256 tokens (32 MiB each) in mapped pinned host
         memory, and
  load   those chunks scattered into a disjoint set of 2048 fresh pages, each page segment
         once its own store has reached host memory,
so both directions of the host link carry data at once.  Each direction moves N = 4 GiB;
value = 2N per step / step time (GB/s).  Inputs (4 GiB each way) exceed L2 (129 MB): no
flush.  The same store and load run back to back on one stream give the per-direction
rooflines.

Also measured in the same run and printed on the same JSON line:
  host_link_peak     pinned cudaMemcpyAsync per direction and both at once (the rooflines);
  exchange_pipeline  the same step as 16 kvx_exchange_chunks launches (context);
  transform          kvx_transform_hbm gather + scatter of the same request with the chunks
                     in HBM, against the measured HBM copy peak and a same-run copy;
  dma_baseline       one cudaMemcpyAsync per (chunk, layer, kv, page) segment, both ways;
  cpu_baseline       the CPU oracle on a bounded sample of the same workload, all host cores
                     and one;
  e2e                the same step timed on the host clock through the C ABI, with the page
                     tables uploaded from pinned host memory and the status word read back;
  extra_workloads    after the timed region, on one GPU: the same store and load on 4 SMs
                     (bulk-copy and register mappings); the MLA latent at 1- and 16-token
                     pages; the batched partial hits (two streams, two I/O partitions, one
                     exchange launch); 16 layers of the 70B-shaped layer streaming under
                     GEMMs; a 1-SM background eviction under a decode GEMV loop.  Scalar
                     summaries of these also sit in the roofline object.

--workload selects the other measurement modes (layer streaming, batched partial hits, the
MLA sweeps, launch-shape sweeps, transfer sizes, the round trip beside GEMMs, background
eviction, small cases for ncu); each prints one JSON line per measured configuration.
--impl reference times the CPU oracle alone (the reference arm of this comparison).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "KV store/load GB/s vs measured host-link peak; HBM transform GB/s vs HBM peak"
GB = 1e9


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-dma-baseline", action="store_true")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the 4-SM, MLA, batched and layer-streaming legs of the default run")
    p.add_argument("--store-cfg", default="", help="sm_cap,ctas,threads,unroll,hint")
    p.add_argument("--load-cfg", default="", help="sm_cap,ctas,threads,unroll,hint")
    p.add_argument("--transform-cfg", default="", help="sm_cap,ctas,threads,unroll,hint")
    p.add_argument("--exchange-cfg", default="", help="sm_cap,ctas,threads,unroll,hint")
    p.add_argument("--roundtrip-cfg", default="", help="sm_cap,ctas,threads,unroll,hint")
    p.add_argument("--workload", default="llama8b",
                   choices=["llama8b", "llama70b", "qwen7b_batch", "mla_sweep", "sm_sweep",
                            "transform_sweep", "profile_small", "batch_sweep", "mla_blocks",
                            "roundtrip_sweep", "size_sweep", "roundtrip_under_gemm",
                            "eviction", "token_major"],
                   help="llama8b is the headline line; the others print measurement lines of "
                        "the other workloads (not the headline)")
    p.add_argument("--profile-op", default="load",
                   choices=["store", "load", "gather", "scatter", "exchange", "roundtrip",
                            "exchange_shared", "gather_cta", "load_bulk", "store_bulk",
                            "load_4sm", "store_token_major", "load_token_major",
                            "roundtrip_token_major"],
                   help="operation of --workload profile_small")
    p.add_argument("--groups", type=int, default=16,
                   help="chunk groups of the pipelined store/load round trip")
    p.add_argument("--group-list", default="8,16,32,64",
                   help="group counts of --workload roundtrip_sweep")
    p.add_argument("--fused-cfgs", default="40:8:1024,32:8:1024,48:8:1024,80:8:512",
                   help="sm_cap:unroll:threads launch shapes of the one-launch round trip in "
                        "--workload roundtrip_sweep")
    p.add_argument("--transform-shapes",
                   default="0:2:256:8:1:0:2,0:4:256:8:1:0:2,0:1:1024:8:1:0:2,0:2:512:8:1:0:2,"
                           "0:2:256:8:1:0:4,0:1:256:8:1:0:2,0:2:128:8:1:0:2,0:2:256:4:1:0:2",
                   help="mapping:ctas_per_sm:threads:unroll:hint:stage_bytes:batch launch "
                        "shapes of --workload transform_sweep")
    p.add_argument("--mla-pages", default="1,16,64",
                   help="page sizes of the MLA round trip in --workload roundtrip_sweep")
    p.add_argument("--mla-cfgs", default="0:0:0:0",
                   help="sm_cap:unroll:threads:batch launch shapes of the MLA round trip in "
                        "--workload roundtrip_sweep (0 = the default of each field)")
    p.add_argument("--chunk-tokens", type=int, default=256,
                   help="tokens per per-layer chunk of --workload llama70b (256 = 1 MiB, the "
                        "closed form; 512 = 2 MiB)")
    p.add_argument("--mapping", default="segment", choices=["segment", "bulk"],
                   help="llama70b: mapping of the per-layer loads")
    p.add_argument("--stages", type=int, default=0, help="bulk mapping: stages per ring")
    p.add_argument("--stage-bytes", type=int, default=0, help="bulk mapping: bytes per stage")
    p.add_argument("--layers", type=int, default=80, help="llama70b: layers streamed")
    p.add_argument("--priorities", default="-1,0",
                   help="llama70b: load stream priorities (-1 high, 0 normal)")
    p.add_argument("--timeline", action="store_true",
                   help="llama70b: per-layer event times of the loads and GEMMs")
    p.add_argument("--partition-sms", default="8,16",
                   help="llama70b: I/O partition sizes (green contexts) to run; empty: none")
    p.add_argument("--partition-sms-qwen", type=int, default=16,
                   help="qwen7b_batch: SMs of each of the two I/O partitions")
    p.add_argument("--sm-caps", default="1,2,4,8,16,32,0",
                   help="SM caps of the llama70b overlap sweep (0 = all SMs)")
    return p.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during a timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers

def parse_cfg(kvx, ctx, op, text):
    c = kvx.kvx_default_launch_cfg(ctx, op)
    if text:
        vals = [int(x) for x in text.split(",")]
        for name, v in zip(("sm_cap", "ctas_per_sm", "threads", "unroll", "store_hint"), vals):
            setattr(c, name, v)
    return c


class EventTimer:
    def __init__(self, stream):
        self.stream = stream
        self.pairs = []

    def start(self):
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def stop(self, e0):
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(self.stream)
        self.pairs.append((e0, e1))

    def ms(self):
        return [a.elapsed_time(b) for a, b in self.pairs]


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank-line or indentation differences."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':  # string literal, kept whole
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return "\n".join(" ".join(line.split()) for line in "".join(out).splitlines()
                     if line.strip())


def source_sha() -> str:
    """Hash of the kernel sources' code (comments and layout ignored): recorded ncu traffic
    is reported only while it still matches."""
    h = hashlib.sha256()
    for f in ("kvx_kernels.cuh", "kvx_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_gather_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, groups: int = 1):
    """DRAM bytes per launch from the committed ncu summary, if taken on this source.

    Exchange launches of the headline move 1/groups of the request each way; the recorded
    figure is for a launch moving 4 GiB each way and scales with the bytes moved."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = source_sha()
    for line in open(path):
        f = dict(x.split("=", 1) for x in line.split() if "=" in x)
        if f.get("kernel") == kernel and f.get("workload") == workload and \
                f.get("source_sha") == sha:
            return float(f["dram_bytes_per_launch"]) / groups
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback (6.8 TB/s)"


# ----------------------------------------------------------------------------- cpu baseline

class CpuSample:
    """The CPU oracle on a bounded sample of the Llama-3.1-8B-shaped workload: 32 chunks of
    256 tokens x 32 layers x K/V (1 GiB per direction).  The source pool holds exactly the
    sample's 512 pages in a seeded random order; the load writes a second pool through
    another random page order.  One pass = oracle store + oracle load."""

    def __init__(self, threads: int):
        import oracle
        from paged_kv_gather_gb300 import workloads as wl

        self.oracle = oracle
        self.threads = threads
        w = wl.llama8b(num_pages=512, n_tokens=8192)
        s = w.shape
        g = torch.Generator()
        g.manual_seed(w.seed)
        layer_bytes = s.num_pages * s.page_size * s.token_bytes
        self.src_flat = torch.randint(0, 256, (s.kv_factor * s.num_layers * layer_bytes,),
                                      dtype=torch.uint8, generator=g).numpy()
        self.dst_flat = np.zeros_like(self.src_flat)

        def as_pool(flat):
            v = flat.reshape(s.kv_factor, s.num_layers, s.num_pages, s.page_size, s.token_bytes)
            return oracle.Pool([[v[k, l] for l in range(s.num_layers)]
                                for k in range(s.kv_factor)], s.page_size)

        self.psrc, self.pdst = as_pool(self.src_flat), as_pool(self.dst_flat)
        self.arena = np.zeros(w.store_arena_bytes, np.uint8)
        self.chunks = [oracle.Chunk(c.request, c.token_begin, c.n_tokens, c.layer_begin,
                                    c.n_layers, c.layout, self.arena[c.offset:])
                       for c in w.store_chunks]
        rng = np.random.default_rng(w.seed)
        self.src = [oracle.Request(rng.permutation(512).astype(np.int32), 8192)]
        self.dst = [oracle.Request(rng.permutation(512).astype(np.int32), 8192)]
        self.bytes_per_pass = 2 * w.store_bytes()

    def one_pass(self):
        self.oracle.store(self.psrc, self.src, self.chunks, threads=self.threads)
        self.oracle.load(self.pdst, self.dst, self.chunks, threads=self.threads)

    def run(self, seconds: float, single_thread_seconds: float = 0.0):
        single = None
        if single_thread_seconds > 0:
            threads, self.threads = self.threads, 1
            single = self._timed(single_thread_seconds)
            self.threads = threads
        out = self._timed(seconds)
        if single is not None:
            out["single_thread"] = {"value": single["value"], "unit": "GB/s", "cores": 1,
                                    "sample": single["sample"]}
        return out

    def _timed(self, seconds: float):
        passes, t0 = 0, time.perf_counter()
        while True:
            self.one_pass()
            passes += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        return {"value": round(self.bytes_per_pass * passes / el / GB, 3), "unit": "GB/s",
                "cores": self.threads, "kind": "oracle",
                "sample": f"{passes} passes of oracle store+load over 32 chunks (8192 tokens x "
                          f"32 layers x K/V = 1 GiB per direction) of the Llama-3.1-8B-shaped "
                          f"workload on {self.threads} host threads, {el:.1f} s"}


def headline_config(world: int, bytes_per_direction: int) -> dict:
    """The headline workload, shared by both arms of the benchmark."""
    return {"workload": "llama8b_kv: 32 layers, 8 KV heads x 128, bf16 N(0,1), 16-token pages, "
                        "32768 tokens on 2048 random pages of a 16384-page pool, 128 "
                        "layer-major chunks of 256 tokens (32 MiB) in mapped pinned host "
                        "memory; step = store all chunks + load them into 2048 fresh pages "
                        "in one kvx_roundtrip_chunks launch (each page segment is loaded once "
                        "its store has reached host memory)",
            "bytes_per_direction": bytes_per_direction,
            "l2": "inputs larger than L2 (4 GiB per direction), no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args):
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    sample = CpuSample(threads)
    for _ in range(args.warmup):
        sample.one_pass()
    ms = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        sample.one_pass()
        ms.append((time.perf_counter() - t0) * 1e3)
    step_ms = statistics.median(ms)
    value = round(sample.bytes_per_pass / (step_ms * 1e-3) / GB, 3)
    base = {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"each step: oracle store+load over 32 of the workload's chunks (8192 "
                      f"tokens x 32 layers x K/V = 1 GiB per direction, a quarter of the "
                      f"workload) on {threads} host threads; GB/s is scaled by bytes moved"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": headline_config(1, 4 << 30),
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

class RoundTrip:
    """The headline step: store the request's 128 chunks to host memory and load them back
    into the fresh page set, pipelined in `groups` chunk groups.  Every launch is one
    kvx_exchange_chunks call on one stream that stores group g and loads group g - 1 (the
    group the previous launch stored), so both directions of the host link carry data at
    once and stream order alone keeps each load after its store.  The pipeline runs on
    across steps: a step's first launch loads the previous step's last group; flush()
    issues the last load."""

    def __init__(self, kvx, ctx, pool, reqs_src, reqs_dst, chunks, num_layers, cfg, groups,
                 dev):
        self.kvx, self.ctx, self.pool = kvx, ctx, pool
        self.rs, self.rd, self.L, self.cfg = reqs_src, reqs_dst, num_layers, cfg
        bounds = np.linspace(0, len(chunks), groups + 1).astype(int)
        self.groups = [np.ascontiguousarray(chunks[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        self.empty = np.zeros(0, dtype=chunks.dtype)
        self.stream = torch.cuda.Stream(device=dev)
        self.pending = None

    def _launch(self, store, load, timer=None):
        e = timer.start() if timer else None
        self.kvx.kvx_exchange_chunks(self.ctx, self.pool, self.rs, store, self.rd,
                                     self.empty if load is None else load, 0, self.L,
                                     self.cfg, self.stream.cuda_stream)
        if e is not None:
            timer.stop(e)

    def step(self, timer=None):
        for ch in self.groups:
            self._launch(ch, self.pending, timer)
            self.pending = ch

    def flush(self, timer=None):
        if self.pending is not None:
            self._launch(self.empty, self.pending, timer)
            self.pending = None

    def launches_per_step(self):
        return len(self.groups)


def few_sm_legs(kvx, ctx, stream, pool, rs, rd, chunks, num_layers, N, link, cap=4):
    """The same store and load of the Llama-3.1-8B-shaped request on `cap` SMs: the bulk
    mapping (two bulk-copy rings per CTA) and the register mapping, each against its
    one-way peak."""
    sh = stream.cuda_stream
    out = {"sm_cap": cap}
    for name, op, fn, rq, mapping, stages, sb in (
            ("load_bulk", kvx.KVX_OP_LOAD, kvx.kvx_load_chunks, rd, "bulk", 3, 32768),
            ("store_bulk", kvx.KVX_OP_STORE, kvx.kvx_store_chunks, rs, "bulk", 6, 16384),
            ("load_segment", kvx.KVX_OP_LOAD, kvx.kvx_load_chunks, rd, "segment", 0, 0),
            ("store_segment", kvx.KVX_OP_STORE, kvx.kvx_store_chunks, rs, "segment", 0, 0)):
        c = io_cfg(kvx, ctx, op, cap, mapping, stages, sb)
        ms = _timed(stream, lambda: fn(ctx, pool, rq, chunks, 0, num_layers, c, sh), 3, 1)
        peak = link["h2d"] if op == kvx.KVX_OP_LOAD else link["d2h"]
        gbs = N / (ms * 1e-3) / GB
        out[name] = {"gbs": round(gbs, 2), "frac": round(gbs / peak, 4), "cfg": c.as_dict()}
    assert kvx.kvx_get_status(ctx, sh) == 0
    return out


def mla_legs(kvx, wl, link, pages=(1, 16), chunk_bytes=1 << 20, reps=3):
    """The MLA latent (61 layers, 1152-byte tokens, 16384 tokens) stored and loaded with the
    library defaults at the given page sizes, per-layer chunks of chunk_bytes."""
    ctx = kvx.kvx_create(0, 64 << 20)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    out = {}
    for P in pages:
        w = wl.mla_sweep(P, chunk_bytes)
        s = w.shape
        pools = _pool_tensor(s, w.seed, wl)
        pool = kvx.Pool.from_tensor(pools, s.page_size)
        src, dst = w.store_requests[0], w.load_requests[0]
        ps = torch.from_numpy(src.page_table).cuda()
        pd = torch.from_numpy(dst.page_table).cuda()
        rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
        rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
        arena = kvx.HostBuffer(w.store_arena_bytes)
        arena.array[:] = 0
        ch = kvx.chunks_array(w.store_chunks, arena.ptr)
        N = w.store_bytes()
        st_ms = _timed(stream, lambda: kvx.kvx_store_chunks(ctx, pool, rs, ch, stream=sh), reps)
        ld_ms = _timed(stream, lambda: kvx.kvx_load_chunks(ctx, pool, rd, ch, stream=sh), reps)
        assert kvx.kvx_get_status(ctx, sh) == 0
        sg, lg = N / (st_ms * 1e-3) / GB, N / (ld_ms * 1e-3) / GB
        out[f"p{P}"] = {"page_tokens": P, "chunk_kib": chunk_bytes >> 10, "bytes": N,
                        "chunks": len(w.store_chunks),
                        "store_gbs": round(sg, 2), "store_frac": round(sg / link["d2h"], 4),
                        "load_gbs": round(lg, 2), "load_frac": round(lg / link["h2d"], 4)}
        arena.close()
        del pools
    kvx.kvx_destroy(ctx)
    return out


def llama70b_legs(kvx, wl, n_layers=16, reps=2):
    """Layer streaming of the Llama-3.1-70B-shaped prefix over its first n_layers layers
    under one bf16 8192^3 GEMM per layer: the bulk mapping on 6, 5 and 4 SMs and the register
    mapping on its default 16 SMs, each on a high-priority load stream, and the register
    mapping on a 16-SM green-context I/O partition beside the GEMMs' compute partition."""
    w, pools, pool, pt, reqs, arena, per_layer = llama70b_setup(kvx, wl, n_layers)
    ctx = kvx.kvx_create(0)
    sb = torch.cuda.Stream()
    A, B, C = gemm_operands(w.seed)
    layer_bytes = w.load_bytes() // n_layers

    def gemm():
        torch.matmul(A, B, out=C)

    with torch.cuda.stream(sb):
        gemm_ms = _timed(sb, gemm, 20, warm=5)
    out = {"layers": n_layers, "layer_bytes": layer_bytes, "gemm_alone_ms": round(gemm_ms, 4)}
    for name, mapping, cap in (("bulk_6sm", "bulk", 6), ("bulk_5sm", "bulk", 5),
                               ("bulk_4sm", "bulk", 4), ("segment_16sm", "segment", 16)):
        sa = torch.cuda.Stream(priority=-1)
        cfg = io_cfg(kvx, ctx, kvx.KVX_OP_LOAD, cap, mapping)
        out[name] = layer_streaming(kvx, ctx, pool, reqs, per_layer, n_layers, layer_bytes,
                                    cfg, sa, sb, gemm, gemm_ms, reps)
    # The loads on a 16-SM green-context I/O partition, the GEMMs on the other SMs.
    try:
        part = kvx.kvx_partition_create(0, 16, -1, 0)
    except kvx.KvxError as e:
        out["partition_16sm"] = {"unavailable": str(e)}
        part = None
    if part is not None:
        sa = torch.cuda.ExternalStream(part.io_stream)
        sc = torch.cuda.ExternalStream(part.compute_stream)
        cfg = io_cfg(kvx, ctx, kvx.KVX_OP_LOAD, 0)
        out["partition_16sm"] = {"io_sms": part.io_sms, "compute_sms": part.compute_sms,
                                 **layer_streaming(kvx, ctx, pool, reqs, per_layer, n_layers,
                                                   layer_bytes, cfg, sa, sc, gemm, gemm_ms,
                                                   reps)}
        torch.cuda.synchronize()
        part.close()
    arena.close()
    kvx.kvx_destroy(ctx)
    del pools, A, B, C
    return out


def flat_extras(seq, few, mla, qwen, l70, evict, link):
    """Scalar summaries of the extra legs, for the roofline object of the JSON line."""
    f = {"store_gbs": seq["store"]["gbs"], "store_frac": seq["store"]["frac"],
         "load_gbs": seq["load"]["gbs"], "load_frac": seq["load"]["frac"]}
    if few:
        for k in ("load_bulk", "store_bulk", "load_segment", "store_segment"):
            f[f"sm4_{k}_frac"] = few[k]["frac"]
    if mla:
        for k, v in mla.items():
            f[f"cfg5_mla_{k}_store_frac"] = v["store_frac"]
            f[f"cfg5_mla_{k}_load_frac"] = v["load_frac"]
    if qwen:
        f["cfg4_qwen7b_bound_ms"] = qwen["bound_ms"]
        f["cfg4_exchange_frac_of_bound"] = qwen["exchange_one_launch"]["frac_of_bound"]
        f["cfg4_two_streams_frac_of_bound"] = qwen["two_streams"]["frac_of_bound"]
        for cap in (16, 6):
            f[f"cfg4_two_streams_store_{cap}sm_frac_of_bound"] = \
                qwen[f"two_streams_store_{cap}sm"]["frac_of_bound"]
        tp = qwen.get("two_partitions", {})
        if "frac_of_bound" in tp:
            f["cfg4_two_partitions_frac_of_bound"] = tp["frac_of_bound"]
    if l70:
        for k in ("bulk_6sm", "bulk_5sm", "bulk_4sm", "segment_16sm", "partition_16sm"):
            r = l70[k]
            if "load_overlap_gbs" not in r:
                continue
            f[f"cfg3_{k}_load_overlap_frac"] = round(r["load_overlap_gbs"] / link["h2d"], 4)
            f[f"cfg3_{k}_gemm_slowdown_pct"] = r["gemm_slowdown_pct"]
            f[f"cfg3_{k}_e2e_vs_model"] = r["e2e_vs_model"]
    if evict:
        f["eviction_1sm_store_gbs"] = evict["store_under_decode_gbs"]
        f["eviction_1sm_decode_slowdown_pct"] = evict["decode_slowdown_pct"]
    return f


def run_ours(args):
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    from paged_kv_gather_gb300.build import build
    if rank == 0:
        build()
    barrier(world)
    from paged_kv_gather_gb300 import kvx
    from paged_kv_gather_gb300 import workloads as wl

    w = wl.llama8b()
    s = w.shape
    N = w.store_bytes()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream

    # Pools: [kv][layer][page][token][bytes], 32 GiB, bf16 N(0,1) values.
    pools = torch.empty((s.kv_factor, s.num_layers, s.num_pages, s.page_size, s.token_bytes),
                        dtype=torch.uint8, device=dev)
    wl.fill_values(pools, s.dtype, wl.values_generator(w.seed, str(dev)))
    torch.cuda.synchronize()  # filled on the current stream; the transfers use others
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src_h = w.store_requests[0].page_table
    dst_h = w.load_requests[0].page_table
    src_d = torch.from_numpy(src_h).to(dev)
    dst_d = torch.from_numpy(dst_h).to(dev)
    reqs_src = kvx.requests_array([(src_d.data_ptr(), src_h, w.store_requests[0].n_tokens)])
    reqs_dst = kvx.requests_array([(dst_d.data_ptr(), dst_h, w.load_requests[0].n_tokens)])
    host = kvx.HostBuffer(w.store_arena_bytes)
    host.array[:] = 0  # fault in every page before timing
    chunks_host = kvx.chunks_array(w.store_chunks, host.ptr)
    ctx = kvx.kvx_create(local)
    cfg_store = parse_cfg(kvx, ctx, kvx.KVX_OP_STORE, args.store_cfg)
    cfg_load = parse_cfg(kvx, ctx, kvx.KVX_OP_LOAD, args.load_cfg)
    cfg_tr = parse_cfg(kvx, ctx, kvx.KVX_OP_GATHER_HBM, args.transform_cfg)
    cfg_x = parse_cfg(kvx, ctx, kvx.KVX_OP_EXCHANGE, args.exchange_cfg)
    cfg_rt = parse_cfg(kvx, ctx, kvx.KVX_OP_ROUNDTRIP, args.roundtrip_cfg)
    rt = RoundTrip(kvx, ctx, pool, reqs_src, reqs_dst, chunks_host, s.num_layers, cfg_x,
                   args.groups, dev)

    # ---- host-link peaks: one 4 GiB pinned copy per direction, then both at once.  A peak
    # is the best of 8 timed copies (the copy engines' concurrent rate varies by run).
    link, samples = measure_link(dev, stream)

    # ---- sequential store then load on one stream (per-direction rooflines)
    def seq_step(t_store=None, t_load=None):
        e = t_store.start() if t_store else None
        kvx.kvx_store_chunks(ctx, pool, reqs_src, chunks_host, 0, s.num_layers, cfg_store, sh)
        if e is not None:
            t_store.stop(e)
        e = t_load.start() if t_load else None
        kvx.kvx_load_chunks(ctx, pool, reqs_dst, chunks_host, 0, s.num_layers, cfg_load, sh)
        if e is not None:
            t_load.stop(e)

    for _ in range(args.warmup):
        seq_step()
    ts, tl = EventTimer(stream), EventTimer(stream)
    for _ in range(max(3, args.steps // 2)):
        seq_step(ts, tl)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    store_ms = statistics.mean(ts.ms())
    load_ms = statistics.mean(tl.ms())
    store_gbs = N / (store_ms * 1e-3) / GB
    load_gbs = N / (load_ms * 1e-3) / GB

    # ---- the timed region: one kvx_roundtrip_chunks launch per step (device clock)
    def roundtrip(rs=reqs_src, rd=reqs_dst):
        kvx.kvx_roundtrip_chunks(ctx, pool, rs, rd, chunks_host, 0, s.num_layers, cfg_rt, sh)

    for _ in range(args.warmup):
        roundtrip()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        e_start = torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        step_events = [e_start]
        for _ in range(args.steps):
            roundtrip()
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            step_events.append(ev)
        e_end = step_events[-1]
        torch.cuda.synchronize()
    total_ms = max_over_ranks(e_start.elapsed_time(e_end), world)
    step_ms = [a.elapsed_time(b) for a, b in zip(step_events, step_events[1:])]
    barrier(world)
    assert kvx.kvx_get_status(ctx, sh) == 0
    items, ctas, threads, desc = kvx.kvx_last_launch(ctx)

    # ---- end to end through the C ABI on the host clock: page tables up, the round trip,
    # the status word back (which waits for the launch)
    pt_host = torch.from_numpy(np.concatenate([src_h, dst_h])).pin_memory()
    pt_dev = torch.empty_like(pt_host, device=dev)
    rs_e2e = kvx.requests_array([(pt_dev.data_ptr(), src_h, w.store_requests[0].n_tokens)])
    rd_e2e = kvx.requests_array([(pt_dev.data_ptr() + 4 * len(src_h), dst_h,
                                  w.load_requests[0].n_tokens)])
    e2e_ms = []
    for i in range(args.warmup + max(3, args.steps // 2)):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            pt_dev.copy_(pt_host, non_blocking=True)
        roundtrip(rs_e2e, rd_e2e)
        assert kvx.kvx_get_status(ctx, sh) == 0   # D2H status word + sync
        if i >= args.warmup:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = {"value": round(2 * N / (statistics.median(e2e_ms) * 1e-3) / GB, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(pt_host.numel() * 4 + desc),
           "d2h_bytes_per_step": 4,
           "payload_link_bytes_per_step": 2 * N,
           "note": "KV payload crosses the host link inside the kernel (zero-copy, mapped "
                   "pinned memory); the counted copies are the page tables, the descriptors "
                   "and the status word"}

    # ---- context: the same step as a pipeline of exchange launches (store group g + load
    # group g - 1 per launch), carried across steps
    for _ in range(2):
        rt.step()
    px = EventTimer(rt.stream)
    for _ in range(max(3, args.steps // 2)):
        e = px.start()
        rt.step()
        px.stop(e)
    rt.flush()
    torch.cuda.synchronize()
    assert kvx.kvx_get_status(ctx, rt.stream.cuda_stream) == 0
    x_ms = statistics.median(px.ms())
    exchange_pipeline = {"groups": args.groups, "launches_per_step": rt.launches_per_step(),
                         "gbs": round(2 * N / (x_ms * 1e-3) / GB, 2),
                         "kernel": "kvx_exchange_kernel", "cfg": cfg_x.as_dict()}

    # ---- HBM transform on the same request (chunks in device memory)
    dchunk = torch.empty(w.store_arena_bytes, dtype=torch.uint8, device=dev)
    chunks_dev = kvx.chunks_array(w.store_chunks, dchunk.data_ptr())
    for _ in range(args.warmup):
        kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, pool, reqs_src, chunks_dev, 0,
                              s.num_layers, cfg_tr, sh)
        kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, pool, reqs_dst, chunks_dev, 0,
                              s.num_layers, cfg_tr, sh)
    tg, tsc = EventTimer(stream), EventTimer(stream)
    for _ in range(args.steps):
        e = tg.start()
        kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, pool, reqs_src, chunks_dev, 0,
                              s.num_layers, cfg_tr, sh)
        tg.stop(e)
        e = tsc.start()
        kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_SCATTER, pool, reqs_dst, chunks_dev, 0,
                              s.num_layers, cfg_tr, sh)
        tsc.stop(e)
    stream.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    hbm_peak, hbm_src = peaks()
    # Context: a plain device-to-device copy of the same 4 GiB in this run (read + write).
    dsrc = torch.empty(N, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(2):
            dchunk.copy_(dsrc)
        tc = EventTimer(stream)
        for _ in range(max(3, args.steps // 2)):
            e = tc.start()
            dchunk.copy_(dsrc)
            tc.stop(e)
    stream.synchronize()
    copy_gbs = 2 * N / (statistics.median(tc.ms()) * 1e-3) / GB
    copy_best_gbs = 2 * N / (min(tc.ms()) * 1e-3) / GB
    del dsrc
    g_ms, s_ms = statistics.mean(tg.ms()), statistics.mean(tsc.ms())
    tr_gbs = {"gather": 2 * N / (g_ms * 1e-3) / GB, "scatter": 2 * N / (s_ms * 1e-3) / GB}
    tr_best = {"gather": 2 * N / (min(tg.ms()) * 1e-3) / GB,
               "scatter": 2 * N / (min(tsc.ms()) * 1e-3) / GB}
    dom_tr = "gather" if g_ms >= s_ms else "scatter"
    transform = {
        "gather_ms": round(g_ms, 4), "scatter_ms": round(s_ms, 4),
        "gather_gbs_2n": round(tr_gbs["gather"], 1), "scatter_gbs_2n": round(tr_gbs["scatter"], 1),
        "gather_gbs_n": round(tr_gbs["gather"] / 2, 1),  # payload N / t, one way
        "scatter_gbs_n": round(tr_gbs["scatter"] / 2, 1),
        "roofline": {"bound": "hbm", "achieved": round(tr_gbs[dom_tr], 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(tr_gbs[dom_tr] / hbm_peak, 4),
                     "traffic": recorded_traffic(f"transform_{dom_tr}", "llama8b"),
                     "kernel": f"kvx_segment_kernel ({dom_tr}, HBM chunks)",
                     "peak_source": hbm_src, "algorithmic_bytes": 2 * N,
                     "best_gbs": round(tr_best[dom_tr], 1),
                     "best_frac": round(tr_best[dom_tr] / hbm_peak, 4),
                     "best_note": "fastest of the timed launches, the statistic of the "
                                  "measured peak (best of 10 copies)",
                     "same_run_copy_gbs": round(copy_gbs, 1),
                     "same_run_copy_best_gbs": round(copy_best_gbs, 1),
                     "frac_of_same_run_copy": round(tr_gbs[dom_tr] / copy_gbs, 4),
                     "same_run_copy_note": "torch copy_ of the same 4 GiB device to device in "
                                           "this run, back to back, read + write counted "
                                           "(median and best)"},
        "cfg": cfg_tr.as_dict()}
    del dchunk

    # ---- per-page DMA baseline (both directions, one pass each after one warm-up)
    dma = None
    if not args.no_dma_baseline:
        res = {}
        for name, direction, reqs in (("store", kvx.KVX_DIR_GATHER, reqs_src),
                                      ("load", kvx.KVX_DIR_SCATTER, reqs_dst)):
            kvx.kvx_dma_baseline(ctx, direction, pool, reqs, chunks_host, 0, s.num_layers, sh)
            stream.synchronize()
            t0 = time.perf_counter()
            n = kvx.kvx_dma_baseline(ctx, direction, pool, reqs, chunks_host, 0, s.num_layers,
                                     sh)
            stream.synchronize()
            el = time.perf_counter() - t0
            res[name] = {"gbs": round(N / el / GB, 2), "copies": n, "ms": round(el * 1e3, 2)}
        dma = res

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = CpuSample(os.cpu_count() or 1).run(args.cpu_seconds,
                                                 single_thread_seconds=args.cpu_seconds / 3)

    # ---- the other workloads of the scope, compactly (1 GPU only): the same request on 4
    # SMs, the MLA latent at 1- and 16-token pages, the batched partial hits, and layer
    # streaming of the 70B-shaped prefix under GEMMs.  Outside the timed region.
    seq = {"note": "store then load on one stream, no overlap: per-direction rooflines",
           "step_gbs": round(2 * N / ((store_ms + load_ms) * 1e-3) / GB, 2),
           "store": {"ms": round(store_ms, 4), "gbs": round(store_gbs, 2),
                     "peak": link["d2h"], "frac": round(store_gbs / link["d2h"], 4),
                     "traffic": recorded_traffic("store", "llama8b")},
           "load": {"ms": round(load_ms, 4), "gbs": round(load_gbs, 2),
                    "peak": link["h2d"], "frac": round(load_gbs / link["h2d"], 4),
                    "traffic": recorded_traffic("load", "llama8b")}}
    few = mla = qwen = l70 = evict = None
    extra_clocks = None
    if world == 1 and not args.no_extras:
        few = few_sm_legs(kvx, ctx, stream, pool, reqs_src, reqs_dst, chunks_host,
                          s.num_layers, N, link)
        evict = eviction_leg(kvx, ctx, pool, reqs_src, chunks_host, s.num_layers, N, w.seed,
                             caps=(1,))[0]
        del pools
        torch.cuda.empty_cache()
        with ClockSampler(local) as ec:
            mla = mla_legs(kvx, wl, link)
            torch.cuda.empty_cache()
            qwen = qwen7b_measure(args, kvx, wl, link, reps=3)
            torch.cuda.empty_cache()
            l70 = llama70b_legs(kvx, wl)
            torch.cuda.synchronize()
        extra_clocks = ec.summary()

    value = 2 * N * args.steps * world / (total_ms * 1e-3) / GB
    step_gbs = 2 * N / (total_ms / args.steps * 1e-3) / GB
    launch_gbs = step_gbs  # one launch per step
    # The I/O-time model with this run's measured link peaks (kvx_estimate_pair_us).
    model = kvx.kvx_default_link_model()
    model.h2d_gbs, model.d2h_gbs, model.bidir_gbs = link["h2d"], link["d2h"], link["bidir"]
    model_ms = kvx.kvx_estimate_pair_us(model, kvx.KVX_OP_ROUNDTRIP, N, N,
                                        s.page_size * s.token_bytes, cfg_rt) * 1e-3
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "step_ms": {"median": round(statistics.median(step_ms), 4),
                    "min": round(min(step_ms), 4), "max": round(max(step_ms), 4),
                    "note": "this rank's steps, device clock"},
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": headline_config(world, N),
        "roofline": {"bound": "host_link", "achieved": round(launch_gbs, 2),
                     "peak": link["bidir"], "unit": "GB/s",
                     "frac": round(launch_gbs / link["bidir"], 4),
                     "step_gbs": round(step_gbs, 2),
                     "achieved_note": "bytes per round-trip launch (both directions) / "
                                      "mean launch duration on the launching stream (one "
                                      "launch per step; the events also hold its descriptor "
                                      "copy and completion-word reset)",
                     "traffic": recorded_traffic("roundtrip", "llama8b"),
                     "model_ms": round(model_ms, 4),
                     "model_note": "kvx_estimate_pair_us with this run's link peaks: fill and "
                                   "drain of one 32 KiB unit per warp at the one-way rates, "
                                   "the rest at the bidirectional peak, plus 10 us per call",
                     "kernel": "kvx_roundtrip_kernel (store + load of every segment in one "
                               "launch)",
                     "peak_source": "measured in this run: best of 8 pairs of 4 GiB pinned "
                                    "cudaMemcpyAsync, H2D and D2H at once (both link "
                                    "directions)",
                     "algorithmic_bytes": 2 * N,
                     "per_launch": {"ms": round(total_ms / args.steps, 4),
                                    "gbs": round(launch_gbs, 2), "bytes_per_launch": 2 * N,
                                    "items_per_launch": items, "ctas": ctas,
                                    "threads": threads},
                     **flat_extras(seq, few, mla, qwen, l70, evict, link),
                     **({"extras_sm_mhz": extra_clocks.get("sm_mhz"),
                         "extras_sm_max_mhz": extra_clocks.get("sm_max_mhz"),
                         "extras_clock_reasons": ",".join(extra_clocks.get("reasons") or [])
                         or "none"} if extra_clocks else {}),
                     "flat_note": "store_/load_: the request stored, then loaded, alone on "
                                  "one stream (library defaults) against the one-way peaks; "
                                  "sm4_: the same on 4 SMs; cfg3_/cfg4_/cfg5_: the 70B "
                                  "layer streaming, batched partial hits and MLA legs of "
                                  "extra_workloads; eviction_: a 1-SM store under a decode "
                                  "GEMV loop"},
        "extra_workloads": {"few_sms": few, "mla_latent": mla, "qwen7b_batched": qwen,
                            "llama70b_layer_streaming": l70, "background_eviction": evict,
                            "clocks": extra_clocks},
        "exchange_pipeline": exchange_pipeline,
        "sequential": seq,
        "cfg": {"roundtrip": cfg_rt.as_dict(), "store": cfg_store.as_dict(),
                "load": cfg_load.as_dict()},
        "host_link_peak": {"h2d_gbs": link["h2d"], "d2h_gbs": link["d2h"],
                           "bidirectional_gbs": link["bidir"], "samples_gbs": samples,
                           "method": "best of 8 timed 4 GiB pinned cudaMemcpyAsync (per "
                                     "direction, and H2D + D2H on two streams at once)",
                           "nominal_gbs_per_direction": 450.0,
                           "nominal_note": "NVLink-C2C 900 GB/s bidirectional"},
        "transform": transform,
        "dma_baseline": dma,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    host.close()
    kvx.kvx_destroy(ctx)


# ----------------------------------------------------------------------------- other workloads

def _timed(stream, fn, reps, warm=2):
    for _ in range(warm):
        fn()
    t = EventTimer(stream)
    for _ in range(reps):
        e = t.start()
        fn()
        t.stop(e)
    stream.synchronize()
    return statistics.median(t.ms())


def _fill_host(arr, nbytes, shape, seed, stream_id, wl):
    g = wl.values_generator(seed, "cuda", stream=stream_id)
    step = 1 << 30
    for s0 in range(0, nbytes, step):
        e = min(nbytes, s0 + step)
        tmp = torch.empty(e - s0, dtype=torch.uint8, device="cuda")
        wl.fill_values(tmp, shape.dtype, g)
        torch.from_numpy(arr[s0:e]).copy_(tmp)


def _pool_tensor(shape, seed, wl):
    t = torch.empty((shape.kv_factor, shape.num_layers, shape.num_pages, shape.page_size,
                     shape.token_bytes), dtype=torch.uint8, device="cuda")
    wl.fill_values(t, shape.dtype, wl.values_generator(seed, "cuda"))
    torch.cuda.synchronize()  # filled on the current stream; the transfers use others
    return t


def _emit(d):
    print(json.dumps(d), flush=True)


def io_cfg(kvx, ctx, op, cap, mapping="segment", stages=0, stage_bytes=0):
    """Launch configuration of a store or load: the default register mapping, or the bulk
    mapping (two bulk-copy rings per CTA) with `stages` stages of `stage_bytes` each."""
    c = kvx.kvx_default_launch_cfg(ctx, op)
    c.sm_cap = cap
    if mapping == "bulk":
        c.mapping, c.threads = kvx.KVX_MAP_BULK, 0
        c.unroll, c.stage_bytes = stages, stage_bytes
    return c


def layer_streaming(kvx, ctx, pool, reqs, per_layer, n_layers, layer_bytes, cfg, io_stream,
                    gemm_stream, gemm, gemm_alone_ms, reps=2, timeline=False):
    """Per-layer loads on io_stream; GEMM(l) on gemm_stream once load(l) is done (an event).
    Returns load GB/s alone and overlapped, the GEMM's mean time beside the loads against
    gemm_alone_ms, end to end, and the I/O-time model's prediction for the same launches.
    timeline: also the last repetition's per-layer event times (ms from its start) of each
    load (its stream reaching the call, the load's end) and each GEMM (start, end)."""
    io_h = io_stream.cuda_stream

    def load_all():
        for l in range(n_layers):
            kvx.kvx_load_chunks(ctx, pool, reqs, per_layer[l], l, l + 1, cfg, io_h)

    total = layer_bytes * n_layers
    alone_ms = _timed(io_stream, load_all, 3, warm=1)
    spans, e2es, gms = [], [], []
    for rep in range(reps):
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        start.record(io_stream)
        gemm_stream.wait_event(start)
        gt = EventTimer(gemm_stream)
        lt = EventTimer(io_stream)
        for l in range(n_layers):
            e_l = lt.start()
            kvx.kvx_load_chunks(ctx, pool, reqs, per_layer[l], l, l + 1, cfg, io_h)
            lt.stop(e_l)
            ev = torch.cuda.Event()
            ev.record(io_stream)
            gemm_stream.wait_event(ev)
            with torch.cuda.stream(gemm_stream):
                e = gt.start()
                gemm()
                gt.stop(e)
        end_a = torch.cuda.Event(enable_timing=True)
        end_a.record(io_stream)
        end_b = torch.cuda.Event(enable_timing=True)
        end_b.record(gemm_stream)
        torch.cuda.synchronize()
        spans.append(start.elapsed_time(end_a))
        e2es.append(start.elapsed_time(end_b))
        gms.append(statistics.mean(gt.ms()))
        if timeline:
            rows = [{"layer": l,
                     "load_start_ms": round(start.elapsed_time(a), 4),
                     "load_end_ms": round(start.elapsed_time(b), 4),
                     "gemm_start_ms": round(start.elapsed_time(c), 4),
                     "gemm_end_ms": round(start.elapsed_time(d), 4)}
                    for l, ((a, b), (c, d)) in enumerate(zip(lt.pairs, gt.pairs))]
    assert kvx.kvx_get_status(ctx, io_h) == 0
    g_ms = statistics.median(gms)
    model = kvx.kvx_default_link_model()
    pred_io = kvx.kvx_estimate_us(model, kvx.KVX_OP_LOAD, layer_bytes, cfg)
    pred_e2e, pred_bubble = kvx.kvx_estimate_stream_us(pred_io, gemm_alone_ms * 1e3, n_layers)
    # The same model fed with this run's own per-layer load time (alone) and GEMM time.
    meas_e2e, _ = kvx.kvx_estimate_stream_us(alone_ms * 1e3 / n_layers, gemm_alone_ms * 1e3,
                                             n_layers)
    e2e = statistics.median(e2es)
    out = {}
    if timeline:
        med = lambda xs: round(statistics.median(xs), 4)  # noqa: E731
        out["timeline"] = {
            "layers": rows,
            "load_ms_median": med([r["load_end_ms"] - r["load_start_ms"] for r in rows]),
            "gemm_ms_median": med([r["gemm_end_ms"] - r["gemm_start_ms"] for r in rows]),
            # how long after its load ended each GEMM started, and the GEMM's share of the
            # next layer's load window spent beside it
            "gemm_start_after_load_end_ms_median":
                med([r["gemm_start_ms"] - r["load_end_ms"] for r in rows]),
            "gemm_overlap_of_next_load_median":
                med([max(0.0, min(rows[i]["gemm_end_ms"], rows[i + 1]["load_end_ms"]) -
                         max(rows[i]["gemm_start_ms"], rows[i + 1]["load_start_ms"])) /
                     (rows[i + 1]["load_end_ms"] - rows[i + 1]["load_start_ms"])
                     for i in range(len(rows) - 1)] or [0.0]),
            "load_gap_between_layers_ms_median":
                med([rows[i + 1]["load_start_ms"] - rows[i]["load_end_ms"]
                     for i in range(len(rows) - 1)] or [0.0]),
            "compute_idle_ms": round(rows[0]["gemm_start_ms"] + sum(
                max(0.0, rows[i + 1]["gemm_start_ms"] - rows[i]["gemm_end_ms"])
                for i in range(len(rows) - 1)), 4)}
    return {**out, "layers": n_layers, "layer_bytes": layer_bytes,
            "load_cfg": cfg.as_dict(),
            "load_alone_ms": round(alone_ms, 3),
            "load_alone_gbs": round(total / (alone_ms * 1e-3) / GB, 2),
            "load_overlap_span_ms": round(statistics.median(spans), 3),
            "load_overlap_gbs": round(total / (statistics.median(spans) * 1e-3) / GB, 2),
            "gemm_alone_ms": round(gemm_alone_ms, 4), "gemm_overlap_ms": round(g_ms, 4),
            "gemm_slowdown_pct": round(100 * (g_ms / gemm_alone_ms - 1), 2),
            "e2e_ms": round(e2e, 3),
            "serial_ms": round(alone_ms + n_layers * gemm_alone_ms, 3),
            "model_e2e_ms": round(pred_e2e * 1e-3, 3),
            "model_bubble_ms": round(pred_bubble * 1e-3, 3),
            "e2e_vs_model": round(e2e / (pred_e2e * 1e-3), 4),
            "model_from_measured_e2e_ms": round(meas_e2e * 1e-3, 3),
            "e2e_vs_model_from_measured": round(e2e / (meas_e2e * 1e-3), 4)}


def llama70b_setup(kvx, wl, n_layers, chunk_tokens=256):
    """Pool, page table, host arena and per-layer chunk arrays of the Llama-3.1-70B-shaped
    prefix, for its first n_layers layers (80 = the whole model)."""
    w = wl.llama70b(tokens_per_chunk=chunk_tokens, num_layers=n_layers)
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    r = w.load_requests[0]
    pt = torch.from_numpy(r.page_table).cuda()
    reqs = kvx.requests_array([(pt.data_ptr(), r.page_table, r.n_tokens)])
    arena = kvx.HostBuffer(w.load_arena_bytes)
    _fill_host(arena.array, w.load_arena_bytes, s, w.seed, 1, wl)
    per_layer = [kvx.chunks_array([c for c in w.load_chunks if c.layer_begin == l], arena.ptr)
                 for l in range(s.num_layers)]
    return w, pools, pool, pt, reqs, arena, per_layer


def gemm_operands(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    A = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16, generator=g)
    B = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16, generator=g)
    C = torch.empty(8192, 8192, device="cuda", dtype=torch.bfloat16)
    return A, B, C


def run_llama70b(args, kvx, wl):
    """Layer-streamed load of a 65536-token prefix (80 layers, 256 MiB per layer) while a
    bf16 8192^3 GEMM per layer runs on a second stream: SM caps and stream priorities for the
    chosen mapping (--mapping segment|bulk), then hard SM partitions (green contexts)."""
    w, pools, pool, pt, reqs, arena, per_layer = llama70b_setup(kvx, wl, args.layers,
                                                               args.chunk_tokens)
    s = w.shape
    ctx = kvx.kvx_create(0)
    sb = torch.cuda.Stream()
    A, B, C = gemm_operands(w.seed)
    layer_bytes = w.load_bytes() // s.num_layers

    def gemm():
        torch.matmul(A, B, out=C)

    with torch.cuda.stream(sb):
        gemm_ms = _timed(sb, gemm, 20, warm=5)
    caps = [int(x) for x in args.sm_caps.split(",")]
    prios = [int(x) for x in args.priorities.split(",")]
    for cap, prio in [(c, p) for p in prios for c in caps]:
        # Loads on a high-priority stream (-1) get SMs as soon as GEMM CTAs retire.
        sa = torch.cuda.Stream(priority=prio)
        cfg = io_cfg(kvx, ctx, kvx.KVX_OP_LOAD, cap, args.mapping, args.stages,
                     args.stage_bytes)
        r = layer_streaming(kvx, ctx, pool, reqs, per_layer, s.num_layers, layer_bytes, cfg,
                            sa, sb, gemm, gemm_ms, timeline=args.timeline)
        _emit({"workload": "llama70b_layer_streaming", "chunk_tokens": args.chunk_tokens,
               "mapping": args.mapping, "sm_cap": cap,
               "load_stream_priority": "high" if prio < 0 else "normal", **r})
    # Hard SM partitions (green contexts): the loads on an I/O partition, the GEMM on the
    # rest of the GPU.
    for io_sms in [int(x) for x in args.partition_sms.split(",") if x]:
        try:
            part = kvx.kvx_partition_create(0, io_sms, -1, 0)
        except kvx.KvxError as e:
            _emit({"workload": "llama70b_layer_streaming", "partition": "unavailable",
                   "reason": str(e)})
            break
        sa = torch.cuda.ExternalStream(part.io_stream)
        sc = torch.cuda.ExternalStream(part.compute_stream)
        cfg = io_cfg(kvx, ctx, kvx.KVX_OP_LOAD, 0, args.mapping, args.stages, args.stage_bytes)

        def gemm_c():
            with torch.cuda.stream(sc):
                torch.matmul(A, B, out=C)

        g_part = _timed(sc, gemm_c, 20, warm=5)
        r = layer_streaming(kvx, ctx, pool, reqs, per_layer, s.num_layers, layer_bytes, cfg,
                            sa, sc, gemm, gemm_ms, timeline=args.timeline)
        _emit({"workload": "llama70b_layer_streaming", "chunk_tokens": args.chunk_tokens,
               "mapping": args.mapping, "partition": "green contexts",
               "io_sms": part.io_sms, "compute_sms": part.compute_sms,
               "gemm_on_compute_partition_ms": round(g_part, 4), **r})
        torch.cuda.synchronize()
        part.close()
    arena.close()
    kvx.kvx_destroy(ctx)


def qwen7b_setup(kvx, wl):
    """Pool, page tables and host arenas of the 64-request batched partial-hit workload."""
    w = wl.qwen7b_batch()
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    dev_tables = [torch.from_numpy(r.page_table).cuda() for r in w.load_requests]
    reqs = kvx.requests_array([(d.data_ptr(), r.page_table, r.n_tokens)
                               for d, r in zip(dev_tables, w.load_requests)])
    ld = kvx.HostBuffer(w.load_arena_bytes)
    _fill_host(ld.array, w.load_arena_bytes, s, w.seed, 2, wl)
    st = kvx.HostBuffer(w.store_arena_bytes)
    st.array[:] = 0
    ch_ld = kvx.chunks_array(w.load_chunks, ld.ptr)
    ch_st = kvx.chunks_array(w.store_chunks, st.ptr)
    return w, pools, pool, dev_tables, reqs, ld, st, ch_ld, ch_st


def concurrent_pair(kvx, ctx_a, ctx_b, pool, reqs, ch_ld, ch_st, sa, sb, cfg_l, cfg_s, reps):
    """The batched load on stream sa and the batched store on stream sb, issued together:
    median (load span, store span, both) in ms from a common start event."""
    spans = []
    for _ in range(reps):
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        start.record(sa)
        sb.wait_event(start)
        kvx.kvx_load_chunks(ctx_a, pool, reqs, ch_ld, cfg=cfg_l, stream=sa.cuda_stream)
        kvx.kvx_store_chunks(ctx_b, pool, reqs, ch_st, cfg=cfg_s, stream=sb.cuda_stream)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(sa)
        eb.record(sb)
        torch.cuda.synchronize()
        spans.append((start.elapsed_time(ea), start.elapsed_time(eb)))
    assert kvx.kvx_get_status(ctx_a, sa.cuda_stream) == 0
    assert kvx.kvx_get_status(ctx_b, sb.cuda_stream) == 0
    return (statistics.median(x[0] for x in spans), statistics.median(x[1] for x in spans),
            statistics.median(max(x) for x in spans))


def qwen7b_measure(args, kvx, wl, link, reps=5, partition_sms=16):
    """Batched partial hits: the load batch and the store batch alone, on two plain streams
    at once (default grids, the store on 8 SMs; and the store on 16 or 6 SMs), on the streams
    of two I/O partitions (green contexts) at once, and in one exchange launch; each against
    the bound max(load / H2D, store / D2H, both / bidir)."""
    w, pools, pool, dev_tables, reqs, ld, st, ch_ld, ch_st = qwen7b_setup(kvx, wl)
    ctx_a, ctx_b = kvx.kvx_create(0, 64 << 20), kvx.kvx_create(0, 64 << 20)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    Nl, Ns = w.load_bytes(), w.store_bytes()
    bound_ms = max(Nl / (link["h2d"] * GB), Ns / (link["d2h"] * GB),
                   (Nl + Ns) / (link["bidir"] * GB)) * 1e3
    load_ms = _timed(sa, lambda: kvx.kvx_load_chunks(ctx_a, pool, reqs, ch_ld,
                                                     stream=sa.cuda_stream), reps)
    store_ms = _timed(sb, lambda: kvx.kvx_store_chunks(ctx_b, pool, reqs, ch_st,
                                                       stream=sb.cuda_stream), reps)
    la, sbm, both = concurrent_pair(kvx, ctx_a, ctx_b, pool, reqs, ch_ld, ch_st, sa, sb,
                                    None, None, reps)
    out = {"workload": "qwen7b_batched_partial_hits", "requests": len(w.load_requests),
           "load_bytes": Nl, "store_bytes": Ns,
           "load_chunks": len(w.load_chunks), "store_chunks": len(w.store_chunks),
           "bound_ms": round(bound_ms, 3),
           "bound_note": "max(load / H2D, store / D2H, (load + store) / bidirectional) with "
                         "this run's measured link peaks",
           "load_alone_gbs": round(Nl / (load_ms * 1e-3) / GB, 2),
           "store_alone_gbs": round(Ns / (store_ms * 1e-3) / GB, 2),
           "two_streams": {"load_gbs": round(Nl / (la * 1e-3) / GB, 2),
                           "store_gbs": round(Ns / (sbm * 1e-3) / GB, 2),
                           "aggregate_gbs": round((Nl + Ns) / (both * 1e-3) / GB, 2),
                           "ms": round(both, 3), "frac_of_bound": round(bound_ms / both, 4)}}
    # Two plain streams with the store on 16 or 6 SMs instead of its default 8: beside a load
    # that saturates H2D a store gets about 10 GB/s per SM, so 6-8 SMs finish it well inside
    # the bound while taking no link bandwidth the load needs; on 16 SMs it takes ~160 GB/s
    # from the load.
    for cap in (16, 6):
        cfg_sc = kvx.kvx_default_launch_cfg(ctx_b, kvx.KVX_OP_STORE)
        cfg_sc.sm_cap = cap
        lac, sbc, bothc = concurrent_pair(kvx, ctx_a, ctx_b, pool, reqs, ch_ld, ch_st, sa, sb,
                                          None, cfg_sc, reps)
        out[f"two_streams_store_{cap}sm"] = {
            "load_gbs": round(Nl / (lac * 1e-3) / GB, 2),
            "store_gbs": round(Ns / (sbc * 1e-3) / GB, 2),
            "aggregate_gbs": round((Nl + Ns) / (bothc * 1e-3) / GB, 2),
            "ms": round(bothc, 3), "frac_of_bound": round(bound_ms / bothc, 4)}
    # Two I/O partitions, one per stream, so the two kernels run on fixed disjoint SM sets.
    try:
        part = kvx.kvx_partition_create(0, partition_sms, -1, 0, io_groups=2)
    except kvx.KvxError as e:
        out["two_partitions"] = {"unavailable": str(e)}
        part = None
    if part is not None:
        pa = torch.cuda.ExternalStream(part.io_streams[0])
        pb = torch.cuda.ExternalStream(part.io_streams[1])
        cfg_l = kvx.kvx_default_launch_cfg(ctx_a, kvx.KVX_OP_LOAD)
        cfg_s = kvx.kvx_default_launch_cfg(ctx_b, kvx.KVX_OP_STORE)
        cfg_l.sm_cap = cfg_s.sm_cap = 0  # each partition bounds its kernel's SMs
        la2, sb2, both2 = concurrent_pair(kvx, ctx_a, ctx_b, pool, reqs, ch_ld, ch_st, pa, pb,
                                          cfg_l, cfg_s, reps)
        out["two_partitions"] = {"io_sms": list(part.io_sms_list),
                                 "load_gbs": round(Nl / (la2 * 1e-3) / GB, 2),
                                 "store_gbs": round(Ns / (sb2 * 1e-3) / GB, 2),
                                 "aggregate_gbs": round((Nl + Ns) / (both2 * 1e-3) / GB, 2),
                                 "ms": round(both2, 3),
                                 "frac_of_bound": round(bound_ms / both2, 4)}
        torch.cuda.synchronize()
        part.close()
    xcfg = parse_cfg(kvx, ctx_a, kvx.KVX_OP_EXCHANGE, getattr(args, "exchange_cfg", ""))
    x_ms = _timed(sa, lambda: kvx.kvx_exchange_chunks(ctx_a, pool, reqs, ch_st, reqs, ch_ld,
                                                       cfg=xcfg, stream=sa.cuda_stream), reps)
    assert kvx.kvx_get_status(ctx_a, sa.cuda_stream) == 0
    out["exchange_one_launch"] = {
        "ms": round(x_ms, 3), "aggregate_gbs": round((Nl + Ns) / (x_ms * 1e-3) / GB, 2),
        "frac_of_bound": round(bound_ms / x_ms, 4),
        "model_ms": round(kvx.kvx_estimate_pair_us(kvx.kvx_default_link_model(),
                                                   kvx.KVX_OP_EXCHANGE, Ns, Nl, 0,
                                                   xcfg) * 1e-3, 3)}
    ld.close()
    st.close()
    kvx.kvx_destroy(ctx_a)
    kvx.kvx_destroy(ctx_b)
    del pools
    return out


def measure_link(dev, stream, gib=4, reps=8):
    """Best-of-reps pinned cudaMemcpyAsync rates: H2D, D2H, and both at once (GB/s)."""
    n = gib << 30
    link, samples = {}, {}
    hp = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dp = torch.empty(n, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for name, fn in (("h2d", lambda: dp.copy_(hp, non_blocking=True)),
                         ("d2h", lambda: hp.copy_(dp, non_blocking=True))):
            for _ in range(2):
                fn()
            t = EventTimer(stream)
            for _ in range(reps):
                e = t.start()
                fn()
                t.stop(e)
            stream.synchronize()
            gbs = [n / (ms * 1e-3) / GB for ms in t.ms()]
            link[name] = round(max(gbs), 1)
            samples[name] = [round(x, 1) for x in gbs]
    hp2 = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dp2 = torch.empty(n, dtype=torch.uint8, device=dev)
    s2 = torch.cuda.Stream(device=dev)
    bid = []
    for rep in range(reps + 1):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s2.wait_event(e0)
        first, second = (stream, s2) if rep % 2 else (s2, stream)
        with torch.cuda.stream(first):
            (dp.copy_(hp, non_blocking=True) if first is stream else
             hp2.copy_(dp2, non_blocking=True))
        with torch.cuda.stream(second):
            (dp.copy_(hp, non_blocking=True) if second is stream else
             hp2.copy_(dp2, non_blocking=True))
        e1, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        e2.record(s2)
        torch.cuda.synchronize()
        if rep:
            ms = max(e0.elapsed_time(e1), e0.elapsed_time(e2))
            bid.append(2 * n / (ms * 1e-3) / GB)
    link["bidir"] = round(max(bid), 1)
    samples["bidir"] = [round(x, 1) for x in bid]
    return link, samples


def run_qwen7b(args, kvx, wl):
    """64 requests with partial prefix hits: one batched load and one batched store at the
    same time, on two plain streams, on two I/O partitions, and in one exchange launch."""
    link, _ = measure_link(torch.device("cuda", 0), torch.cuda.Stream(), reps=4)
    _emit({**qwen7b_measure(args, kvx, wl, link, partition_sms=args.partition_sms_qwen),
           "link_peaks_gbs": link})


def run_mla_sweep(args, kvx, wl):
    """MLA latent cache (61 layers x 1152 B per token), page size x chunk size grid, kernel
    against the per-page DMA baseline, both directions."""
    ctx = kvx.kvx_create(0, 64 << 20)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    for P in wl.MLA_PAGE_SIZES:
        for Cb in wl.MLA_CHUNK_BYTES:
            w = wl.mla_sweep(P, Cb)
            s = w.shape
            pools = _pool_tensor(s, w.seed, wl)
            pool = kvx.Pool.from_tensor(pools, s.page_size)
            src, dst = w.store_requests[0], w.load_requests[0]
            ps = torch.from_numpy(src.page_table).cuda()
            pd = torch.from_numpy(dst.page_table).cuda()
            rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
            rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
            arena = kvx.HostBuffer(w.store_arena_bytes)
            arena.array[:] = 0
            ch = kvx.chunks_array(w.store_chunks, arena.ptr)
            N = w.store_bytes()
            st_ms = _timed(stream, lambda: kvx.kvx_store_chunks(ctx, pool, rs, ch, stream=sh), 5)
            ld_ms = _timed(stream, lambda: kvx.kvx_load_chunks(ctx, pool, rd, ch, stream=sh), 5)
            segs = kvx.kvx_last_launch(ctx)[0]
            # Host cost of one call: validation, descriptor packing, copy and launch (the
            # kernel runs asynchronously after the call returns).
            stream.synchronize()
            host_us = []
            for _ in range(5):
                t0 = time.perf_counter()
                kvx.kvx_load_chunks(ctx, pool, rd, ch, stream=sh)
                host_us.append((time.perf_counter() - t0) * 1e6)
                stream.synchronize()
            dma = {}
            for name, d, rq in (("store", kvx.KVX_DIR_GATHER, rs),
                                ("load", kvx.KVX_DIR_SCATTER, rd)):
                kvx.kvx_dma_baseline(ctx, d, pool, rq, ch, stream=sh)
                stream.synchronize()
                t0 = time.perf_counter()
                n = kvx.kvx_dma_baseline(ctx, d, pool, rq, ch, stream=sh)
                stream.synchronize()
                dma[name] = (N / (time.perf_counter() - t0) / GB, n)
            assert kvx.kvx_get_status(ctx, sh) == 0
            _emit({"workload": "mla_sweep", "page_size": P, "chunk_kib": Cb >> 10,
                   "tokens_per_chunk": w.store_chunks[0].n_tokens, "chunks": len(w.store_chunks),
                   "segments": segs, "bytes": N,
                   "store_gbs": round(N / (st_ms * 1e-3) / GB, 2),
                   "load_gbs": round(N / (ld_ms * 1e-3) / GB, 2),
                   "dma_store_gbs": round(dma["store"][0], 2),
                   "dma_load_gbs": round(dma["load"][0], 2), "dma_copies": dma["store"][1],
                   "host_us_per_call": round(statistics.median(host_us), 1),
                   "descriptor_bytes": kvx.kvx_last_launch(ctx)[3]})
            arena.close()
            del pools
    kvx.kvx_destroy(ctx)


def run_sm_sweep(args, kvx, wl):
    """SM cap x unroll x threads for store and load of the Llama-3.1-8B-shaped request."""
    w = wl.llama8b()
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src, dst = w.store_requests[0], w.load_requests[0]
    ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
    rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
    rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
    arena = kvx.HostBuffer(w.store_arena_bytes)
    arena.array[:] = 0
    ch = kvx.chunks_array(w.store_chunks, arena.ptr)
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    N = w.store_bytes()
    shapes = [("segment", 1024, 8, 1, 0), ("segment", 512, 8, 1, 0),
              ("bulk", 96, 3, 1, 32768), ("bulk", 96, 2, 1, 49152), ("bulk", 96, 6, 1, 16384),
              ("bulk", 96, 2, 1, 32768)]
    for cap in [int(x) for x in args.sm_caps.split(",")]:
        for mapping, threads, unroll, ctas, stage in shapes:
            row = {"workload": "llama8b_sm_sweep", "sm_cap": cap, "mapping": mapping,
                   "threads": threads, "unroll": unroll, "ctas_per_sm": ctas,
                   "stage_bytes": stage}
            for name, op, fn, rq in (("store", kvx.KVX_OP_STORE, kvx.kvx_store_chunks, rs),
                                     ("load", kvx.KVX_OP_LOAD, kvx.kvx_load_chunks, rd)):
                c = kvx.kvx_default_launch_cfg(ctx, op)
                c.sm_cap, c.threads, c.unroll, c.ctas_per_sm = cap, threads, unroll, ctas
                c.mapping = kvx.KVX_MAP_BULK if mapping == "bulk" else kvx.KVX_MAP_WARP_SEGMENT
                c.stage_bytes = stage
                ms = _timed(stream, lambda: fn(ctx, pool, rq, ch, 0, s.num_layers, c, sh), 3, 1)
                row[f"{name}_gbs"] = round(N / (ms * 1e-3) / GB, 2)
            _emit(row)
    assert kvx.kvx_get_status(ctx, sh) == 0
    arena.close()
    kvx.kvx_destroy(ctx)


def run_transform_sweep(args, kvx, wl):
    """Launch shapes of the HBM transform (chunks in device memory), Llama-3.1-8B shape."""
    w = wl.llama8b()
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src, dst = w.store_requests[0], w.load_requests[0]
    ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
    rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
    rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
    dchunk = torch.empty(w.store_arena_bytes, dtype=torch.uint8, device="cuda")
    ch = kvx.chunks_array(w.store_chunks, dchunk.data_ptr())
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    N = w.store_bytes()
    hbm, _ = peaks()
    # Reference: a plain device-to-device copy of the same bytes in this run.
    dsrc = torch.empty(N, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        copy_ms = _timed(stream, lambda: dchunk.copy_(dsrc), 10, 3)
    del dsrc
    copy_gbs = 2 * N / (copy_ms * 1e-3) / GB
    _emit({"workload": "llama8b_transform_sweep", "reference": "torch copy_ 4 GiB",
           "gbs_2n": round(copy_gbs, 1), "frac": round(copy_gbs / hbm, 4)})
    shapes = [tuple(int(v) for v in x.split(":")) for x in args.transform_shapes.split(",")
              if x] * 2
    for mapping, ctas, threads, unroll, hint, stage, batch in shapes:
        if True:
            row = {"workload": "llama8b_transform_sweep",
                   "mapping": ["segment", "bulk", "cta"][mapping], "ctas_per_sm": ctas,
                   "threads": threads, "unroll": unroll, "store_hint": hint,
                   "stage_bytes": stage, "batch": batch}
            for name, d, rq in (("gather", kvx.KVX_DIR_GATHER, rs),
                                ("scatter", kvx.KVX_DIR_SCATTER, rd)):
                c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_GATHER_HBM)
                c.sm_cap, c.ctas_per_sm, c.threads = 0, ctas, threads
                c.unroll, c.store_hint = unroll, hint
                c.mapping, c.stage_bytes, c.batch = mapping, stage, batch
                ms = _timed(stream, lambda: kvx.kvx_transform_hbm(ctx, d, pool, rq, ch, 0,
                                                                  s.num_layers, c, sh), 10, 3)
                gbs = 2 * N / (ms * 1e-3) / GB
                row[f"{name}_gbs_2n"] = round(gbs, 1)
                row[f"{name}_frac"] = round(gbs / hbm, 4)
                row[f"{name}_of_copy"] = round(gbs / copy_gbs, 4)
            _emit(row)
    assert kvx.kvx_get_status(ctx, sh) == 0
    kvx.kvx_destroy(ctx)


def run_batch_sweep(args, kvx, wl):
    """Segments resolved per warp at once, on the MLA latent shape with short segments."""
    ctx = kvx.kvx_create(0, 64 << 20)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    for P in (1, 8):
        w = wl.mla_sweep(P, 1 << 20)
        s = w.shape
        pools = _pool_tensor(s, w.seed, wl)
        pool = kvx.Pool.from_tensor(pools, s.page_size)
        src, dst = w.store_requests[0], w.load_requests[0]
        ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
        rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
        rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
        arena = kvx.HostBuffer(w.store_arena_bytes)
        arena.array[:] = 0
        ch = kvx.chunks_array(w.store_chunks, arena.ptr)
        N = w.store_bytes()
        for batch in (0, 1, 2, 4, 8, 16, 28, 32):
            for cap in (16, 32):
                row = {"workload": "mla_batch_sweep", "page_size": P, "batch": batch,
                       "sm_cap": cap}
                for name, op, fn, rq in (("store", kvx.KVX_OP_STORE, kvx.kvx_store_chunks, rs),
                                         ("load", kvx.KVX_OP_LOAD, kvx.kvx_load_chunks, rd)):
                    c = kvx.kvx_default_launch_cfg(ctx, op)
                    c.batch, c.sm_cap = batch, cap
                    ms = _timed(stream, lambda: fn(ctx, pool, rq, ch, 0, s.num_layers, c, sh), 5)
                    row[f"{name}_gbs"] = round(N / (ms * 1e-3) / GB, 2)
                _emit(row)
        arena.close()
        del pools
    assert kvx.kvx_get_status(ctx, sh) == 0
    kvx.kvx_destroy(ctx)


def run_token_major(args, kvx, wl):
    """Store and load of the MLA latent (1, 2 and 16 tokens per page) and of the llama8b
    request in token-major chunks of about 2 MiB over all layers, whose page segments of more
    than one token are strided rows on the chunk side, on 4 and 16 SMs and without a
    configuration, and the one-launch round trip and an exchange of two such batches
    without a configuration."""
    ctx = kvx.kvx_create(0, 64 << 20)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    for name, P in (("mla", 1), ("mla", 2), ("mla", 16), ("llama8b", 16)):
        w = wl.mla_sweep(P, 1 << 20) if name == "mla" else wl.llama8b()
        s = w.shape
        tpc = max((2 << 20) // (s.token_bytes * s.num_layers * s.kv_factor), 16)
        specs = wl.split_tokens(0, 0, w.store_requests[0].n_tokens, tpc, 0, s.num_layers,
                                wl.TOKEN_MAJOR)
        wl.place_chunks(specs, s)
        pools = _pool_tensor(s, w.seed, wl)
        pool = kvx.Pool.from_tensor(pools, s.page_size)
        src, dst = w.store_requests[0], w.load_requests[0]
        ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
        rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
        rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
        arena = kvx.HostBuffer(wl._arena_bytes(specs, s))
        arena.array[:] = 0
        ch = kvx.chunks_array(specs, arena.ptr)
        N = sum(c.nbytes(s) for c in specs)
        for cap in (4, 16, None):
            row = {"workload": f"{name}_token_major", "page_size": P, "chunks": len(specs),
                   "sm_cap": cap if cap else "default"}
            for op_name, op, fn, rq in (("store", kvx.KVX_OP_STORE, kvx.kvx_store_chunks, rs),
                                        ("load", kvx.KVX_OP_LOAD, kvx.kvx_load_chunks, rd)):
                c = None
                if cap:
                    c = kvx.kvx_default_launch_cfg(ctx, op)
                    c.sm_cap = cap
                ms = _timed(stream, lambda: fn(ctx, pool, rq, ch, 0, s.num_layers, c, sh), 3)
                row[f"{op_name}_gbs"] = round(N / (ms * 1e-3) / GB, 2)
            if cap is None:
                # The one-launch round trip, both directions; and an exchange storing the
                # request into the chunks while loading a second arena into the other pages.
                ms = _timed(stream, lambda: kvx.kvx_roundtrip_chunks(
                    ctx, pool, rs, rd, ch, 0, s.num_layers, None, sh), 3)
                row["roundtrip_gbs"] = round(2 * N / (ms * 1e-3) / GB, 2)
                other = kvx.HostBuffer(wl._arena_bytes(specs, s))
                other.array[:] = 0
                ch2 = kvx.chunks_array(specs, other.ptr)
                ms = _timed(stream, lambda: kvx.kvx_exchange_chunks(
                    ctx, pool, rs, ch, rd, ch2, 0, s.num_layers, None, sh), 3)
                row["exchange_gbs"] = round(2 * N / (ms * 1e-3) / GB, 2)
                other.close()
            _emit(row)
        arena.close()
        del pools
        torch.cuda.empty_cache()
    assert kvx.kvx_get_status(ctx, sh) == 0
    kvx.kvx_destroy(ctx)


def run_mla_blocks(args, kvx, wl):
    """Per-block object layout (STRIPED chunks, one per page, 61 layer objects each,
    4096-aligned): one store of all layers, 61 per-layer loads, and the per-object DMA
    baseline."""
    ctx = kvx.kvx_create(0, 64 << 20)
    stream = torch.cuda.Stream(priority=-1)
    sh = stream.cuda_stream
    for P in (16, 32, 64):
        w = wl.mla_blocks(P)
        s = w.shape
        pools = _pool_tensor(s, w.seed, wl)
        pool = kvx.Pool.from_tensor(pools, s.page_size)
        src, dst = w.store_requests[0], w.load_requests[0]
        ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
        rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
        rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
        arena = kvx.HostBuffer(w.store_arena_bytes)
        arena.array[:] = 0
        ch = kvx.chunks_array(w.store_chunks, arena.ptr)
        N = 16384 * s.num_layers * s.token_bytes
        st_ms = _timed(stream, lambda: kvx.kvx_store_chunks(ctx, pool, rs, ch, stream=sh), 5)

        def per_layer():
            for l in range(s.num_layers):
                kvx.kvx_load_chunks(ctx, pool, rd, ch, l, l + 1, stream=sh)

        ld_ms = _timed(stream, per_layer, 5)
        # The same per-layer loads as prepared plans, launched one by one and as one graph.
        plans = [kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, pool, rd, ch, l, l + 1, None, sh)
                 for l in range(s.num_layers)]

        def per_layer_plans():
            for pl in plans:
                kvx.kvx_plan_launch(pl, sh)

        plan_ms = _timed(stream, per_layer_plans, 5)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            cs = torch.cuda.current_stream().cuda_stream
            for pl in plans:
                kvx.kvx_plan_launch(pl, cs)
        def replay():
            with torch.cuda.stream(stream):
                graph.replay()

        graph_ms = _timed(stream, replay, 5)
        # The same plans launched to overlap (programmatic dependent launch): each layer's
        # load may start while the previous one drains.
        oc = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_LOAD)
        oc.overlap = 1
        oplans = [kvx.kvx_plan_create(ctx, kvx.KVX_OP_LOAD, pool, rd, ch, l, l + 1, oc, sh)
                  for l in range(s.num_layers)]

        def per_layer_overlap():
            for pl in oplans:
                kvx.kvx_plan_launch(pl, sh)

        overlap_ms = _timed(stream, per_layer_overlap, 5)

        def per_layer_calls_overlap():
            for l in range(s.num_layers):
                kvx.kvx_load_chunks(ctx, pool, rd, ch, l, l + 1, oc, sh)

        ocall_ms = _timed(stream, per_layer_calls_overlap, 5)
        ograph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ograph, stream=stream):
            cs = torch.cuda.current_stream().cuda_stream
            for pl in oplans:
                kvx.kvx_plan_launch(pl, cs)

        def oreplay():
            with torch.cuda.stream(stream):
                ograph.replay()

        ograph_ms = _timed(stream, oreplay, 5)
        torch.cuda.synchronize()
        del graph, ograph
        for pl in plans + oplans:
            kvx.kvx_plan_destroy(pl)
        kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_GATHER, pool, rs, ch, stream=sh)
        stream.synchronize()
        t0 = time.perf_counter()
        n = kvx.kvx_dma_baseline(ctx, kvx.KVX_DIR_GATHER, pool, rs, ch, stream=sh)
        stream.synchronize()
        dma_s = time.perf_counter() - t0
        assert kvx.kvx_get_status(ctx, sh) == 0
        _emit({"workload": "mla_block_objects", "page_size": P, "blocks": len(w.store_chunks),
               "object_bytes": P * s.token_bytes,
               "object_stride": -(-P * s.token_bytes // 4096) * 4096,
               "payload_bytes": N, "arena_bytes": w.store_arena_bytes,
               "store_gbs": round(N / (st_ms * 1e-3) / GB, 2),
               "per_layer_load_gbs": round(N / (ld_ms * 1e-3) / GB, 2),
               "per_layer_load_ms": round(ld_ms / s.num_layers, 4),
               "per_layer_load_overlap_gbs": round(N / (ocall_ms * 1e-3) / GB, 2),
               "per_layer_plans_gbs": round(N / (plan_ms * 1e-3) / GB, 2),
               "per_layer_graph_gbs": round(N / (graph_ms * 1e-3) / GB, 2),
               "per_layer_plans_overlap_gbs": round(N / (overlap_ms * 1e-3) / GB, 2),
               "per_layer_graph_overlap_gbs": round(N / (ograph_ms * 1e-3) / GB, 2),
               "dma_store_gbs": round(N / dma_s / GB, 2), "dma_copies": n})
        arena.close()
        del pools
    kvx.kvx_destroy(ctx)


def eviction_leg(kvx, ctx, pool, rs, ch, num_layers, N, seed, caps=(1, 2, 4)):
    """Background eviction: a store of the request by a 1-, 2- or 4-SM kernel on a
    low-priority stream while a decode-like, HBM-bound bf16 GEMV loop runs on a
    high-priority stream; decode step time alone vs with the eviction running."""
    low = torch.cuda.Stream(priority=0)
    high = torch.cuda.Stream(priority=-1)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    Wm = torch.randn(16384, 32768, device="cuda", dtype=torch.bfloat16, generator=g)  # 1 GiB
    x = torch.randn(32768, 1, device="cuda", dtype=torch.bfloat16, generator=g)
    y = torch.empty(16384, 1, device="cuda", dtype=torch.bfloat16)

    def decode(n):
        with torch.cuda.stream(high):
            for _ in range(n):
                torch.matmul(Wm, x, out=y)

    decode(20)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(high)
    decode(200)
    e1.record(high)
    torch.cuda.synchronize()
    step_alone = e0.elapsed_time(e1) / 200
    rows = []
    for cap in caps:
        cfg = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_STORE)
        cfg.sm_cap = cap
        cfg.store_hint = kvx.KVX_HINT_DEFAULT
        # Store alone on the low-priority stream.
        st_ms = _timed(low, lambda: kvx.kvx_store_chunks(ctx, pool, rs, ch, 0, num_layers,
                                                         cfg, low.cuda_stream), 2, 1)
        n_steps = max(50, int(st_ms / step_alone))
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(low)
        kvx.kvx_store_chunks(ctx, pool, rs, ch, 0, num_layers, cfg, low.cuda_stream)
        a1.record(low)
        d0.record(high)
        decode(n_steps)
        d1.record(high)
        torch.cuda.synchronize()
        assert kvx.kvx_get_status(ctx, low.cuda_stream) == 0
        step_with = d0.elapsed_time(d1) / n_steps
        rows.append({"workload": "background_eviction", "sm_cap": cap,
                     "store_alone_gbs": round(N / (st_ms * 1e-3) / GB, 2),
                     "store_under_decode_gbs": round(N / (a0.elapsed_time(a1) * 1e-3) / GB, 2),
                     "decode_step_alone_ms": round(step_alone, 4),
                     "decode_step_with_eviction_ms": round(step_with, 4),
                     "decode_slowdown_pct": round(100 * (step_with / step_alone - 1), 2),
                     "decode_steps": n_steps,
                     "decode_gemv": "bf16 [16384 x 32768] x [32768], 1 GiB of weights per "
                                    "step"})
    del Wm, x, y
    return rows


def run_eviction(args, kvx, wl):
    """Background eviction of the llama8b request under a decode-like GEMV loop."""
    w = wl.llama8b()
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src = w.store_requests[0]
    ps = torch.from_numpy(src.page_table).cuda()
    rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
    arena = kvx.HostBuffer(w.store_arena_bytes)
    arena.array[:] = 0
    ch = kvx.chunks_array(w.store_chunks, arena.ptr)
    ctx = kvx.kvx_create(0)
    for row in eviction_leg(kvx, ctx, pool, rs, ch, s.num_layers, w.store_bytes(), w.seed):
        _emit(row)
    arena.close()
    kvx.kvx_destroy(ctx)


def run_profile_small(args, kvx, wl):
    """A small case for ncu captures: the Llama-3.1-8B shape cut to 8192 tokens (1 GiB per
    direction, above the 129 MB L2) in a 1024-page pool (2 GiB), one operation 3 times
    with the library's default launch configuration.  The *_token_major operations use
    token-major chunks of 16 tokens over all layers instead of the layer-major ones."""
    w = wl.llama8b(num_pages=1024, n_tokens=8192)
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src, dst = w.store_requests[0], w.load_requests[0]
    ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
    rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
    rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
    ctx = kvx.kvx_create(0)
    sh = torch.cuda.current_stream().cuda_stream
    specs = w.store_chunks
    if args.profile_op.endswith("_token_major"):  # 16-token chunks over all layers (2 MiB)
        specs = wl.split_tokens(0, 0, src.n_tokens, 16, 0, s.num_layers, wl.TOKEN_MAJOR)
        wl.place_chunks(specs, s)
    if args.profile_op in ("store", "load", "exchange", "roundtrip", "exchange_shared",
                           "load_bulk", "store_bulk", "load_4sm", "store_token_major",
                           "load_token_major", "roundtrip_token_major"):
        buf = kvx.HostBuffer(wl._arena_bytes(specs, s))
        buf.array[:] = 0
        ch = kvx.chunks_array(specs, buf.ptr)
    else:
        dchunk = torch.zeros(w.store_arena_bytes, dtype=torch.uint8, device="cuda")
        ch = kvx.chunks_array(w.store_chunks, dchunk.data_ptr())
    half = len(w.store_chunks) // 2
    for _ in range(3):
        if args.profile_op in ("roundtrip", "roundtrip_token_major"):
            # store every chunk and load it into other pages
            kvx.kvx_roundtrip_chunks(ctx, pool, rs, rd, ch, stream=sh)
        elif args.profile_op == "exchange_shared":  # store a quarter, load three quarters
            q = len(w.store_chunks) // 4
            kvx.kvx_exchange_chunks(ctx, pool, rs, np.ascontiguousarray(ch[:q]), rd,
                                    np.ascontiguousarray(ch[q:]), stream=sh)
        elif args.profile_op == "load_bulk":  # the load, bulk-copy mapping on 4 SMs
            c = io_cfg(kvx, ctx, kvx.KVX_OP_LOAD, 4, "bulk", 3, 32768)
            kvx.kvx_load_chunks(ctx, pool, rd, ch, cfg=c, stream=sh)
        elif args.profile_op == "store_bulk":  # the store, bulk-copy mapping on 4 SMs
            c = io_cfg(kvx, ctx, kvx.KVX_OP_STORE, 4, "bulk", 6, 16384)
            kvx.kvx_store_chunks(ctx, pool, rs, ch, cfg=c, stream=sh)
        elif args.profile_op == "load_4sm":  # the load, register mapping on 4 SMs
            c = io_cfg(kvx, ctx, kvx.KVX_OP_LOAD, 4)
            kvx.kvx_load_chunks(ctx, pool, rd, ch, cfg=c, stream=sh)
        elif args.profile_op == "gather_cta":  # the HBM gather, CTA-per-segment mapping
            c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_GATHER_HBM)
            c.mapping, c.ctas_per_sm, c.threads, c.unroll = kvx.KVX_MAP_CTA, 2, 512, 8
            kvx.kvx_transform_hbm(ctx, kvx.KVX_DIR_GATHER, pool, rs, ch, cfg=c, stream=sh)
        elif args.profile_op == "exchange":  # store the first half, load the second half
            kvx.kvx_exchange_chunks(ctx, pool, rs, np.ascontiguousarray(ch[:half]), rd,
                                    np.ascontiguousarray(ch[half:]), stream=sh)
        elif args.profile_op in ("store", "store_token_major"):
            kvx.kvx_store_chunks(ctx, pool, rs, ch, stream=sh)
        elif args.profile_op in ("load", "load_token_major"):
            kvx.kvx_load_chunks(ctx, pool, rd, ch, stream=sh)
        else:
            d = kvx.KVX_DIR_GATHER if args.profile_op == "gather" else kvx.KVX_DIR_SCATTER
            kvx.kvx_transform_hbm(ctx, d, pool, rs if d == kvx.KVX_DIR_GATHER else rd, ch,
                                  stream=sh)
    torch.cuda.synchronize()
    assert kvx.kvx_get_status(ctx, sh) == 0
    items, ctas, threads, _ = kvx.kvx_last_launch(ctx)
    _emit({"workload": "profile_small", "op": args.profile_op,
           "bytes": sum(c.nbytes(s) for c in specs),
           "items": items, "ctas": ctas, "threads": threads})
    kvx.kvx_destroy(ctx)


def run_roundtrip_sweep(args, kvx, wl):
    """The headline round trip (llama8b, store all chunks + load them into fresh pages) in
    G chunk groups, issued three ways: one kvx_exchange_chunks call per launch, prepared
    exchange plans, and the plans captured in one CUDA graph per step.  Two step shapes:
    pipelined (a step's first launch loads the previous step's last group) and
    self-contained (first launch stores only, last launch loads only)."""
    w = wl.llama8b()
    s = w.shape
    N = w.store_bytes()
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src_h, dst_h = w.store_requests[0].page_table, w.load_requests[0].page_table
    src_d, dst_d = torch.from_numpy(src_h).cuda(), torch.from_numpy(dst_h).cuda()
    rs = kvx.requests_array([(src_d.data_ptr(), src_h, w.store_requests[0].n_tokens)])
    rd = kvx.requests_array([(dst_d.data_ptr(), dst_h, w.load_requests[0].n_tokens)])
    host = kvx.HostBuffer(w.store_arena_bytes)
    host.array[:] = 0
    chunks = kvx.chunks_array(w.store_chunks, host.ptr)
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    empty = np.zeros(0, dtype=chunks.dtype)
    reps = max(5, args.steps // 2)
    # One kvx_roundtrip_chunks launch per step, over a few launch shapes.
    for cap, unroll, threads in [tuple(int(v) for v in x.split(":"))
                                 for x in args.fused_cfgs.split(",") if x]:
        c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_ROUNDTRIP)
        c.sm_cap, c.unroll, c.threads = cap, unroll, threads

        def fused():
            kvx.kvx_roundtrip_chunks(ctx, pool, rs, rd, chunks, cfg=c, stream=sh)

        for _ in range(3):
            fused()
        t = EventTimer(stream)
        host_ms = []
        for _ in range(reps):
            stream.synchronize()
            t0 = time.perf_counter()
            e = t.start()
            fused()
            t.stop(e)
            stream.synchronize()
            host_ms.append((time.perf_counter() - t0) * 1e3)
        assert kvx.kvx_get_status(ctx, sh) == 0
        ms = statistics.median(t.ms())
        _emit({"workload": "llama8b_roundtrip_fused", "cfg": c.as_dict(),
               "ctas": kvx.kvx_last_launch(ctx)[1],
               "step_ms": round(ms, 4), "gbs": round(2 * N / (ms * 1e-3) / GB, 2),
               "min_gbs": round(2 * N / (min(t.ms()) * 1e-3) / GB, 2),
               "host_gbs": round(2 * N / (statistics.median(host_ms) * 1e-3) / GB, 2)})
    for G in [int(x) for x in args.group_list.split(",") if x]:
        bounds = np.linspace(0, len(chunks), G + 1).astype(int)
        groups = [np.ascontiguousarray(chunks[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        # launch list of one step: (store, load) pairs
        pipelined = [(groups[0], groups[-1])] + [(groups[k], groups[k - 1]) for k in range(1, G)]
        selfc = ([(groups[0], empty)] + [(groups[k], groups[k - 1]) for k in range(1, G)] +
                 [(empty, groups[-1])])
        plans = {}

        def plan_of(pair):
            key = (id(pair[0]), id(pair[1]))
            if key not in plans:
                plans[key] = kvx.kvx_plan_create_exchange(ctx, pool, rs, pair[0], rd, pair[1],
                                                          stream=sh)
            return plans[key]

        def by_call(seq):
            for st, ld in seq:
                kvx.kvx_exchange_chunks(ctx, pool, rs, st, rd, ld, stream=sh)

        def by_plan(seq):
            for pair in seq:
                kvx.kvx_plan_launch(plan_of(pair), sh)

        for pair in selfc + pipelined:
            plan_of(pair)  # all plans exist before any graph capture
        graphs = {}
        for name, seq in (("pipelined", pipelined), ("self_contained", selfc)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                cs = torch.cuda.current_stream().cuda_stream
                for pair in seq:
                    kvx.kvx_plan_launch(plan_of(pair), cs)
            graphs[name] = g

        def by_graph(name):
            def run(_seq):
                with torch.cuda.stream(stream):
                    graphs[name].replay()
            return run

        row = {"workload": "llama8b_roundtrip_sweep", "groups": G,
               "group_bytes_each_way": int(N // G)}
        for mode, fn_p, fn_s in (("call", by_call, by_call), ("plan", by_plan, by_plan),
                                 ("graph", by_graph("pipelined"), by_graph("self_contained"))):
            # pipelined: prime with a self-contained step minus its flush
            fn_s(selfc[:-1]) if mode != "graph" else by_call(selfc[:-1])
            for _ in range(2):
                fn_p(pipelined)
            t = EventTimer(stream)
            for _ in range(reps):
                e = t.start()
                fn_p(pipelined)
                t.stop(e)
            by_call(selfc[-1:])
            stream.synchronize()
            pip_ms = statistics.median(t.ms())
            # self-contained, device clock and host clock (sync after each step)
            for _ in range(2):
                fn_s(selfc)
            t = EventTimer(stream)
            host_ms = []
            for _ in range(reps):
                stream.synchronize()
                t0 = time.perf_counter()
                e = t.start()
                fn_s(selfc)
                t.stop(e)
                stream.synchronize()
                host_ms.append((time.perf_counter() - t0) * 1e3)
            sc_ms = statistics.median(t.ms())
            row[mode] = {"pipelined_gbs": round(2 * N / (pip_ms * 1e-3) / GB, 2),
                         "self_contained_gbs": round(2 * N / (sc_ms * 1e-3) / GB, 2),
                         "self_contained_host_gbs": round(
                             2 * N / (statistics.median(host_ms) * 1e-3) / GB, 2)}
        assert kvx.kvx_get_status(ctx, sh) == 0
        _emit(row)
        del graphs
        torch.cuda.synchronize()
        for h in plans.values():
            kvx.kvx_plan_destroy(h)
    host.close()
    del pools
    torch.cuda.empty_cache()
    # The one-launch round trip on the MLA latent (61 layers, 1152-byte tokens, per-layer
    # chunks of 1 MiB): short page segments use the batched lookup.
    for P in [int(x) for x in args.mla_pages.split(",") if x]:
        m = wl.mla_sweep(page_size=P, chunk_bytes=1 << 20)
        ms_ = m.shape
        Nm = m.store_bytes()
        mp = _pool_tensor(ms_, m.seed, wl)
        mpool = kvx.Pool.from_tensor(mp, P)
        a, b = m.store_requests[0], m.load_requests[0]
        ad, bd = torch.from_numpy(a.page_table).cuda(), torch.from_numpy(b.page_table).cuda()
        mrs = kvx.requests_array([(ad.data_ptr(), a.page_table, a.n_tokens)])
        mrd = kvx.requests_array([(bd.data_ptr(), b.page_table, b.n_tokens)])
        mh = kvx.HostBuffer(m.store_arena_bytes)
        mh.array[:] = 0
        mch = kvx.chunks_array(m.store_chunks, mh.ptr)
        for shape_ in [tuple(int(v) for v in x.split(":")) for x in args.mla_cfgs.split(",") if x]:
            c = None  # all fields 0: the library's defaults (cfg = NULL)
            if any(shape_):
                c = kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_ROUNDTRIP)
                for field, val in zip(("sm_cap", "unroll", "threads", "batch"), shape_):
                    if val:
                        setattr(c, field, val)
            ms = _timed(stream, lambda: kvx.kvx_roundtrip_chunks(ctx, mpool, mrs, mrd, mch, cfg=c,
                                                                 stream=sh), reps)
            assert kvx.kvx_get_status(ctx, sh) == 0
            items, ctas, threads, _ = kvx.kvx_last_launch(ctx)
            # The time model with the unit and SM cap the library picked (default link model).
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            unit, cap = kvx.kvx_roundtrip_unit(P, ms_.token_bytes, c, sms)
            mc = c if c is not None else kvx.kvx_default_launch_cfg(ctx, kvx.KVX_OP_ROUNDTRIP)
            mc.sm_cap = cap
            model_ms = kvx.kvx_estimate_pair_us(kvx.kvx_default_link_model(),
                                                kvx.KVX_OP_ROUNDTRIP, Nm, Nm, unit, mc) * 1e-3
            _emit({"workload": "mla_roundtrip_one_launch", "page_size": P,
                   "chunk_bytes": 1 << 20, "cfg": c.as_dict() if c else "defaults",
                   "ctas": ctas, "threads": threads, "bytes_each_way": Nm,
                   "segments_each_way": items // 2, "unit_bytes": unit,
                   "ms": round(ms, 4), "gbs": round(2 * Nm / (ms * 1e-3) / GB, 2),
                   "model_ms": round(model_ms, 4)})
        mh.close()
        del mp
    kvx.kvx_destroy(ctx)


def run_size_sweep(args, kvx, wl):
    """Store and load of 1 to 2048 one-page chunks (all 32 layers, 2 MiB each) of the
    Llama-3.1-8B-shaped request, per call on the device clock, next to the I/O-time model's
    prediction (kvx_estimate_us) for the same bytes."""
    w = wl.llama8b()
    s = w.shape
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src, dst = w.store_requests[0], w.load_requests[0]
    ps, pd = torch.from_numpy(src.page_table).cuda(), torch.from_numpy(dst.page_table).cuda()
    rs = kvx.requests_array([(ps.data_ptr(), src.page_table, src.n_tokens)])
    rd = kvx.requests_array([(pd.data_ptr(), dst.page_table, dst.n_tokens)])
    specs = wl.split_tokens(0, 0, src.n_tokens, s.page_size, 0, s.num_layers, wl.LAYER_MAJOR)
    wl.place_chunks(specs, s)
    arena = kvx.HostBuffer(wl._arena_bytes(specs, s))
    arena.array[:] = 0
    ch = kvx.chunks_array(specs, arena.ptr)
    ctx = kvx.kvx_create(0)
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    model = kvx.kvx_default_link_model()
    n = 1
    while n <= len(specs):
        part = np.ascontiguousarray(ch[:n])
        nbytes = n * specs[0].nbytes(s)
        row = {"workload": "llama8b_size_sweep", "chunks": n, "bytes": nbytes}
        for name, op, fn, rq in (("store", kvx.KVX_OP_STORE, kvx.kvx_store_chunks, rs),
                                 ("load", kvx.KVX_OP_LOAD, kvx.kvx_load_chunks, rd)):
            def call():
                fn(ctx, pool, rq, part, stream=sh)

            ms = _timed(stream, call, 10, 3)
            row[f"{name}_us"] = round(ms * 1e3, 2)
            row[f"{name}_gbs"] = round(nbytes / (ms * 1e-3) / GB, 2)
            row[f"{name}_model_us"] = round(kvx.kvx_estimate_us(model, op, nbytes), 2)
            if nbytes > (64 << 20):
                continue
            # Where a small call's fixed cost goes: host time of the call alone, calls issued
            # back to back (the host runs ahead), a prepared plan, and that plan as a graph.
            host = []
            for _ in range(20):
                stream.synchronize()
                t0 = time.perf_counter()
                call()
                host.append(time.perf_counter() - t0)
            stream.synchronize()
            reps = 20
            row[f"{name}_host_us"] = round(statistics.median(host) * 1e6, 2)
            row[f"{name}_back_to_back_us"] = round(
                _timed(stream, lambda: [call() for _ in range(reps)], 5, 2) * 1e3 / reps, 2)
            plan = kvx.kvx_plan_create(ctx, op, pool, rq, part, 0, None, None, sh)
            row[f"{name}_plan_us"] = round(
                _timed(stream, lambda: kvx.kvx_plan_launch(plan, sh), 10, 3) * 1e3, 2)
            # The same plan, overlapped (programmatic dependent launch), launched back to back:
            # the repeated transfer moves the same bytes, so each launch may overlap the last.
            oc = kvx.kvx_default_launch_cfg(ctx, op)
            oc.overlap = 1
            oplan = kvx.kvx_plan_create(ctx, op, pool, rq, part, 0, None, oc, sh)
            row[f"{name}_plan_overlap_back_to_back_us"] = round(
                _timed(stream, lambda: [kvx.kvx_plan_launch(oplan, sh) for _ in range(reps)], 5,
                       2) * 1e3 / reps, 2)
            kvx.kvx_plan_destroy(oplan)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                kvx.kvx_plan_launch(plan, torch.cuda.current_stream().cuda_stream)

            def replay():
                with torch.cuda.stream(stream):
                    graph.replay()

            row[f"{name}_graph_us"] = round(_timed(stream, replay, 10, 3) * 1e3, 2)
            torch.cuda.synchronize()
            del graph
            kvx.kvx_plan_destroy(plan)
        _emit(row)
        n *= 2
    assert kvx.kvx_get_status(ctx, sh) == 0
    arena.close()
    kvx.kvx_destroy(ctx)


def run_roundtrip_under_gemm(args, kvx, wl):
    """The headline round trip (llama8b, one launch) beside a stream of bf16 8192^3 GEMMs:
    round-trip GB/s and GEMM slowdown, on a high-priority stream with the default 16-SM
    grid, and on a 16-SM green-context partition with the GEMMs on the rest."""
    w = wl.llama8b()
    s = w.shape
    N = w.store_bytes()
    pools = _pool_tensor(s, w.seed, wl)
    pool = kvx.Pool.from_tensor(pools, s.page_size)
    src_h, dst_h = w.store_requests[0].page_table, w.load_requests[0].page_table
    src_d, dst_d = torch.from_numpy(src_h).cuda(), torch.from_numpy(dst_h).cuda()
    rs = kvx.requests_array([(src_d.data_ptr(), src_h, w.store_requests[0].n_tokens)])
    rd = kvx.requests_array([(dst_d.data_ptr(), dst_h, w.load_requests[0].n_tokens)])
    host = kvx.HostBuffer(w.store_arena_bytes)
    host.array[:] = 0
    chunks = kvx.chunks_array(w.store_chunks, host.ptr)
    ctx = kvx.kvx_create(0)
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    A = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16, generator=g)
    B = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16, generator=g)
    C = torch.empty(8192, 8192, device="cuda", dtype=torch.bfloat16)
    n_gemm = 60  # about 33 ms of GEMMs, longer than one round trip

    def measure(io_stream, gemm_stream):
        def rt():
            kvx.kvx_roundtrip_chunks(ctx, pool, rs, rd, chunks, stream=io_stream.cuda_stream)

        def gemms():
            with torch.cuda.stream(gemm_stream):
                for _ in range(n_gemm):
                    torch.matmul(A, B, out=C)

        rt_alone = _timed(io_stream, rt, 3, 1)
        with torch.cuda.stream(gemm_stream):
            g_alone = _timed(gemm_stream, gemms, 3, 1)
        both = []
        for _ in range(3):
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(gemm_stream)
            io_stream.wait_event(e0)
            a0 = torch.cuda.Event(enable_timing=True)
            a0.record(io_stream)
            rt()
            a1 = torch.cuda.Event(enable_timing=True)
            a1.record(io_stream)
            gemms()
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(gemm_stream)
            torch.cuda.synchronize()
            both.append((a0.elapsed_time(a1), e0.elapsed_time(e1)))
        rt_ms = statistics.median(x[0] for x in both)
        g_ms = statistics.median(x[1] for x in both)
        assert kvx.kvx_get_status(ctx, io_stream.cuda_stream) == 0
        return {"roundtrip_alone_gbs": round(2 * N / (rt_alone * 1e-3) / GB, 2),
                "roundtrip_beside_gemm_gbs": round(2 * N / (rt_ms * 1e-3) / GB, 2),
                "gemm_alone_ms": round(g_alone, 3), "gemm_beside_roundtrip_ms": round(g_ms, 3),
                "gemm_slowdown_pct": round(100 * (g_ms / g_alone - 1), 2)}

    row = {"workload": "llama8b_roundtrip_under_gemm", "gemms": n_gemm,
           "gemm": "bf16 8192^3 torch.matmul"}
    row["high_priority_stream"] = measure(torch.cuda.Stream(priority=-1), torch.cuda.Stream())
    try:
        part = kvx.kvx_partition_create(0, 16, -1, 0)
        row["green_contexts_16_io_sms"] = measure(torch.cuda.ExternalStream(part.io_stream),
                                                  torch.cuda.ExternalStream(part.compute_stream))
        torch.cuda.synchronize()
        part.close()
    except kvx.KvxError as e:
        row["green_contexts_16_io_sms"] = {"unavailable": str(e)}
    _emit(row)
    host.close()
    kvx.kvx_destroy(ctx)


def run_workload(args):
    torch.cuda.set_device(0)
    from paged_kv_gather_gb300.build import build
    build()
    from paged_kv_gather_gb300 import kvx
    from paged_kv_gather_gb300 import workloads as wl
    {"llama70b": run_llama70b, "qwen7b_batch": run_qwen7b, "mla_sweep": run_mla_sweep,
     "sm_sweep": run_sm_sweep, "transform_sweep": run_transform_sweep,
     "profile_small": run_profile_small, "batch_sweep": run_batch_sweep,
     "mla_blocks": run_mla_blocks, "eviction": run_eviction, "token_major": run_token_major,
     "roundtrip_sweep": run_roundtrip_sweep, "size_sweep": run_size_sweep,
     "roundtrip_under_gemm": run_roundtrip_under_gemm}[args.workload](
        args, kvx, wl)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "llama8b":
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
