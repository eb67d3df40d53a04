#!/usr/bin/env python
"""Benchmark of the TACO fused compress + decompress-reduce hot path on GB300.

One step = compress P bf16 shards [N, h] (one launch) + decompress-reduce
P shards into bf16 [N, h] (one launch), the two kernels of the operator.
The decompress-reduce input is the bundle compressed one buffer set later
(the "received" bundle); buffer sets rotate so that every step reads data
that left L2 long ago. Inputs are synthetic and already resident in HBM.

value = bf16 bytes of the step's P input shards / step time (GB/s),
summed over ranks for N > 1 (each rank its own data: weak scaling).

--impl reference times the CPU oracle (numpy, fp64) on a bounded sample of
the same workload on the host cores, rank 0 only.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import pathlib
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parent
METRIC = "compress / decompress-reduce GB/s (bf16 in) and % of GB300 HBM roofline"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_TARGET_ENERGY = 4096.0


# ------------------------------------------------------------- helpers ----
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["taco", "reference"], default="taco")
    ap.add_argument("--workload", default=None, help="workload name (default: the Qwen-7B long-sequence activation, the largest)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def job_throughput(bytes_per_rank_step: float, world: int, steps: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return bytes_per_rank_step * world * steps / (max_ms * 1e-3) / 1e9


def reduce_max_over_ranks(value: float, device=None) -> float:
    """Max of a float over the ranks of the default process group (identity alone)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text())
        except json.JSONDecodeError:
            pass
    return {}


# The sources each timed kernel is built and launched from (its own file,
# the shared device header, the launch interface and the C ABI's grid sizing).
KERNEL_SOURCES = {
    "compress": "compress_mma.cu",           # the step's compress: tensor-core Hadamard
    "compress_fwht": "compress.cu",          # CUDA-core FWHT alternative
    "decompress_reduce": "decompress_reduce.cu",
    "reduce_recompress": "decompress_reduce.cu",
    "reduce_recompress_pw": "decompress_pw.cu",   # n = 64: the producer-warp kernel
    "decompress_reduce_pw": "decompress_pw.cu",
}
COMMON_SOURCES = ("taco_device.cuh", "taco_launch.h", "taco_abi.cu")


_C_COMMENT = re.compile(r"/\*.*?\*/|//[^\n]*", re.S)


def _code_only(text: str) -> bytes:
    """C/C++ source without comments and trailing blanks: what the compiler sees."""
    lines = [ln.rstrip() for ln in _C_COMMENT.sub("", text).splitlines()]
    return "\n".join(ln for ln in lines if ln).encode()


def source_hash(kernel: str) -> str:
    """Hash of one kernel's sources, comments left out: ties an ncu traffic
    figure to the code it measured."""
    h = hashlib.sha256()
    csrc = ROOT / "grads_taco_compress_gb300" / "csrc"
    for name in (KERNEL_SOURCES[kernel], *COMMON_SOURCES):
        h.update(name.encode())
        h.update(_code_only((csrc / name).read_text()))
    h.update(_code_only((ROOT / "include" / "taco.h").read_text()))
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it matches these sources."""
    f = ROOT / "profiles" / f"{kernel}_{workload}.md"
    if not f.exists():
        return None
    text = f.read_text()
    mh = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    mt = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not mh or not mt or mh.group(1) != source_hash(kernel):
        return None
    return float(mt.group(1))


# --------------------------------------------------------- clock sampler ----
CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


def start_clock_sampler(uuid: str | None):
    cmd = ["nvidia-smi", "--query-gpu=" + ",".join(CLOCK_FIELDS), "--format=csv,noheader,nounits",
           "-lms", "20"]
    if uuid:
        cmd.insert(1, f"--id={uuid}")
    try:
        return subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
    except OSError:
        return None


def stop_clock_sampler(proc) -> dict:
    if proc is None:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}
    proc.terminate()
    try:
        out, _ = proc.communicate(timeout=5)
    except subprocess.TimeoutExpired:
        proc.kill()
        out, _ = proc.communicate()
    return parse_clock_samples(out)


def parse_clock_samples(text: str) -> dict:
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) != len(CLOCK_FIELDS):
            continue
        try:
            sm.append(float(parts[0]))
            smax.append(float(parts[1]))
        except ValueError:
            continue
        for name, val in zip(names, parts[4:]):
            if val.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle ----
def oracle_step(block: int, x_rows: np.ndarray) -> None:
    """Oracle compress of P shards' rows and decompress-reduce of the result."""
    from oracle import taco_oracle as O
    parts = [O.compress(x_rows[p], block, DEFAULT_TARGET_ENERGY) for p in range(x_rows.shape[0])]
    codes = np.stack([c for c, _, _, _ in parts])
    alpha = np.stack([a for _, a, _, _ in parts])
    s = np.stack([s_ for _, _, s_, _ in parts])
    O.decompress_reduce(codes, alpha, s, block)


# The oracle over row ranges on all host cores: one worker process per core
# (started with spawn: a pool forked after CUDA initialisation can hang), one
# BLAS thread each, the sample in shared memory. The oracle itself runs as it
# stands on each range; blocks are independent, so the ranges are too.
_POOL_X = None


def _pool_init(shm_name, shape, block_size):
    from multiprocessing import shared_memory
    global _POOL_X, _POOL_SHM, _POOL_BLOCK
    _POOL_SHM = shared_memory.SharedMemory(name=shm_name)
    _POOL_X = np.ndarray(shape, dtype=np.uint16, buffer=_POOL_SHM.buf)
    _POOL_BLOCK = block_size


def _pool_run(job):
    lo, hi, reps = job
    if hi <= lo:
        return 0.0
    xs = np.ascontiguousarray(_POOL_X[:, lo:hi])
    for _ in range(reps):
        oracle_step(_POOL_BLOCK, xs)
    return 1.0


class OraclePool:
    """Worker processes that time the oracle over row ranges of one sample."""

    def __init__(self, x: np.ndarray, block: int, workers: int | None = None):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        self.workers = max(1, workers or os.cpu_count() or 1)
        self.shm = shared_memory.SharedMemory(create=True, size=max(1, x.nbytes))
        np.ndarray(x.shape, dtype=np.uint16, buffer=self.shm.buf)[...] = x
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(self.workers, initializer=_pool_init,
                                 initargs=(self.shm.name, x.shape, block))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.pool.map(_pool_run, [(0, 1, 1)] * self.workers)      # import and warm every worker

    def time(self, rows: int, reps: int) -> float:
        """Wall seconds of `reps` oracle steps over the first `rows` rows, split across workers."""
        cuts = [rows * i // self.workers for i in range(self.workers + 1)]
        jobs = [(cuts[i], cuts[i + 1], reps) for i in range(self.workers)]
        t0 = time.perf_counter()
        self.pool.map(_pool_run, jobs, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()
        self.shm.close()
        self.shm.unlink()


def cpu_baseline(w, x: np.ndarray, seconds: float) -> dict:
    """The oracle, as it stands, on all host cores over a bounded sample sized to about `seconds`."""
    pool = OraclePool(x, w.block)
    try:
        probe_rows = min(w.N, 4 * pool.workers)
        wall = pool.time(probe_rows, 1)
        rows = int(min(w.N, max(probe_rows, probe_rows * seconds / max(wall, 1e-3))))
        wall = pool.time(rows, 1)
    finally:
        pool.close()
    gbs = x.shape[0] * rows * w.h * 2 / wall / 1e9
    return {"value": round(gbs, 6), "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
            "sample": f"{rows} of {w.N} rows of each of the {x.shape[0]} shards [{w.N},{w.h}] "
                      f"(compress + decompress-reduce, numpy fp64), row ranges over {pool.workers} "
                      f"worker processes, {wall:.1f} s wall"}


def run_reference(args, w) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from grads_taco_compress_gb300 import workloads as W
    x = W.make_shards(w)
    pool = OraclePool(x, w.block)
    try:
        # size each step so that warm-up + timed steps take about two minutes
        probe_rows = min(w.N, 4 * pool.workers)
        per_row = pool.time(probe_rows, 1) / probe_rows
        rows = int(max(1, min(w.N, 120.0 / max(args.steps + args.warmup, 1) / per_row)))
        for _ in range(args.warmup):
            pool.time(rows, 1)
        wall = pool.time(rows, args.steps)
    finally:
        pool.close()
    step_ms = wall / args.steps * 1e3
    value = x.shape[0] * rows * w.h * 2 * args.steps / wall / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "shape": [w.N, w.h], "block": w.block, "P": w.P,
                   "target_energy": DEFAULT_TARGET_ENERGY, "variant": "dual",
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
                         "sample": f"{rows} of {w.N} rows of each of {x.shape[0]} shards per step, "
                                   f"row ranges over {pool.workers} worker processes"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm ----
class StepBuffers:
    """Rotating buffer sets of one workload on the device: P bf16 input
    shards, the compressed bundle, the headers and the bf16 output per set,
    as many sets as make the inputs larger than three L2s in total, so that
    every launch reads data that left L2 long ago."""

    def __init__(self, w, x_host, dev, l2, default_stream):
        import torch

        import grads_taco_compress_gb300 as taco
        self.taco, self.lib, self.w = taco, taco.library(), w
        P, N, h, n = w.P, w.N, w.h, w.block
        self.sb = taco.shard_bytes(N, h, n)
        self.in_bytes = P * N * h * 2
        self.set_bytes = self.in_bytes + P * self.sb + N * h * 2
        self.R = max(3, math.ceil(3 * l2 / self.set_bytes))
        x0 = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).to(dev)
        self.xs = [x0] + [x0.clone() for _ in range(self.R - 1)]
        self.bundles = [torch.empty((P, self.sb), dtype=torch.uint8, device=dev) for _ in range(self.R)]
        self.headers = [torch.empty((P, taco.HEADER_BYTES), dtype=torch.uint8, device=dev)
                        for _ in range(self.R)]
        self.outs = [torch.empty((N, h), dtype=torch.bfloat16, device=dev) for _ in range(self.R)]
        self.ws = taco.new_workspace(P, dev)
        self.sptr = default_stream.cuda_stream
        self.xp = [t.data_ptr() for t in self.xs]
        self.bp = [t.data_ptr() for t in self.bundles]
        self.hp = [t.data_ptr() for t in self.headers]
        self.op = [t.data_ptr() for t in self.outs]
        K = h // n
        self.c_bytes = P * N * h * 3 + P * N * K * 8          # compress: bf16 in, codes + (alpha, s) out
        self.d_bytes = P * N * h + P * N * K * 8 + N * h * 2  # decompress-reduce: P shards in, bf16 out

    def compress(self, k, sp=None):
        w = self.w
        st = self.lib.taco_compress_shards_mma(self.xp[k], w.P, w.N, w.h, w.block, DEFAULT_TARGET_ENERGY, 0,
                                               self.bp[k], self.hp[k], self.ws.data_ptr(), self.ws.numel(),
                                               sp or self.sptr)
        if st:
            raise self.taco.TacoError(st, "taco_compress_shards_mma")

    def decompress(self, k, src, sp=None):
        w = self.w
        st = self.lib.taco_decompress_reduce(self.bp[src], w.P, w.N, w.h, w.block, self.op[k], sp or self.sptr)
        if st:
            raise self.taco.TacoError(st, "taco_decompress_reduce")


def time_region(stream, iters, fn) -> float:
    """Seconds per call of `fn(i)` over `iters` back-to-back calls, CUDA events on `stream`."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(iters):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters * 1e-3


def time_graph_batch(stream, launches: int, fn, replays: int = 20) -> float:
    """Seconds per launch when `launches` calls of `fn(i, stream_ptr)` are
    captured in one CUDA graph and the graph is replayed."""
    import torch
    side = torch.cuda.Stream(stream.device)
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for i in range(launches):
            fn(i, side.cuda_stream)
    stream.wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    t = time_region(torch.cuda.current_stream(), replays, lambda i: g.replay())
    del g
    return t / launches


def measure_workload(w, x_host, dev, stream, l2, hbm, iters, bufs=None) -> dict:
    """Compress and decompress-reduce of one workload, each timed alone over
    back-to-back launches on rotating buffer sets (fraction of the HBM peak
    from the algorithmic bytes of one launch)."""
    import torch
    b = bufs or StepBuffers(w, x_host, dev, l2, stream)
    for k in range(b.R):
        b.compress(k)
    for i in range(5):
        b.decompress(i % b.R, (i + 1) % b.R)
    t_c = time_region(stream, iters, lambda i: b.compress(i % b.R))
    t_d = time_region(stream, iters, lambda i: b.decompress(i % b.R, (i + 1) % b.R))
    r = {"shape": [w.N, w.h], "block": w.block, "P": w.P,
         "compress": {"us": round(t_c * 1e6, 3), "alg_bytes": b.c_bytes,
                      "hbm_gbs": round(b.c_bytes / t_c / 1e9, 1),
                      "bf16_in_gbs": round(b.in_bytes / t_c / 1e9, 1),
                      "frac": round(b.c_bytes / t_c / 1e9 / hbm, 4)},
         "decompress_reduce": {"us": round(t_d * 1e6, 3), "alg_bytes": b.d_bytes,
                               "hbm_gbs": round(b.d_bytes / t_d / 1e9, 1),
                               "bf16_in_gbs": round(b.in_bytes / t_d / 1e9, 1),
                               "frac": round(b.d_bytes / t_d / 1e9 / hbm, 4)},
         "rotating_sets": b.R}
    if b.set_bytes * b.R < 8 * l2 and b.c_bytes < 16 * 2**20:
        # a launch this small is bound by launch latency and pipeline fill:
        # the same launches captured in one CUDA graph, per launch
        G = 64
        tg_c = time_graph_batch(stream, G, lambda i, sp: b.compress(i % b.R, sp))
        tg_d = time_graph_batch(stream, G, lambda i, sp: b.decompress(i % b.R, (i + 1) % b.R, sp))
        r["compress"]["graph_batch"] = {"launches": G, "us_per_launch": round(tg_c * 1e6, 3),
                                        "frac": round(b.c_bytes / tg_c / 1e9 / hbm, 4)}
        r["decompress_reduce"]["graph_batch"] = {"launches": G, "us_per_launch": round(tg_d * 1e6, 3),
                                                 "frac": round(b.d_bytes / tg_d / 1e9 / hbm, 4)}
        r["note"] = ("launch-latency bound: %.1f MB per compress launch moves in well under the "
                     "~3 us that filling and draining a launch costs, so 70%% of the HBM peak is not "
                     "reachable per launch at this size" % (b.c_bytes / 1e6))
    if bufs is None:
        del b
        torch.cuda.empty_cache()
    return r


def run_taco(args, w) -> None:
    import torch
    import torch.distributed as dist

    import grads_taco_compress_gb300 as taco
    from grads_taco_compress_gb300 import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = dataclasses.replace(w, seed=w.seed + rank)              # each rank its own batch
    lib = taco.library()
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    P, N, h, n = w.P, w.N, w.h, w.block
    K = h // n
    x_host = W.make_shards(w)                                     # bf16 bits [P, N, h]
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 2**20) or 129 * 2**20
    bufs = StepBuffers(w, x_host, dev, l2, stream)
    sb, in_bytes, set_bytes, R = bufs.sb, bufs.in_bytes, bufs.set_bytes, bufs.R
    xs, bundles, headers, outs, ws = bufs.xs, bufs.bundles, bufs.headers, bufs.outs, bufs.ws
    wsb = ws.numel()
    E = float(DEFAULT_TARGET_ENERGY)
    xp, bp, hp, op = bufs.xp, bufs.bp, bufs.hp, bufs.op
    compress, decompress = bufs.compress, bufs.decompress

    for k in range(R):                                            # every bundle holds codes
        compress(k)
    for i in range(args.warmup):
        compress(i % R)
        decompress(i % R, (i + 1) % R)
    torch.cuda.synchronize()

    steps = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    sampler = start_clock_sampler(f"GPU-{uuid}" if uuid else None)
    time.sleep(0.3)                                               # let the sampler start
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        k = i % R
        compress(k)
        decompress(k, (k + 1) % R)
    end.record(stream)
    torch.cuda.synchronize()

    # Launch duration of each kernel: its own timed region of back-to-back
    # launches on the same stream and buffers (events between the two kernels
    # of a step would break the launch overlap the step enjoys).
    kern_iters = max(100, steps // 2)

    def region(fn):
        return time_region(stream, kern_iters, fn)

    t_c = region(lambda i: compress(i % R))
    t_d = region(lambda i: decompress(i % R, (i + 1) % R))
    # the fused reduce -> recompress of the same bundles (next step of the
    # two-shot AllReduce), compressed sum only
    rc_shards = [torch.empty(sb, dtype=torch.uint8, device=dev) for _ in range(R)]
    rc_hdr = torch.empty(taco.HEADER_BYTES, dtype=torch.uint8, device=dev)
    ws1 = taco.new_workspace(1, dev)

    def recompress(k, src):
        st = lib.taco_reduce_recompress(bp[src], P, N, h, n, E, 0, rc_shards[k].data_ptr(),
                                        rc_hdr.data_ptr(), None, ws1.data_ptr(), ws1.numel(), sptr)
        if st:
            raise taco.TacoError(st, "taco_reduce_recompress")

    t_r = region(lambda i: recompress(i % R, (i + 1) % R))

    # the same compress with the rotation as a CUDA-core FWHT (measured
    # alternative; same outputs within the parity bar)
    fwht_bundles = [torch.empty((P, sb), dtype=torch.uint8, device=dev) for _ in range(R)]

    def compress_fwht(k):
        st = lib.taco_compress_shards_fwht(xp[k], P, N, h, n, E, 0, fwht_bundles[k].data_ptr(), hp[k],
                                      ws.data_ptr(), wsb, sptr)
        if st:
            raise taco.TacoError(st, "taco_compress_shards_fwht")

    for k in range(3):
        compress_fwht(k % R)
    t_f = region(lambda i: compress_fwht(i % R))

    # the INT8 fallback format: compress (tensor cores) and decompress-reduce
    # of its own bundles (same bytes per element as the FP8 format)
    def compress_int8(k):
        st = lib.taco_compress_shards_int8(xp[k], P, N, h, n, E, 0, fwht_bundles[k].data_ptr(), hp[k],
                                           ws.data_ptr(), wsb, sptr)
        if st:
            raise taco.TacoError(st, "taco_compress_shards_int8")

    def decompress_int8(k, src):
        st = lib.taco_decompress_reduce_int8(fwht_bundles[src].data_ptr(), P, N, h, n, op[k], sptr)
        if st:
            raise taco.TacoError(st, "taco_decompress_reduce_int8")

    for k in range(R):
        compress_int8(k)
    t_ci = region(lambda i: compress_int8(i % R))
    t_di = region(lambda i: decompress_int8(i % R, (i + 1) % R))

    # decompress-reduce with the inverse rotation on the tensor cores
    # (block 64 and 128), on the step's own bundles
    t_dm = None
    if n in (64, 128):
        def decompress_mma(k, src):
            st = lib.taco_decompress_reduce_mma(bp[src], P, N, h, n, op[k], sptr)
            if st:
                raise taco.TacoError(st, "taco_decompress_reduce_mma")

        for k in range(3):
            decompress_mma(k % R, (k + 1) % R)
        t_dm = region(lambda i: decompress_mma(i % R, (i + 1) % R))

    # Context for the roofline fractions: a plain device copy (torch copy_)
    # that reads and writes the same number of bytes as one launch of each
    # step kernel, timed the same way. The measured peak is a 4 GB copy; at
    # these sizes launch ramp-up and drain cost a copy a visible share too.
    def copy_same_bytes(total_bytes: int) -> float:
        nel = max(8, total_bytes // 4)
        reps = max(3, math.ceil(3 * l2 / (4 * nel)) + 1)
        src = [torch.empty(nel, dtype=torch.bfloat16, device=dev) for _ in range(reps)]
        dst = [torch.empty(nel, dtype=torch.bfloat16, device=dev) for _ in range(reps)]
        for i in range(5):
            dst[i % reps].copy_(src[i % reps])
        t = region(lambda i: dst[i % reps].copy_(src[i % reps]))
        del src, dst
        return t

    t_copy_c = copy_same_bytes(P * N * h * 3 + P * N * K * 8)
    t_copy_d = copy_same_bytes(P * N * h + P * N * K * 8 + N * h * 2)

    # The whole compressed two-shot AllReduce among P logical ranks (the P
    # input tensors of the step), captured in a CUDA graph and replayed.
    from grads_taco_compress_gb300.allreduce import EmulatedTwoShotAllReduce
    ar = EmulatedTwoShotAllReduce(P, N, h, n, E)
    ar(xs[0])
    torch.cuda.synchronize()
    graph = ar.capture(xs[0])
    t_ar = region(lambda i: graph.replay())
    ar_launches, ar_batched = ar.launches(), ar.batched
    del graph, ar
    # the same AllReduce in row segments on three streams (compress, reduce,
    # expand overlapped), one graph
    from grads_taco_compress_gb300.allreduce import PipelinedTwoShotAllReduce
    ar_seg = 4 if N % (4 * P) == 0 else 1
    par = PipelinedTwoShotAllReduce(P, N, h, n, segments=ar_seg, target_energy=E)
    par(xs[0])
    torch.cuda.synchronize()
    pgraph = par.capture(xs[0])
    t_par = region(lambda i: pgraph.replay())
    par_launches = par.launches()
    del pgraph, par

    # Every configuration of the operator's workloads, each kernel timed alone
    # the same way (the headline workload on its own buffers, the others on
    # fresh rotating sets of their own seeded inputs).
    peaks = measured_peaks()
    hbm = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
    peak_src = "measured" if peaks.get("hbm_gbs") else "fallback"
    by_workload = {}
    for name, w2 in W.WORKLOADS.items():
        if name == w.name:
            by_workload[name] = measure_workload(w, x_host, dev, stream, l2, hbm, kern_iters, bufs=bufs)
        else:
            w2 = dataclasses.replace(w2, seed=w2.seed + rank)
            by_workload[name] = measure_workload(w2, W.make_shards(w2), dev, stream, l2, hbm,
                                                 max(200, min(kern_iters, 2000)))
    if world > 1:
        dist.barrier()
    clocks = stop_clock_sampler(sampler)
    local_ms = start.elapsed_time(end)
    max_ms = reduce_max_over_ranks(local_ms, dev)

    # ---- end to end through the public API, host buffers in and out ----
    # Every step copies its P input shards in from pinned host memory,
    # compresses them, decompress-reduces the bundle and copies the bf16
    # result back. Pipelined on three streams: the host->device copy of step
    # t+1 and the device->host copy of step t-1 overlap the kernels of step t;
    # events keep the reuse of each buffer set in order. The serial form (one
    # stream, nothing overlapped) is reported beside it.
    x_pin = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_pins = [torch.empty((N, h), dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    e2e_steps = max(1, args.e2e_steps)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(R)]
    ev_comp = [torch.cuda.Event() for _ in range(R)]
    ev_out = [torch.cuda.Event() for _ in range(R)]
    t_count = [0]

    def e2e_step_pipelined():
        t = t_count[0]
        t_count[0] += 1
        k = t % R
        if t >= R:
            s_in.wait_event(ev_comp[k])        # step t-R's compress has read xs[k]
        with torch.cuda.stream(s_in):
            xs[k].copy_(x_pin, non_blocking=True)
        ev_in[k].record(s_in)
        s_comp.wait_event(ev_in[k])
        if t >= R:
            s_comp.wait_event(ev_out[k])       # step t-R's result has left outs[k]
        taco.taco_compress_shards_mma(xs[k], n, E, bundle=bundles[k], headers=headers[k], workspace=ws,
                                      stream=s_comp)
        taco.taco_decompress_reduce(bundles[k], P, N, h, n, out=outs[k], stream=s_comp)
        ev_comp[k].record(s_comp)
        s_out.wait_event(ev_comp[k])
        with torch.cuda.stream(s_out):
            out_pins[k].copy_(outs[k], non_blocking=True)
        ev_out[k].record(s_out)
        return ev_out[k]

    def e2e_step_serial(k):
        xs[k].copy_(x_pin, non_blocking=True)
        taco.taco_compress_shards_mma(xs[k], n, E, bundle=bundles[k], headers=headers[k], workspace=ws,
                                      stream=stream)
        taco.taco_decompress_reduce(bundles[k], P, N, h, n, out=outs[k], stream=stream)
        out_pins[k].copy_(outs[k], non_blocking=True)

    def timed_e2e(pipelined: bool) -> float:
        for i in range(3):
            e2e_step_pipelined() if pipelined else e2e_step_serial(i % R)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if pipelined:
            for s in (s_in, s_comp, s_out):
                s.wait_event(e0)
            last = None
            for i in range(e2e_steps):
                last = e2e_step_pipelined()
            stream.wait_event(last)
        else:
            for i in range(e2e_steps):
                e2e_step_serial(i % R)
        e1.record(stream)
        torch.cuda.synchronize()
        return reduce_max_over_ranks(e0.elapsed_time(e1), dev)

    e2e_ms = timed_e2e(True)
    e2e_serial_ms = timed_e2e(False)

    if rank == 0:
        c_bytes = P * N * h * 3 + P * N * K * 8
        d_bytes = P * N * h + P * N * K * 8 + N * h * 2
        r_bytes = (P + 1) * (N * h + N * K * 8)
        kern = {
            "compress": {"us": round(t_c * 1e6, 3), "alg_bytes": c_bytes,
                         "hbm_gbs": round(c_bytes / t_c / 1e9, 1),
                         "bf16_in_gbs": round(in_bytes / t_c / 1e9, 1),
                         "frac": round(c_bytes / t_c / 1e9 / hbm, 4),
                         "copy_same_bytes_frac": round(c_bytes / t_copy_c / 1e9 / hbm, 4),
                         "impl": "tcgen05 tensor-core Hadamard (taco_compress_shards_mma)"},
            "decompress_reduce": {"us": round(t_d * 1e6, 3), "alg_bytes": d_bytes,
                                  "hbm_gbs": round(d_bytes / t_d / 1e9, 1),
                                  "bf16_in_gbs": round(in_bytes / t_d / 1e9, 1),
                                  "frac": round(d_bytes / t_d / 1e9 / hbm, 4),
                                  "copy_same_bytes_frac": round(d_bytes / t_copy_d / 1e9 / hbm, 4)},
            "reduce_recompress": {"us": round(t_r * 1e6, 3), "alg_bytes": r_bytes,
                                  "hbm_gbs": round(r_bytes / t_r / 1e9, 1),
                                  "bf16_in_gbs": round(in_bytes / t_r / 1e9, 1),
                                  "frac": round(r_bytes / t_r / 1e9 / hbm, 4)},
            "compress_fwht": {"us": round(t_f * 1e6, 3), "alg_bytes": c_bytes,
                              "hbm_gbs": round(c_bytes / t_f / 1e9, 1),
                              "bf16_in_gbs": round(in_bytes / t_f / 1e9, 1),
                              "frac": round(c_bytes / t_f / 1e9 / hbm, 4),
                              "impl": "CUDA-core FWHT (taco_compress_shards_fwht), not in the timed step"},
            "compress_int8": {"us": round(t_ci * 1e6, 3), "alg_bytes": c_bytes,
                              "hbm_gbs": round(c_bytes / t_ci / 1e9, 1),
                              "frac": round(c_bytes / t_ci / 1e9 / hbm, 4),
                              "impl": "INT8 fallback codes, tensor cores, not in the timed step"},
            "decompress_reduce_int8": {"us": round(t_di * 1e6, 3), "alg_bytes": d_bytes,
                                       "hbm_gbs": round(d_bytes / t_di / 1e9, 1),
                                       "frac": round(d_bytes / t_di / 1e9 / hbm, 4),
                                       "impl": "INT8 fallback codes, not in the timed step"},
        }
        if t_dm is not None:
            kern["decompress_reduce_mma"] = {
                "us": round(t_dm * 1e6, 3), "alg_bytes": d_bytes,
                "hbm_gbs": round(d_bytes / t_dm / 1e9, 1),
                "frac": round(d_bytes / t_dm / 1e9 / hbm, 4),
                "impl": "tcgen05 E4M3 tensor-core inverse rotation, not in the timed step"}
        kern["emulated_two_shot_allreduce"] = {
            "us": round(t_ar * 1e6, 3), "ranks": P, "tensor": [N, h], "launches": ar_launches,
            "algbw_gbs": round(N * h * 2 / t_ar / 1e9, 1),
            "note": ("one CUDA graph: " + ("one compress launch for all ranks, one batched reduce-recompress, "
                                            "one expand" if ar_batched else
                                            "compress per rank, reduce-recompress per rank, one expand"))}
        kern["emulated_two_shot_allreduce_pipelined"] = {
            "us": round(t_par * 1e6, 3), "ranks": P, "tensor": [N, h], "segments": ar_seg,
            "launches": par_launches, "algbw_gbs": round(N * h * 2 / t_par / 1e9, 1),
            "note": "one CUDA graph: row segments through compress, reduce-recompress and expand on three "
                    "streams; the same bits as the serial graph"}
        dom = "compress" if t_c >= t_d else "decompress_reduce"
        achieved = kern[dom]["hbm_gbs"]
        line = {
            "metric": METRIC,
            "value": round(job_throughput(in_bytes, world, steps, max_ms), 3),
            "unit": "GB/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(max_ms / steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "shape": [N, h], "block": n, "P": P,
                       "target_energy": E, "variant": "dual",
                       "l2": f"inputs larger than L2: {R} rotating buffer sets of "
                             f"{set_bytes / 1e6:.1f} MB ({R * set_bytes / 1e6:.0f} MB vs "
                             f"{l2 / 1e6:.0f} MB L2)",
                       "parallelism": f"{world} independent rank(s), no data-path collective"},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm,
                         "peak_source": peak_src, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4),
                         "traffic": profiled_traffic(dom, w.name)},
            "kernels": kern,
            "by_workload": by_workload,
            "e2e": {"value": round(job_throughput(in_bytes, world, e2e_steps, e2e_ms), 3),
                    "unit": "GB/s", "h2d_bytes_per_step": in_bytes,
                    "d2h_bytes_per_step": N * h * 2, "steps": e2e_steps,
                    "schedule": "copies in, kernels and copies out of consecutive steps overlapped on 3 streams",
                    "serial_value": round(job_throughput(in_bytes, world, e2e_steps, e2e_serial_ms), 3)},
            "gpu_launches": 2 * steps,
            "clocks": clocks,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, x_host, args.cpu_baseline_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    sys.path.insert(0, str(ROOT))
    from grads_taco_compress_gb300 import workloads as W
    w = W.WORKLOADS[args.workload or W.BENCH_WORKLOAD]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_taco(args, w)


if __name__ == "__main__":
    main()
