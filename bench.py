"""Benchmark of the asynchronous global->shared streaming ring on GB300.

Default workload: the tiled scale y = 2x over 2**20 tiles of 256 float32
(1 GiB in, 1 GiB out) through the 2-stage ring (ap_scale), the configuration
the headline metric is quoted on. One step = one ap_scale call over the whole
input. Prints ONE JSON line (rank 0): achieved HBM GB/s (read + write bytes
per step / time), the roofline of the ring kernel against the measured copy
bandwidth, the synchronous baseline kernel on the same input, the oracle timed
on the host cores, and an end-to-end figure with host buffers.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl reference]
    python bench.py --workload all      # one line per workload of the sweep

Under torchrun (N > 1) every rank streams its own 1 GiB shard on its own GPU
(the operation is elementwise, so shards are independent and no collective
touches the data); the timing is the max over ranks and the value the bytes
of all ranks over that time (weak scaling).
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (read+write) and % of GB300 HBM roofline per kernel, 1 GPU"
GIB = 1 << 30
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000

# ----------------------------------------------------------------------------- helpers


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def hbm_peak() -> tuple[float, str]:
    pk = measured_peaks()
    if "hbm_gbs" in pk:
        return float(pk["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (~8 TB/s)

RING_SOURCES = ["stream_ring.cu", "stream_plan.h", "ptx.cuh", "device_common.cuh"]


def ring_source_hash() -> str:
    h = hashlib.sha256()
    for f in RING_SOURCES:
        with open(os.path.join(ROOT, "async_global_shared_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled(profile: str, pattern: str) -> float | None:
    """A figure from a committed ncu summary, if the summary was taken on the
    current kernel source (it records the source hash)."""
    p = os.path.join(ROOT, "profiles", profile)
    try:
        text = open(p).read()
    except OSError:
        return None
    m_hash = re.search(r"^source_hash:\s*(\w+)", text, re.M)
    m_val = re.search(pattern, text, re.M)
    if not m_hash or not m_val or m_hash.group(1) != ring_source_hash():
        return None
    return float(m_val.group(1))


def profiled_traffic(profile: str) -> float | None:
    """DRAM bytes per launch from a committed ncu summary (see _profiled)."""
    return _profiled(profile, r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)")


def profiled_dram_pct(profile: str) -> float | None:
    """ncu's gpu__dram_throughput (% of its DRAM peak) for the same launch."""
    return _profiled(profile, r"^\s*gpu__dram_throughput\s+([0-9.]+)\s*%")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = (
        "timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
        "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
        "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"
    )

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            self._wait_for_samples()
        except OSError:
            self.proc = None
        return self

    def _wait_for_samples(self, need: int = 2, limit_s: float = 10.0):
        """Return once nvidia-smi has written `need` samples (or has exited, or
        `limit_s` passed). Its start-up can hold the driver for most of a
        second; a timed region that overlapped it lost that time to idle."""
        t_end = time.monotonic() + limit_s
        while time.monotonic() < t_end and self.proc.poll() is None:
            try:
                with open(self.path) as fh:
                    if sum(1 for line in fh if line.strip()) >= need:
                        return
            except OSError:
                pass
            time.sleep(0.05)

    def mark_start(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _rows(self):
        if self.proc is None or self.path is None:
            return []
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        except OSError:
            pass
        return rows

    def window(self, t0, t1, rows=None) -> dict | None:
        """Median SM clock and active throttle reasons of the samples taken
        between t0 and t1 (the nearest sample if the window is shorter than
        the sampling period)."""
        rows = self._rows() if rows is None else rows
        if not rows:
            return None
        lo = t0 - datetime.timedelta(seconds=0.06)
        hi = t1 + datetime.timedelta(seconds=0.06)
        inside = [r for r in rows if lo <= r[0] <= hi]
        if not inside:
            mid = t0 + (t1 - t0) / 2
            inside = [min(rows, key=lambda r: abs((r[0] - mid).total_seconds()))]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        mhz = sorted(r[1] for r in inside)
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}

    def summary(self) -> dict | None:
        out = self.window(self.t0, self.t1)
        if self.path is not None and os.path.exists(self.path):
            os.unlink(self.path)
        return out


def time_steps(fn, steps: int, warmup: int, stream, dist_ctx=None) -> float:
    """Milliseconds for `steps` calls of fn(), CUDA events on `stream`, after
    `warmup` untimed calls; barrier + synchronize on both sides."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist_ctx:
        dist_ctx.barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    if dist_ctx:
        dist_ctx.barrier()
    return start.elapsed_time(end)


def time_each(fn, steps: int, warmup: int, stream) -> list:
    """Milliseconds of each of `steps` back-to-back calls of fn(): one CUDA
    event recorded on `stream` between consecutive calls, after `warmup`
    untimed calls."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        fn()
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if self.pg.get_backend() == "nccl":
                import torch

                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, v: float) -> float:
        if self.pg is None:
            return v
        import torch

        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------- oracle (CPU baseline)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_parallel_rate(fn, arrays, n: int, bytes_per_elem: float, threads: int, min_seconds: float,
                         max_passes: int) -> tuple[float, int, float]:
    """The oracle's own loops over [0, n) split into `threads` contiguous ranges
    run from Python threads (ctypes releases the GIL in foreign calls): bytes/s."""
    import threading

    bounds = [(t * n // threads, (t + 1) * n // threads) for t in range(threads)]
    passes = 0
    t0 = time.perf_counter()
    while True:
        ths = [threading.Thread(target=fn, args=(*[a[lo:hi] for a in arrays], hi - lo)) for lo, hi in bounds]
        for th in ths:
            th.start()
        for th in ths:
            th.join()
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= max_passes:
            break
    return bytes_per_elem * n * passes / el, passes, el


def oracle_scale_rate(x_host, alpha: float, min_seconds: float, max_passes: int) -> tuple[float, int, float]:
    """Bytes/s of the oracle's scale over x_host, passes until min_seconds."""
    import numpy as np

    import oracle

    orc = oracle.load()
    passes = 0
    t0 = time.perf_counter()
    while True:
        orc.scale(x_host, alpha)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= max_passes:
            break
    return 8.0 * x_host.size * passes / el, passes, el


# ----------------------------------------------------------------------------- workloads

SCALE_TILES = 1 << 20
SCALE_TILE = 256


E2E_CHUNKS = 16


def pipelined_host_step(ap, xh, yh, xd, yd, n_tiles, tile, alpha, stages, chunks, main):
    """A step that copies pinned host xh to the device, scales it with
    ap_scale and copies the result to pinned host yh, chunk by chunk on three
    streams (copy in, compute, copy out) so transfers overlap the kernel."""
    import torch

    s_in, s_c, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    per = n_tiles // chunks
    bounds = [(c * per, (c + 1) * per if c < chunks - 1 else n_tiles) for c in range(chunks)]

    def step():
        start = torch.cuda.Event()
        start.record(main)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for t0, t1 in bounds:
            a, b = t0 * tile, t1 * tile
            with torch.cuda.stream(s_in):
                xd[a:b].copy_(xh[a:b], non_blocking=True)
            e1 = torch.cuda.Event()
            e1.record(s_in)
            s_c.wait_event(e1)
            ap.ap_scale(xd[a:b], yd[a:b], t1 - t0, tile, alpha, stages, s_c)
            e2 = torch.cuda.Event()
            e2.record(s_c)
            s_out.wait_event(e2)
            with torch.cuda.stream(s_out):
                yh[a:b].copy_(yd[a:b], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        main.wait_event(done)

    return step


def bench_scale(args, d: Dist) -> dict:
    import numpy as np
    import torch

    import async_global_shared_gb300 as ap
    import synth

    dev = torch.device("cuda", d.local)
    torch.cuda.set_device(dev)
    n = SCALE_TILES * SCALE_TILE
    nbytes = 8 * n
    x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    assert ap.ap_check() == 0

    ring = lambda: ap.ap_scale(x, y, SCALE_TILES, SCALE_TILE, 2.0, 2, stream)  # noqa: E731
    sync = lambda: ap.ap_scale_sync(x, y, SCALE_TILES, SCALE_TILE, 2.0, stream)  # noqa: E731

    with ClockSampler(d.local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        for _ in range(args.warmup):
            ring()
        torch.cuda.synchronize()
        clk.mark_start()
        ms = time_steps(ring, args.steps, 0, stream, d)
        clk.mark_end()
        # the same launches back to back for about a second right after the
        # timed region, so the clock record rests on many samples under the
        # same load (the timed region itself may last a few milliseconds)
        sustain_steps = max(args.steps, int(1000.0 / max(ms / args.steps, 1e-3)))
        t_s0 = datetime.datetime.now()
        ms_sustained = time_steps(ring, sustain_steps, 0, stream, d)
        t_s1 = datetime.datetime.now()
    rows = clk._rows()  # complete once the sampler has exited
    clocks_sustained = clk.window(t_s0, t_s1, rows) if rows else None
    clocks = clk.summary()
    ms_sustained = d.max(ms_sustained)
    status = ap.ap_check()
    if status != 0:
        raise RuntimeError(f"device status {ap.ap_status_string(status)}")
    grid = ap.ap_debug_get(ap.AP_DBG_LAST_GRID)
    stage_elems = ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS)
    ms = d.max(ms)
    ms_step = ms / args.steps

    ms_sync = d.max(time_steps(sync, args.steps, args.warmup, stream, d)) / args.steps
    assert ap.ap_check() == 0

    # end to end: pinned host input -> device -> ap_scale -> pinned host output,
    # every step, in E2E_CHUNKS chunks so the two copy directions and the
    # kernel overlap (copy-in stream, compute stream, copy-out stream)
    xh = torch.empty(n, dtype=torch.float32, pin_memory=True)
    xh.copy_(x)
    yh = torch.empty(n, dtype=torch.float32, pin_memory=True)
    xd = torch.empty_like(x)
    e2e_step = pipelined_host_step(ap, xh, yh, xd, y, SCALE_TILES, SCALE_TILE, 2.0, 2, E2E_CHUNKS, stream)

    e2e_steps = max(3, min(args.steps, 20))
    ms_e2e = d.max(time_steps(e2e_step, e2e_steps, args.warmup, stream, d)) / e2e_steps
    assert ap.ap_check() == 0
    if not (torch.equal(yh[:4096], (xh[:4096] * 2.0)) and torch.equal(yh[-4096:], (xh[-4096:] * 2.0))):
        raise RuntimeError("end-to-end output check failed")
    # and directly: ap_scale on the pinned host buffers themselves, the kernel
    # reading and writing host memory over the host link (one launch a step)
    yh.fill_(float("nan"))
    direct_step = lambda: ap.ap_scale(xh, yh, SCALE_TILES, SCALE_TILE, 2.0, 2, stream)
    ms_direct = d.max(time_steps(direct_step, e2e_steps, args.warmup, stream, d)) / e2e_steps
    assert ap.ap_check() == 0
    if not (torch.equal(yh[:4096], (xh[:4096] * 2.0)) and torch.equal(yh[-4096:], (xh[-4096:] * 2.0))):
        raise RuntimeError("end-to-end (direct) output check failed")

    peak, peak_kind = hbm_peak()
    achieved = nbytes / (ms_step * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(d.world * nbytes / (ms_step * 1e-3) / 1e9, 1),
        "unit": "GB/s",
        "n_gpus": d.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": "tiled scale y=2.0*x, 2^20 tiles x 256 fp32 (1 GiB in + 1 GiB out), 2-stage ring (ap_scale)",
            "n_tiles": SCALE_TILES,
            "tile_elems": SCALE_TILE,
            "alpha": 2.0,
            "stages": 2,
            "stage_elems": stage_elems,
            "grid": grid,
            "input": "seeded uniform[-1,1) 24-bit grid, splitmix64",
            "l2": "inputs larger than L2 (1 GiB read + 1 GiB written per step vs 129 MB L2), no flush",
            "parallelism": f"{d.world} independent shard(s), no collective",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_kind": f"{peak_kind} copy bandwidth",
            "traffic": profiled_traffic("ring_scale_2p28.txt"),
            # the other two denominators: the nominal HBM3e figure, and ncu's own
            # DRAM peak for the full-size launch (from the same capture as traffic)
            "nominal_peak": NOMINAL_HBM_GBS,
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "ncu_dram_pct_of_peak": profiled_dram_pct("ring_scale_2p28.txt"),
            "kernel": "ring_kernel<OpScaleDev>",
            "algorithmic_bytes_per_launch": nbytes,
        },
        "baseline_sync": {
            "kernel": "scale_sync_kernel (load -> __syncthreads -> compute -> __syncthreads -> store)",
            "value": round(nbytes / (ms_sync * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "ms_per_step": round(ms_sync, 5),
        },
        "e2e": {
            "value": round(d.world * nbytes / (ms_direct * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": 4 * n,
            "d2h_bytes_per_step": 4 * n,
            "steps": e2e_steps,
            "pipeline": "ap_scale on pinned host input and output: the kernel reads and writes host memory "
                        "over the host link, one launch a step",
            "ms_per_step": round(ms_direct, 4),
            "copy_pipeline": {
                "value": round(d.world * nbytes / (ms_e2e * 1e-3) / 1e9, 1),
                "unit": "GB/s",
                "pipeline": f"{E2E_CHUNKS} chunks; H2D copy, ap_scale on device memory and D2H copy on three streams",
                "ms_per_step": round(ms_e2e, 4),
            },
        },
        "gpu_launches": args.steps,
        "clocks": clocks,
        "sustained": {
            "steps": sustain_steps,
            "ms_per_step": round(ms_sustained / sustain_steps, 5),
            "value": round(d.world * nbytes / (ms_sustained / sustain_steps * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "clocks": clocks_sustained,
            "note": "the same launches for about a second right after the timed region (not the headline)",
        },
    }
    if not args.no_per_kernel:
        del xh, yh, xd
        res["per_kernel"] = per_kernel_lines(ap, synth, dev, stream, peak, x, y)
    if d.rank == 0 and d.world == 1 and not args.no_cpu_baseline:
        import numpy as np  # noqa: F811

        x_host = x.cpu().numpy()
        rate, passes, el = oracle_scale_rate(x_host, 2.0, 10.0, 40)
        res["cpu_baseline"] = {
            "value": round(rate / 1e9, 3),
            "unit": "GB/s",
            "cores": 1,
            "kind": "oracle",
            "sample": f"{passes} full passes of the oracle's scale over the 2^28-float input ({el:.1f} s, 1 thread)",
        }
        import ctypes

        import numpy as np

        import oracle

        lib = oracle.load()._lib
        y_host = np.empty_like(x_host)
        cores = host_cores()
        fn = lambda a, b, m: lib.orc_scale(a.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),  # noqa: E731
                                           b.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), m, ctypes.c_float(2.0))
        prate, ppasses, pel = oracle_parallel_rate(fn, [x_host, y_host], x_host.size, 8.0, cores, 5.0, 40)
        res["cpu_baseline_all_cores"] = {
            "value": round(prate / 1e9, 3),
            "unit": "GB/s",
            "cores": cores,
            "kind": "oracle",
            "sample": f"{ppasses} passes over the 2^28-float input, the oracle's loop on {cores} contiguous ranges "
                      f"in {cores} threads ({pel:.1f} s)",
        }
    return res


def per_kernel_lines(ap, synth, dev, stream, peak, x, y) -> dict:
    """Every kernel of the path at its workload's full size, 20 timed launches
    after 3 warm-up (CUDA events), as GB/s (read + write bytes) over the mean
    launch and the fraction of the measured copy, with the median and best
    single launch of 20 more beside them. Timed separately from the headline: the
    synchronous and the pages' asynchronous scale, the ring's scale and row
    shift at every ring depth, the cluster calls, the masked copy, all 16
    (degree, depth) cells of the polynomial sweep and the two FP32 roofs."""
    import torch

    out = {}

    def put(name, nbytes, fn, **extra):
        # 20 launches back to back after 3 warm-up, timed as one region (the
        # mean launch: the rates below); then 20 more with an event between
        # launches for the median and best single launch (an event between
        # two launches keeps the second from starting under the first's tail,
        # which costs a 0.3 ms launch about 2 us)
        ms = time_steps(fn, 20, 3, stream) / 20
        each = sorted(time_each(fn, 20, 0, stream))
        gb = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"GB/s": round(gb, 1), "frac": round(gb / peak, 4), "ms": round(ms, 4),
                     "ms_median": round((each[9] + each[10]) / 2, 4), "ms_best": round(each[0], 4), **extra}
        return ms

    n = x.numel()  # 2^28 floats
    put("scale_sync (baseline), 2^20 x 256", 8 * n, lambda: ap.ap_scale_sync(x, y, n // 256, 256, 2.0, stream))
    put("scale, the pages' 2 x 1 KiB per-thread cp.async pipeline, 2^20 x 256", 8 * n,
        lambda: ap.ap_debug_scale_pages_async(x, y, n // 256, 256, 2.0, stream))
    for S in (2, 3, 4, 5, 6):
        put(f"scale ring S={S}, 2^20 x 256", 8 * n, lambda: ap.ap_scale(x, y, n // 256, 256, 2.0, S, stream))
    # context, not this library's kernel: torch's vectorized elementwise
    # multiply over the same 2^28 floats, a plain load/store streaming kernel
    put("context: torch.mul(x, 2) (torch's vectorized elementwise kernel), 2^28", 8 * n,
        lambda: torch.mul(x, 2.0, out=y))
    for S in (2, 3, 4, 5, 6):
        ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, S)
        put(f"row roll 2^26 x 4, shift 1, S={S}", 8 * n, lambda: ap.ap_row_roll(x, y, n // 4, 4, 1, stream))
    ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, 0)
    put("row roll 2^26 x 4, A + 4 bytes", 8 * (n - 4), lambda: ap.ap_row_roll(x[1:n - 3], y[:n - 4], (n - 4) // 4, 4, 1,
                                                                                   stream))
    for cs in (2, 4, 8):
        put(f"cluster exchange cs={cs}, 32 KiB chunks", 8 * n,
            lambda: ap.ap_cluster_exchange(x, y, n, cs, 32768, stream))
    put("cluster exchange_ex cs=16, 32 KiB chunks", 8 * n,
        lambda: ap.ap_cluster_exchange_ex(x, y, n, 16, 32768, 1, stream))
    for cs in (4, 8, 16):
        put(f"cluster all-to-all cs={cs}, 32 KiB chunks", 8 * n,
            lambda: ap.ap_cluster_all_to_all(x, y, n, cs, 32768, stream))
    # The mixed pattern, then the same codes taken apart: a chunk left
    # unchanged (code -1) beside a written one leaves its 32-byte sector half
    # written, and the L2 fetches such a sector from DRAM before writing it
    # back; half and zeroed chunks, or chunks left in whole sectors, do not.
    plain_ms = None
    for name, pattern in (("all chunks copied", [16]),
                          ("1/8 off, 1/8 half, 1/8 zeroed, 5/8 copied", [-1, 8, -2, 16, 16, 16, 16, 16]),
                          ("1/8 half, 1/8 zeroed, 6/8 copied (no chunk left)", [8, -2, 16, 16, 16, 16, 16, 16]),
                          ("1/8 off, 7/8 copied (a half-written sector in four)", [-1, 16, 16, 16, 16, 16, 16, 16]),
                          ("2/8 off in whole sectors, 6/8 copied", [-1, -1, 16, 16, 16, 16, 16, 16])):
        codes = torch.tensor(pattern, dtype=torch.int8).repeat(n // 4 // len(pattern)).to(dev)
        # per 16-byte chunk: the bytes it reads, the 16 it writes unless predicated off, 1 code byte
        rd = sum(max(c, 0) for c in pattern) / len(pattern)
        wr = sum(16 for c in pattern if c != -1) / len(pattern)
        key = f"masked copy, {name}"
        ms = put(key, (n // 4) * (rd + wr + 1), lambda: ap.ap_masked_copy(x, y, n // 4, codes, 4, stream))
        if plain_ms is None:
            plain_ms = ms
        else:
            out[key]["time_vs_all_copied"] = round(ms / plain_ms, 4)
        del codes
    xp = synth.uniform_pm1_torch(synth.SEED_POLY, 1 << 30, dev)
    yp = torch.empty_like(xp)
    for K in (0, 8, 32, 128):
        c = synth.coeffs_np(K).tolist()
        for S in (2, 3, 4, 6):
            key = f"poly K={K}, 2^30, S={S}"
            ms = put(key, 8 * (1 << 30), lambda: ap.ap_poly(xp, yp, 1 << 30, c, K, S, stream))
            out[key]["fp32_tflops"] = round(2.0 * K * (1 << 30) / (ms * 1e-3) / 1e12, 2)
            if K == 0:
                # degree 0 needs only the writes: its rate over the 4 B an element
                # that minimum moves, beside the 8 B the ring streams
                out[key]["write_only_GB/s"] = round(4 * (1 << 30) / (ms * 1e-3) / 1e9, 1)
    del xp, yp
    # The FP32 roofs under the same clocks: register-only fma chains, and the
    # operand pattern of the Horner loop (a coefficient read from shared memory
    # as the third operand), which is what a run-time polynomial can reach.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    probe = torch.empty(sms * 1024, dtype=torch.float32, device=dev)
    roofs = {}
    for key, fn, fma in (("fp32 fma probe, registers only", ap.ap_debug_fma_probe, sms * 1024 * 32 * (1 << 14)),
                         ("fp32 fma probe, Horner operands", ap.ap_debug_fma_probe_horner,
                          sms * 512 * 24 * 128 * (1 << 10))):
        iters = 1 << 14 if fn is ap.ap_debug_fma_probe else 1 << 10
        ms = time_steps(lambda: fn(probe, probe.numel(), iters, stream), 20, 3, stream) / 20
        roofs[key] = 2.0 * fma / (ms * 1e-3) / 1e12
        out[key] = {"fp32_tflops": round(roofs[key], 2), "ms": round(ms, 4)}
    del probe
    for S in (2, 3, 4, 6):
        k128 = out[f"poly K=128, 2^30, S={S}"]
        k128["frac_of_register_probe"] = round(k128["fp32_tflops"] / roofs["fp32 fma probe, registers only"], 4)
        k128["frac_of_horner_probe"] = round(k128["fp32_tflops"] / roofs["fp32 fma probe, Horner operands"], 4)
    st = ap.ap_check()
    if st != 0:
        raise RuntimeError(f"device status {ap.ap_status_string(st)}")
    return out


def run_reference(args, d: Dist):
    """The CPU oracle, as it stands, on the same workload and metric."""
    if d.rank != 0:
        return
    import numpy as np

    import oracle
    import synth

    sample = 1 << 24  # 1/16 of the 2^28-float workload per step
    x = synth.uniform_pm1_np(synth.SEED_SCALE, sample)
    orc = oracle.load()
    for _ in range(args.warmup):
        orc.scale(x, 2.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.scale(x, 2.0)
    el = time.perf_counter() - t0
    gbs = 8.0 * sample * args.steps / el / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 3),
        "unit": "GB/s",
        "n_gpus": d.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": "tiled scale y=2.0*x, 2^20 tiles x 256 fp32 (1 GiB in + 1 GiB out), 2-stage ring (ap_scale)",
            "n_tiles": SCALE_TILES,
            "tile_elems": SCALE_TILE,
            "alpha": 2.0,
        },
        "cpu_baseline": {
            "value": round(gbs, 3),
            "unit": "GB/s",
            "cores": 1,
            "kind": "oracle",
            "sample": "each step: the oracle's scale over the first 2^24 floats (1/16) of the workload, 1 thread",
        },
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, "reference")


# ----------------------------------------------------------------------------- sweep (per-kernel lines)


def _gbs(nbytes: float, ms: float) -> float:
    return nbytes / (ms * 1e-3) / 1e9


def sweep(which: str, args):
    """One line per (kernel, configuration): GB/s from CUDA events over
    `steps` launches and the fraction of the measured copy bandwidth. Also the
    FP32 rate of the polynomial for the compute-bound degrees."""
    import torch

    import async_global_shared_gb300 as ap
    import synth

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peak, _ = hbm_peak()
    steps, warm = max(5, min(args.steps, 50)), args.warmup
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = (["scale", "poly", "roll", "exchange", "alltoall", "masked", "small"] if which == "all"
              else which.split(","))

    window = {}

    single = {}  # the median and best single launch of the last run()

    def line(workload, kernel, nbytes, ms, **extra):
        gb = _gbs(nbytes, ms)
        d = {"workload": workload, "kernel": kernel, "ms": round(ms, 5), "GB/s": round(gb, 1),
             "frac_of_measured_hbm": round(gb / peak, 4)}
        d.update(single)
        single.clear()
        d.update(extra)
        if ap.ap_check() != 0:
            d["device_status"] = "error"
        d["_window"] = (window["t0"], window["t1"])
        return d

    def run(fn):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        window["t0"] = datetime.datetime.now()
        ms = time_steps(fn, steps, 0, stream) / steps
        # then up to 20 launches with an event between them, for the median
        # and best single launch (rates stay those of the back-to-back region)
        each = sorted(time_each(fn, min(steps, 20), 0, stream))
        window["t1"] = datetime.datetime.now()
        single.update(ms_median=round(each[len(each) // 2], 5), ms_best=round(each[0], 5))
        return ms

    if "scale" in groups:
        n_t, t = SCALE_TILES, SCALE_TILE
        n = n_t * t
        x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
        y = torch.empty_like(x)
        ms = run(lambda: ap.ap_scale_sync(x, y, n_t, t, 2.0))
        yield line("scale 2^28 f32", "scale_sync", 8 * n, ms)
        ms = run(lambda: ap.ap_debug_scale_pages_async(x, y, n_t, t, 2.0))
        yield line("scale 2^28 f32", "the pages' async pipeline (2 x 1 KiB, per-thread cp.async)", 8 * n, ms)
        for S in (2, 3, 4, 5, 6):
            ms = run(lambda: ap.ap_scale(x, y, n_t, t, 2.0, S))
            yield line("scale 2^28 f32", f"ring S={S}", 8 * n, ms,
                       stage_elems=ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS),
                       grid=ap.ap_debug_get(ap.AP_DBG_LAST_GRID))
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)  # the tensor-map producer
        for S in (2, 3, 4, 5, 6):
            ms = run(lambda: ap.ap_scale(x, y, n_t, t, 2.0, S))
            yield line("scale 2^28 f32", f"ring tensor-map producer S={S}", 8 * n, ms,
                       stage_elems=ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS),
                       grid=ap.ap_debug_get(ap.AP_DBG_LAST_GRID), flags=ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS))
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 0)
        del x, y
    if "poly" in groups:
        n = 1 << 30
        x = synth.uniform_pm1_torch(synth.SEED_POLY, n, dev)
        y = torch.empty_like(x)
        for K in (0, 8, 32, 128):
            c = synth.coeffs_np(K).tolist()
            for S in (2, 3, 4, 6):
                ms = run(lambda: ap.ap_poly(x, y, n, c, K, S))
                tflops = 2.0 * K * n / (ms * 1e-3) / 1e12
                yield line("poly 2^30 f32", f"ring S={S} K={K} (defaults)", 8 * n, ms,
                           fp32_tflops=round(tflops, 2), fma_per_elem=K,
                           stage_elems=ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS))
        # the FP32 roofs measured under the same conditions: register-only fma
        # chains, and the Horner loop's operand pattern without memory
        probe = torch.empty(sms * 1024, dtype=torch.float32, device=dev)
        for kern, fn, iters, fma in (
                ("fma_probe_kernel (registers only)", ap.ap_debug_fma_probe, 1 << 16, sms * 1024 * 32),
                ("fma_probe_horner_kernel (Horner operands)", ap.ap_debug_fma_probe_horner, 1 << 10,
                 sms * 512 * 24 * 128)):
            ms = run(lambda: fn(probe, probe.numel(), iters))
            d = line("fp32 fma probe", kern, 0, ms, fp32_tflops=round(2.0 * fma * iters / (ms * 1e-3) / 1e12, 2))
            d.pop("GB/s")
            d.pop("frac_of_measured_hbm")
            yield d
        del x, y, probe
    if "roll" in groups:
        rows, cols = 1 << 26, 4
        n = rows * cols
        abuf = torch.empty(n + 4, dtype=torch.float32, device=dev)
        bbuf = torch.empty(n + 4, dtype=torch.float32, device=dev)
        synth.uniform_pm1_torch(synth.SEED_ROLL, n + 4, dev, out=abuf)
        for name, sa, sb in (("aligned", 0, 0), ("A+4B", 1, 0), ("B+4B", 0, 1), ("A+4B,B+4B", 1, 1)):
            A, B = abuf[sa:sa + n], bbuf[sb:sb + n]
            ms = run(lambda: ap.ap_row_roll(A, B, rows, cols, 1))
            yield line("roll 2^26x4 f32", f"ring {name}", 8 * n, ms,
                       flags=ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS), stages=ap.ap_debug_get(ap.AP_DBG_LAST_STAGES))
        # the tensor-map producer (aligned variant): each stage one 2-D box of
        # 1 KiB lines of the input, the stage that wraps as 1-D boxes
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
        for r, c in ((rows, cols), (n // 64, 64)):
            for S in (2, 3, 4):
                ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, S)
                A, B = abuf[:n], bbuf[:n]
                ms = run(lambda: ap.ap_row_roll(A, B, r, c, 1))
                fl = ap.ap_debug_get(ap.AP_DBG_LAST_FLAGS)
                yield line(f"roll {r}x{c} f32", f"ring tensor-map producer S={S}",
                           8 * n, ms, flags=fl, stage_elems=ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS))
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 0)
        ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, 0)
        del abuf, bbuf
    if "exchange" in groups:
        n = 1 << 28
        x = synth.uniform_pm1_torch(synth.SEED_EXCHANGE, n, dev)
        y = torch.empty_like(x)
        # small chunks (the pages' example moves 256 bytes): batched against plain pieces
        for chunk in (256, 1024, 4096):
            for batch in (0, 1):
                ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, batch)
                for cs in (2, 4, 8):
                    ms = run(lambda: ap.ap_cluster_exchange(x, y, n, cs, chunk))
                    yield line(f"exchange 2^28 f32, {chunk} B chunks",
                               f"cluster cs={cs} {'batched (auto)' if batch == 0 else 'pieces'}", 8 * n, ms,
                               slots=ap.ap_debug_get(ap.AP_DBG_LAST_STAGES),
                               item_bytes=4 * ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS))
                    if chunk % (16 * cs) == 0:
                        ms = run(lambda: ap.ap_cluster_all_to_all(x, y, n, cs, chunk))
                        yield line(f"all-to-all 2^28 f32, {chunk} B chunks",
                                   f"cluster a2a cs={cs} {'batched (auto)' if batch == 0 else 'pieces'}", 8 * n, ms,
                                   slots=ap.ap_debug_get(ap.AP_DBG_LAST_STAGES),
                                   item_bytes=4 * ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS))
        ap.ap_debug_set(ap.AP_DBG_EXCHANGE_BATCH, 0)
        for cs, shift in ((3, 1), (6, 2), (16, 1), (16, 5)):
            ms = run(lambda: ap.ap_cluster_exchange_ex(x, y, n, cs, 32768, shift))
            yield line("exchange 2^28 f32, 32 KiB chunks", f"cluster_ex cs={cs} shift={shift}", 8 * n, ms,
                       grid=ap.ap_debug_get(ap.AP_DBG_LAST_GRID))
        for cs in (1, 2, 4, 8):
            ms = run(lambda: ap.ap_cluster_exchange(x, y, n, cs, 32768))
            yield line("exchange 2^28 f32, 32 KiB chunks", f"cluster cs={cs} (defaults)", 8 * n, ms,
                       grid=ap.ap_debug_get(ap.AP_DBG_LAST_GRID), slots=ap.ap_debug_get(ap.AP_DBG_LAST_STAGES))
        del x, y
    if "alltoall" in groups:
        n = 1 << 28
        x = synth.uniform_pm1_torch(synth.SEED_EXCHANGE, n, dev)
        y = torch.empty_like(x)
        for cs in (1, 2, 4, 8, 16):
            ms = run(lambda: ap.ap_cluster_all_to_all(x, y, n, cs, 32768))
            yield line("all-to-all 2^28 f32, 32 KiB chunks", f"cluster a2a cs={cs} (defaults)", 8 * n, ms,
                       grid=ap.ap_debug_get(ap.AP_DBG_LAST_GRID), slots=ap.ap_debug_get(ap.AP_DBG_LAST_STAGES),
                       piece_bytes=4 * ap.ap_debug_get(ap.AP_DBG_LAST_STAGE_ELEMS))
        del x, y
    if "autotune" in groups:
        n = 1 << 28
        x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
        y = torch.empty_like(x)
        for name, op, S, deg in (("scale", ap.AP_TUNE_SCALE, 2, 0), ("scale", ap.AP_TUNE_SCALE, 4, 0),
                                 ("roll", ap.AP_TUNE_ROW_ROLL, 3, 0), ("poly K=32", ap.AP_TUNE_POLY, 3, 32)):
            t0 = time.perf_counter()
            shape = ap.ap_autotune(op, x, y, n, S, deg)
            yield {"workload": "autotune 2^28 f32", "kernel": f"{name} S={S}", "chosen": shape,
                   "tuning_seconds": round(time.perf_counter() - t0, 2)}
        ap.ap_autotune_reset()
        del x, y
    if "masked" in groups:
        n_chunks = 1 << 26
        x = synth.uniform_pm1_torch(synth.SEED_SCALE, 4 * n_chunks, dev)
        y = torch.empty_like(x)
        for name, pattern in (("all 16 (plain copy)", [16]),
                              ("1/8 off, 1/8 half, 1/8 zeroed, 5/8 copies", [-1, 8, -2, 16, 16, 16, 16, 16]),
                              ("1/8 half, 1/8 zeroed, 6/8 copies (no chunk left)", [8, -2, 16, 16, 16, 16, 16, 16]),
                              ("1/8 off, 7/8 copies", [-1, 16, 16, 16, 16, 16, 16, 16]),
                              ("2/8 off in whole sectors, 6/8 copies", [-1, -1, 16, 16, 16, 16, 16, 16])):
            pat = torch.tensor(pattern, dtype=torch.int8)
            codes = pat.repeat(n_chunks // len(pattern)).to(dev)
            rd = sum(max(c, 0) for c in pattern) / len(pattern)
            wr = sum(16 for c in pattern if c != -1) / len(pattern)
            nbytes = n_chunks * (rd + wr + 1)
            for S in (2, 3, 4, 6):
                ms = run(lambda: ap.ap_masked_copy(x, y, n_chunks, codes, S))
                yield line("masked copy 2^26 chunks", f"{name} S={S}", nbytes, ms,
                           grid=ap.ap_debug_get(ap.AP_DBG_LAST_GRID))
        del x, y
    if "e2e" in groups:
        n_t, t = SCALE_TILES, SCALE_TILE
        n = n_t * t
        x = synth.uniform_pm1_torch(synth.SEED_SCALE, n, dev)
        xh = torch.empty(n, dtype=torch.float32, pin_memory=True)
        xh.copy_(x)
        yh = torch.empty(n, dtype=torch.float32, pin_memory=True)
        xd = torch.empty_like(x)
        yd = torch.empty_like(x)
        main = torch.cuda.current_stream()
        # the host link alone: one direction at a time, then both at once
        s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
        ms = run(lambda: xd.copy_(xh, non_blocking=True))
        yield line("host link", "H2D 1 GiB pinned", 4 * n, ms)
        ms = run(lambda: yh.copy_(yd, non_blocking=True))
        yield line("host link", "D2H 1 GiB pinned", 4 * n, ms)

        def both():
            ev = torch.cuda.Event()
            ev.record(main)
            s_a.wait_event(ev)
            s_b.wait_event(ev)
            with torch.cuda.stream(s_a):
                xd.copy_(xh, non_blocking=True)
            with torch.cuda.stream(s_b):
                yh.copy_(yd, non_blocking=True)
            for st in (s_a, s_b):
                e = torch.cuda.Event()
                e.record(st)
                main.wait_event(e)

        ms = run(both)
        yield line("host link", "H2D + D2H 1 GiB each, concurrent", 8 * n, ms)
        for chunks in (16,):
            for n_in in (1,):
                s_in = [torch.cuda.Stream() for _ in range(n_in)]
                s_out = [torch.cuda.Stream() for _ in range(n_in)]
                s_c = torch.cuda.Stream()
                per = n_t // chunks

                def step():
                    ev0 = torch.cuda.Event()
                    ev0.record(main)
                    done = []
                    for c in range(chunks):
                        a, b = c * per * t, (c + 1) * per * t
                        si, so = s_in[c % n_in], s_out[c % n_in]
                        si.wait_event(ev0)
                        with torch.cuda.stream(si):
                            xd[a:b].copy_(xh[a:b], non_blocking=True)
                        e1 = torch.cuda.Event()
                        e1.record(si)
                        s_c.wait_event(e1)
                        ap.ap_scale(xd[a:b], yd[a:b], per, t, 2.0, 2, s_c)
                        e2 = torch.cuda.Event()
                        e2.record(s_c)
                        so.wait_event(e2)
                        with torch.cuda.stream(so):
                            yh[a:b].copy_(yd[a:b], non_blocking=True)
                        e3 = torch.cuda.Event()
                        e3.record(so)
                        done.append(e3)
                    for e in done:
                        main.wait_event(e)

                for _ in range(3):
                    step()
                torch.cuda.synchronize()
                window["t0"] = datetime.datetime.now()
                ms = time_steps(step, 10, 0, main)
                window["t1"] = datetime.datetime.now()
                ok = torch.equal(yh[-4096:], xh[-4096:] * 2.0)
                yield line("e2e scale 2^28 f32 pinned host", f"chunks={chunks} copy_streams={n_in}", 8 * n, ms / 10,
                           output_ok=ok)
        del x, xd, yd
    if "oracle" in groups:
        # the CPU oracle on each workload: one thread, and (where its loop splits
        # into independent ranges) the same loop on every host core
        import ctypes

        import numpy as np

        import oracle

        orc = oracle.load()
        lib = orc._lib
        fp = ctypes.POINTER(ctypes.c_float)
        cores = host_cores()

        def rate1(fn, nbytes, min_s=2.0):
            t0 = time.perf_counter()
            k = 0
            while True:
                fn()
                k += 1
                el = time.perf_counter() - t0
                if el >= min_s or k >= 20:
                    return nbytes * k / el / 1e9

        n = 1 << 28
        x = synth.uniform_pm1_np(synth.SEED_SCALE, n)
        y = np.empty_like(x)
        r1 = rate1(lambda: orc.scale(x, 2.0), 8.0 * n)
        sc = lambda a, b, m: lib.orc_scale(a.ctypes.data_as(fp), b.ctypes.data_as(fp), m, ctypes.c_float(2.0))  # noqa
        rN = oracle_parallel_rate(sc, [x, y], n, 8.0, cores, 2.0, 20)[0] / 1e9
        yield {"workload": "oracle: scale 2^28 f32", "GB/s 1 core": round(r1, 2), f"GB/s {cores} cores": round(rN, 2)}
        A = x[: 1 << 28].reshape(-1, 4)
        r1 = rate1(lambda: orc.row_roll(A, 1), 8.0 * n)
        yield {"workload": "oracle: row roll 2^26x4 f32", "GB/s 1 core": round(r1, 2),
               "note": "one call over the whole matrix (the wrap couples its ends)"}
        r1 = rate1(lambda: orc.cluster_exchange(x, 4, 32768), 8.0 * n)
        ex = lambda a, b, m: lib.orc_cluster_exchange(a.ctypes.data_as(fp), b.ctypes.data_as(fp), m, 4, 32768)  # noqa
        n_groups = n // (4 * 8192)
        # the threads' ranges must hold whole groups of 4 chunks
        rN = oracle_parallel_rate(ex, [x, y], n, 8.0, cores, 2.0, 20)[0] / 1e9 if n_groups % cores == 0 else None
        yield {"workload": "oracle: cluster exchange cs=4 2^28 f32", "GB/s 1 core": round(r1, 2),
               f"GB/s {cores} cores": None if rN is None else round(rN, 2)}
        m = 1 << 22
        xs = x[:m]
        ys = np.empty_like(xs)
        for K in (8, 32, 128):
            c = synth.coeffs_np(K)
            r1 = rate1(lambda: orc.poly(xs, c), 8.0 * m)
            pf = lambda a, b, mm: lib.orc_poly(a.ctypes.data_as(fp), b.ctypes.data_as(fp), mm,  # noqa: E731
                                               c.ctypes.data_as(fp), K)
            rN = oracle_parallel_rate(pf, [xs, ys], m, 8.0, cores, 2.0, 20)[0] / 1e9
            yield {"workload": f"oracle: poly K={K} (2^22-float sample)", "GB/s 1 core": round(r1, 3),
                   f"GB/s {cores} cores": round(rN, 3), "GFLOP/s 1 core": round(r1 / 8 * 2 * K, 2)}
        del x, y
    if "small" in groups:
        A = torch.arange(256, dtype=torch.float32, device=dev).reshape(64, 4)
        B = torch.empty_like(A)
        ms = run(lambda: ap.ap_row_roll(A, B, 64, 4, 1))
        yield {"workload": "roll 64x4 f32 (one CTA, 64 threads)", "kernel": "roll_small",
               "us_per_call": round(ms * 1e3, 2), "note": "launch-latency bound; no roofline",
               "_window": (window["t0"], window["t1"])}
        # the same calls replayed from a CUDA graph (100 calls per graph),
        # captured on a side stream and replayed on the timed stream
        calls = 100
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            ap.ap_row_roll(A, B, 64, 4, 1, gs)
        gs.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            for _ in range(calls):
                ap.ap_row_roll(A, B, 64, 4, 1, gs)
        ms = run(g.replay) / calls
        yield {"workload": "roll 64x4 f32 (one CTA, 64 threads)", "kernel": "roll_small, 100 calls per CUDA graph",
               "us_per_call": round(ms * 1e3, 2), "note": "graph replay removes the per-call launch cost",
               "_window": (window["t0"], window["t1"])}
        del g
    yield {"workload": "device", "sms": sms, "hbm_peak_gbs": peak}


# ----------------------------------------------------------------------------- profiling cases

PROFILE_CASES = ("scale", "scale_s3", "scale_s4", "scale_s5", "scale_s6", "sync", "pages_async",
                 "poly0", "poly0_s3", "poly0_s4", "poly0_s6", "poly8", "poly8_s3", "poly8_s4", "poly8_s6",
                 "poly32_s2", "poly32", "poly32_s4", "poly32_s6", "poly40_s2", "poly48_s2", "poly128", "poly128_s3",
                 "poly128_s4", "poly128_s6",
                 "roll", "roll_s3", "roll_s4", "roll_s5", "roll_s6", "roll_mis", "roll_tensor",
                 "exchange2", "exchange4", "exchange8", "exchange16",
                 "a2a4", "a2a8", "a2a16", "exchange4_256B", "masked", "masked_mixed", "masked_all", "masked_off1",
                 "masked_offpair", "masked_halfzero", "torch_mul_2p28")


def profile_case(name: str, args):
    """Run one kernel on a small case (inputs still larger than L2, a few
    hundred MiB on the device) `warmup + steps` times, for ncu captures."""
    import torch

    import async_global_shared_gb300 as ap
    import synth

    dev = torch.device("cuda", 0)
    if name == "torch_mul_2p28":
        # a plain vectorized load/store kernel (torch's elementwise multiply,
        # not this library's) over the headline's 2^28 floats, at full size;
        # the inputs come from fill kernels, so the multiply is the first
        # float elementwise kernel of the process
        a = torch.empty(1 << 28, dtype=torch.float32, device=dev).fill_(1.5)
        b = torch.empty_like(a)
        for _ in range(args.warmup + args.steps):
            torch.mul(a, 2.0, out=b)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": name, "launches": args.warmup + args.steps, "status": 0}), flush=True)
        return
    n = 1 << 26  # 256 MiB in + 256 MiB out
    x = synth.uniform_pm1_torch(synth.SEED_SCALE, n + 4, dev)
    y = torch.empty_like(x)
    codes = torch.tensor([-1, 8, -2, 16, 16, 16, 16, 16], dtype=torch.int8).repeat(n // 32).to(dev)
    codes16 = torch.full((n // 4,), 16, dtype=torch.int8, device=dev)

    def pattern(p):  # per-chunk codes repeating p over the case's n / 4 chunks
        return torch.tensor(p, dtype=torch.int8).repeat(n // 4 // len(p)).to(dev)

    rest = [16] * 6
    calls = {
        "scale": lambda: ap.ap_scale(x[:n], y[:n], n // 256, 256, 2.0, 2),
        "sync": lambda: ap.ap_scale_sync(x[:n], y[:n], n // 256, 256, 2.0),
        "poly32": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(32).tolist(), 32, 3),
        "poly128": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(128).tolist(), 128, 2),
        "poly32_s4": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(32).tolist(), 32, 4),
        "poly32_s6": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(32).tolist(), 32, 6),
        "poly128_s6": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(128).tolist(), 128, 6),
        "poly0": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(0).tolist(), 0, 2),
        "poly8": lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(8).tolist(), 8, 2),
        "exchange2": lambda: ap.ap_cluster_exchange(x[:n], y[:n], n, 2, 32768),
        "exchange8": lambda: ap.ap_cluster_exchange(x[:n], y[:n], n, 8, 32768),
        "scale_s6": lambda: ap.ap_scale(x[:n], y[:n], n // 256, 256, 2.0, 6),
        "roll": lambda: ap.ap_row_roll(x[:n], y[:n], n // 4, 4, 1),
        "roll_mis": lambda: ap.ap_row_roll(x[1:n + 1], y[:n], n // 4, 4, 1),
        "exchange4": lambda: ap.ap_cluster_exchange(x[:n], y[:n], n, 4, 32768),
        "exchange16": lambda: ap.ap_cluster_exchange_ex(x[:n], y[:n], n, 16, 32768, 1),
        "a2a4": lambda: ap.ap_cluster_all_to_all(x[:n], y[:n], n, 4, 32768),
        "a2a8": lambda: ap.ap_cluster_all_to_all(x[:n], y[:n], n, 8, 32768),
        "exchange4_256B": lambda: ap.ap_cluster_exchange(x[:n], y[:n], n, 4, 256),
        "a2a16": lambda: ap.ap_cluster_all_to_all(x[:n], y[:n], n, 16, 32768),
        "roll_tensor": lambda: ap.ap_row_roll(x[:n], y[:n], n // 4, 4, 1),
        "masked": lambda: ap.ap_masked_copy(x[:n], y[:n], n // 4, codes, 4),
        "masked_mixed": lambda: ap.ap_masked_copy(x[:n], y[:n], n // 4, codes, 4),
        "masked_all": lambda: ap.ap_masked_copy(x[:n], y[:n], n // 4, codes16, 4),
    }
    calls["pages_async"] = lambda: ap.ap_debug_scale_pages_async(x[:n], y[:n], n // 256, 256, 2.0)
    # every (degree, depth) cell of the polynomial sweep and every depth of the
    # scale and the row shift: polyK_sS, scale_sS, roll_sS (the row shift's
    # depth through AP_DBG_ROLL_STAGES)
    m = re.fullmatch(r"poly(\d+)_s(\d)", name)
    if m and name not in calls:
        deg, depth = int(m.group(1)), int(m.group(2))
        calls[name] = lambda: ap.ap_poly(x[:n], y[:n], n, synth.coeffs_np(deg).tolist(), deg, depth)
    m = re.fullmatch(r"(scale|roll)_s(\d)", name)
    if m and name not in calls:
        depth = int(m.group(2))
        if m.group(1) == "scale":
            calls[name] = lambda: ap.ap_scale(x[:n], y[:n], n // 256, 256, 2.0, depth)
        else:
            ap.ap_debug_set(ap.AP_DBG_ROLL_STAGES, depth)
            calls[name] = lambda: ap.ap_row_roll(x[:n], y[:n], n // 4, 4, 1)
    # the mixed pattern taken apart: one chunk left in eight, two adjacent
    # chunks left (whole sectors), a half and a zeroed chunk in eight
    for key, p in (("masked_off1", [-1, 16] + rest), ("masked_offpair", [-1, -1] + rest),
                   ("masked_halfzero", [8, -2] + rest)):
        if name == key:
            pc = pattern(p)
            calls[key] = lambda: ap.ap_masked_copy(x[:n], y[:n], n // 4, pc, 4)
    if name == "roll_tensor":
        ap.ap_debug_set(ap.AP_DBG_FORCE_PATH, 3)
    fn = calls[name]
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    st = ap.ap_check()
    print(json.dumps({"profile_case": name, "launches": args.warmup + args.steps, "status": st}), flush=True)
    if st != 0:
        raise SystemExit(1)


# ----------------------------------------------------------------------------- results log
RESULTS_DIR = os.path.join(ROOT, "results")
_PROVENANCE = None


def provenance() -> dict:
    """Where a result came from: GPU, git commit (when the tree has .git), a
    hash of the CUDA sources, time and command line."""
    global _PROVENANCE
    if _PROVENANCE is None:
        sha = None
        try:
            r = subprocess.run(["git", "rev-parse", "HEAD"], cwd=ROOT, capture_output=True, text=True, timeout=10)
            if r.returncode == 0 and r.stdout.strip():
                sha = r.stdout.strip()
        except (OSError, subprocess.SubprocessError):
            pass
        h = hashlib.sha256()
        src = os.path.join(ROOT, "async_global_shared_gb300", "csrc")
        for f in sorted(os.listdir(src)):
            with open(os.path.join(src, f), "rb") as fh:
                h.update(f.encode() + b"\0" + fh.read())
        gpu = None
        try:
            import torch

            if torch.cuda.is_available():
                gpu = torch.cuda.get_device_name(0)
        except Exception:  # noqa: BLE001 - provenance is best effort
            pass
        _PROVENANCE = {"gpu": gpu, "git_sha": sha, "source_hash": h.hexdigest()[:16], "argv": sys.argv[1:]}
    return dict(_PROVENANCE, time=datetime.datetime.now(datetime.timezone.utc).isoformat(timespec="seconds"))


def emit(line: dict, kind: str) -> None:
    """Print one JSON result line and append it, with its provenance, to
    results/<kind>.jsonl (bench: the headline line; sweep: per-kernel lines;
    reference: the oracle arm)."""
    print(json.dumps(line), flush=True)
    try:
        os.makedirs(RESULTS_DIR, exist_ok=True)
        with open(os.path.join(RESULTS_DIR, f"{kind}.jsonl"), "a") as f:
            f.write(json.dumps(dict(line, provenance=provenance())) + "\n")
    except OSError:
        pass


def main(argv=None):
    ap_ = argparse.ArgumentParser()
    ap_.add_argument("--gpus", type=int, default=1)
    ap_.add_argument("--steps", type=int, default=1000)
    ap_.add_argument("--warmup", type=int, default=5)
    ap_.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap_.add_argument("--workload", default="scale")
    ap_.add_argument("--no-cpu-baseline", action="store_true")
    ap_.add_argument("--no-per-kernel", action="store_true")
    ap_.add_argument("--profile-case", choices=PROFILE_CASES, default=None)
    args = ap_.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    d = Dist()
    try:
        if args.impl == "reference":
            run_reference(args, d)
            return
        import __graft_entry__

        __graft_entry__.build()
        if args.profile_case:
            if d.rank == 0:
                profile_case(args.profile_case, args)
        elif args.workload == "scale":
            res = bench_scale(args, d)
            if d.rank == 0:
                emit(res, "bench")
        elif d.rank == 0:
            with ClockSampler(0) as clk:
                lines = list(sweep(args.workload, args))
            rows = clk._rows()
            if clk.path and os.path.exists(clk.path):
                os.unlink(clk.path)
            for line in lines:
                w = line.pop("_window", None)
                if w is not None:
                    line["clocks"] = clk.window(w[0], w[1], rows)
                emit(line, "sweep")
    finally:
        d.close()


if __name__ == "__main__":
    main()
